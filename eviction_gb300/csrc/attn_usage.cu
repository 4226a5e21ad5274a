// attn_usage.cu -- attention usage of the cache by the window queries, on the
// 5th-generation tensor cores (tcgen05 + TMEM) with TMA-staged operands.
//
// What it computes ("Adaptive Mass-Segmented KV Compression for Long-Form
// Reasoning", Method, Key design 1; "SkipKV: ...", A2 token importance score):
// for every unit (layer, sequence, KV head), every query row r = (head g of the
// GQA group, window index j) and every cache slot i it can see (pad <= i <=
// T-W+j), p = softmax_i(scale * q_r . k_i); the usage of slot i is the sum of
// p over the rows.  The fill of unseen entries and everything after it is
// done by the mass kernel.
//
// Each softmax row needs its normaliser before its probabilities can be summed
// per slot, and the normaliser spans every slot.  The work is therefore split
// into two tensor-core passes over the same QK^T:
//   pass 1: rows on TMEM lanes (A = 128 query rows, B = 128-slot chunks of K);
//           each epilogue thread owns one row and keeps an online max / sum;
//           out: per row (scaled log2 max, sum of exp2 relative to it).
//   pass 2: slots on TMEM lanes (A = 128 cached keys, B = 128-row chunks of
//           Q); each epilogue thread owns one slot and sums
//           exp2(scale*log2e*z - b_r) over the rows, b_r = log2 normaliser.
// Both passes are persistent, warp-specialised kernels: warp 0 issues TMA
// loads into a 4-stage ring, warp 1 issues tcgen05.mma into two TMEM
// accumulators, and two epilogue warpgroups (warps 2-5 and 6-9) drain them:
// warpgroup w takes every accumulator of parity w and writes partial results
// (per-row statistics, per-slot sums) to its own half of the workspace; the
// consumers combine the two halves.  Every wait is bounded.
#include <cmath>
#include <cstdio>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kEpiWarps = 8;                    // two warpgroups
constexpr int kThreads = 64 + 32 * kEpiWarps;   // + TMA warp + MMA warp
constexpr int BM = 128;        // A-operand rows (TMEM lanes)
constexpr int BN = 128;        // B-operand rows per chunk (TMEM columns)
constexpr int kStages = 4;     // B ring depth
constexpr int kAccCols = 2 * BN;  // two accumulators

struct Params {
  int U, T, R, W, B, H;
  int n_items, n_tiles, r_local;  // r_local: rows of row constants per buffer
  float scale_log2;
  const int32_t* pad;
  float2* rowpart;   // [2][U][R] per-warpgroup row statistics
  float* usage;      // [2][U][T] per-warpgroup slot sums
  uint32_t* status;
};

struct Item {
  int u, tile, pad, n_ch, a_row, b_row0, c_start;
};

template <int PASS>
__device__ __forceinline__ Item decode(const Params& p, int item) {
  Item it;
  it.u = item / p.n_tiles;
  it.tile = item - it.u * p.n_tiles;
  const int b = (it.u / p.H) % p.B;
  it.pad = min(max(p.pad[b], 0), p.T);
  if (PASS == 1) {
    it.c_start = (it.pad / BN) * BN;
    it.n_ch = (it.pad < p.T) ? (p.T - it.c_start + BN - 1) / BN : 0;
    it.a_row = it.u * p.R + it.tile * BM;
    it.b_row0 = it.u * p.T + it.c_start;
  } else {
    const int p0 = it.tile * BM;
    it.c_start = 0;
    it.n_ch = (p0 + BM > it.pad && it.pad < p.T) ? (p.R + BN - 1) / BN : 0;
    it.a_row = it.u * p.T + p0;
    it.b_row0 = it.u * p.R;
  }
  return it;
}

template <int D>
struct Layout {
  static constexpr int kKB = D / 64;               // 64-element (128 B) K blocks
  static constexpr int kABytes = BM * D * 2;
  static constexpr int kBBytes = BN * D * 2;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = 2 * kABytes;
  static constexpr int kOffBars = kOffB + kStages * kBBytes;
  static constexpr int kNumBars = 2 * kStages + 6 + 1 + 4;
  static_assert(kNumBars <= 24, "barrier area holds 24 barriers");
  static constexpr int kOffMisc = kOffBars + 24 * 8;
  static constexpr int kOffRowB = kOffMisc + 16;   // pass 2: row constants [2 wg][2 buf]
  static size_t bytes(int r_local) {
    return 1024 + kOffRowB + 4 * static_cast<size_t>(r_local) * 4;
  }
};

// Rows of row constants one warpgroup holds per item: its share of the chunks.
__host__ __device__ inline int rows_local(int R) {
  const int n_ch = (R + BN - 1) / BN;
  return ((n_ch + 1) / 2) * BN;
}

// Warp-uniform wait for the epilogue warps: lane 0 waits, the result is
// broadcast, so that the collective TMEM loads that follow run converged.
__device__ __forceinline__ bool epi_wait(uint64_t* bar, uint32_t parity,
                                         volatile int* abort, uint32_t* status,
                                         int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           uint32_t* status) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, status);
}

__device__ __forceinline__ float4 lds128(const float* ptr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(ptr)));
  return v;
}

__device__ __forceinline__ float lds32(const float* ptr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(smem_u32(ptr)));
  return v;
}

__device__ __forceinline__ void sts32(float* ptr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(smem_u32(ptr)), "f"(v) : "memory");
}

// Row normaliser b_r = log2 sum_i exp2(x_i) from the two warpgroups' partial
// (max, sum) pairs (x = scaled logits); +inf for a row that sees nothing.
__device__ __forceinline__ float combine_row_b(float2 a, float2 b) {
  const float m = fmaxf(a.x, b.x);
  if (m == -INFINITY) return INFINITY;
  const float s = a.y * ex2(a.x - m) + b.y * ex2(b.x - m);
  return s > 0.f ? m + log2f(s) : INFINITY;
}

template <int D, int PASS>
__global__ void __launch_bounds__(kThreads, 1)
    usage_kernel(const __grid_constant__ CUtensorMap map_a,
                 const __grid_constant__ CUtensorMap map_b, Params p) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle, as an offset from the shared
  // array so that the compiler keeps the shared address space
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* smem = smem_raw + ((1024u - mis) & 1023u);
  uint8_t* a_buf = smem + Ly::kOffA;
  uint8_t* b_buf = smem + Ly::kOffB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kOffBars);
  uint64_t* full = bars;                  // [kStages]
  uint64_t* empty = bars + kStages;       // [kStages]
  uint64_t* afull = bars + 2 * kStages;   // [2]
  uint64_t* aempty = afull + 2;           // [2]
  uint64_t* accfull = aempty + 2;         // [2]
  uint64_t* accempty = accfull + 2;       // [2] (one arrival per epilogue warp)
  uint64_t* done = accempty + 2;          // [1]
  uint64_t* rb_full = done + 1;           // [2 wg][2 buf] row constants written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + Ly::kOffMisc + 4);
  float* row_b_all = reinterpret_cast<float*>(smem + Ly::kOffRowB);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 1);
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 4);
    }
    mbar_init(done, 1);
    for (int b = 0; b < 4; ++b) mbar_init(&rb_full[b], 128);
    *abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kAccCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int a_iter = 0, b_iter = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
        const Item it = decode<PASS>(p, item);
        if (it.n_ch == 0) continue;
        const int ab = a_iter & 1;
        if (!mbar_wait(&aempty[ab], ((a_iter >> 1) & 1) ^ 1, abort, p.status)) {
          ok = false;
          break;
        }
        ++a_iter;
        mbar_arrive_expect_tx(&afull[ab], Ly::kABytes);
        for (int kb = 0; kb < Ly::kKB; ++kb)
          tma_load_2d(a_buf + ab * Ly::kABytes + kb * BM * 128, &map_a, kb * 64,
                      it.a_row, &afull[ab]);
        for (int c = 0; c < it.n_ch; ++c) {
          const int s = b_iter % kStages;
          if (!mbar_wait(&empty[s], ((b_iter / kStages) & 1) ^ 1, abort,
                         p.status)) {
            ok = false;
            break;
          }
          ++b_iter;
          mbar_arrive_expect_tx(&full[s], Ly::kBBytes);
          for (int kb = 0; kb < Ly::kKB; ++kb)
            tma_load_2d(b_buf + s * Ly::kBBytes + kb * BN * 128, &map_b,
                        kb * 64, it.b_row0 + c * BN, &full[s]);
        }
      }
      // drain: every issued load must land before the CTA may exit
      for (int i = (b_iter > kStages ? b_iter - kStages : 0); i < b_iter; ++i)
        drain_wait(&full[i % kStages], (i / kStages) & 1, p.status);
      for (int i = (a_iter > 2 ? a_iter - 2 : 0); i < a_iter; ++i)
        drain_wait(&afull[i & 1], (i >> 1) & 1, p.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      const uint32_t a_base = smem_u32(a_buf), b_base = smem_u32(b_buf);
      int a_iter = 0, b_iter = 0, acc_iter = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
        const Item it = decode<PASS>(p, item);
        if (it.n_ch == 0) continue;
        const int ab = a_iter & 1;
        if (!mbar_wait(&afull[ab], (a_iter >> 1) & 1, abort, p.status)) {
          ok = false;
          break;
        }
        ++a_iter;
        for (int c = 0; c < it.n_ch; ++c) {
          const int acc = acc_iter & 1;
          const int s = b_iter % kStages;
          if (!mbar_wait(&accempty[acc], ((acc_iter >> 1) & 1) ^ 1, abort,
                         p.status) ||
              !mbar_wait(&full[s], (b_iter / kStages) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tile = a_base + ab * Ly::kABytes;
          const uint32_t b_tile = b_base + s * Ly::kBBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const int kb = k / 4, kk = k % 4;
            const uint64_t ad = sw128_desc(a_tile + kb * BM * 128 + kk * 32);
            const uint64_t bd = sw128_desc(b_tile + kb * BN * 128 + kk * 32);
            mma_bf16(tmem + acc * BN, ad, bd, idesc, k > 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          mma_commit(&accfull[acc]);
          ++b_iter;
          ++acc_iter;
        }
        if (ok) mma_commit(&aempty[ab]);
      }
      mma_commit(done);
      drain_wait(done, 0, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = (warp - 2) >> 2;   // warpgroup: accumulators of parity wg
    const int quarter = warp & 3;     // TMEM lane quarter this warp may access
    const int lrow = quarter * 32 + lane;
    const uint32_t t_acc =
        tmem + (static_cast<uint32_t>(quarter * 32) << 16) + wg * BN;
    const float c = p.scale_log2;
    int k_iter = 0;   // accumulators consumed by this warpgroup
    int g = 0;        // global chunk index of the item's first chunk
    int rb_iter = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
      const Item it = decode<PASS>(p, item);
      const int first = (wg - g) & 1;   // first chunk of this item that is ours
      g += it.n_ch;
      if (PASS == 1) {
        const int r = it.tile * BM + lrow;
        const int qpos = p.T - p.W + (r % p.W);
        const bool row_valid = (r < p.R) && (qpos >= it.pad) && (it.n_ch > 0);
        float mz = -INFINITY, sum = 0.f;  // max in raw logit units, sum rel. to it
        for (int ch = first; ch < it.n_ch; ch += 2) {
          if (!epi_wait(&accfull[wg], k_iter & 1, abort, p.status, lane)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int c0 = it.c_start + ch * BN;
          const int lo = max(it.pad, c0), hi = min(qpos, c0 + BN - 1);
          const bool fast = __all_sync(0xffffffffu,
                                       row_valid && lo == c0 && hi == c0 + BN - 1);
#pragma unroll 1
          for (int bt = 0; bt < BN / 32; ++bt) {
            uint32_t v[32];
            __syncwarp();
            tmem_ld32(t_acc + bt * 32, v);
            tmem_ld_wait();
            if (fast) {
              float bm0 = __uint_as_float(v[0]), bm1 = __uint_as_float(v[1]);
#pragma unroll
              for (int i = 2; i < 32; i += 2) {
                bm0 = fmaxf(bm0, __uint_as_float(v[i]));
                bm1 = fmaxf(bm1, __uint_as_float(v[i + 1]));
              }
              const float bm = fmaxf(bm0, bm1);
              if (bm > mz) {
                sum *= ex2((mz - bm) * c);
                mz = bm;
              }
              const float neg = -mz * c;
              float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                s0 += ex2(fmaf(__uint_as_float(v[i]), c, neg));
                s1 += ex2(fmaf(__uint_as_float(v[i + 1]), c, neg));
                s2 += ex2(fmaf(__uint_as_float(v[i + 2]), c, neg));
                s3 += ex2(fmaf(__uint_as_float(v[i + 3]), c, neg));
              }
              sum += (s0 + s1) + (s2 + s3);
            } else if (row_valid) {
              const int p0 = c0 + bt * 32;
              float bm = -INFINITY;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (p0 + i >= lo && p0 + i <= hi) bm = fmaxf(bm, __uint_as_float(v[i]));
              if (bm > mz) {
                sum *= ex2((mz - bm) * c);
                mz = bm;
              }
              const float neg = -mz * c;
              float s0 = 0.f;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (p0 + i >= lo && p0 + i <= hi)
                  s0 += ex2(fmaf(__uint_as_float(v[i]), c, neg));
              sum += s0;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[wg]);
          ++k_iter;
        }
        if (!ok) break;
        if (r < p.R) {
          const float2 st = (row_valid && sum > 0.f) ? make_float2(mz * c, sum)
                                                     : make_float2(-INFINITY, 0.f);
          p.rowpart[(static_cast<size_t>(wg) * p.U + it.u) * p.R + r] = st;
        }
      } else {
        if (it.n_ch == 0) continue;
        // Row constants of the chunks this warpgroup takes, double buffered
        // across items: every thread of the warpgroup writes its share and
        // arrives; a thread only rewrites a buffer after the whole warpgroup
        // arrived for the following item, i.e. finished with it.
        const int rb = rb_iter & 1;
        float* row_b = row_b_all + (wg * 2 + rb) * p.r_local;
        {
          int l = 0;
          for (int ch = first; ch < it.n_ch; ch += 2, ++l) {
            const int r = ch * BN + lrow;
            float bv = INFINITY;
            if (r < p.R) {
              const size_t o = static_cast<size_t>(it.u) * p.R + r;
              bv = combine_row_b(p.rowpart[o],
                                 p.rowpart[static_cast<size_t>(p.U) * p.R + o]);
            }
            sts32(row_b + l * BN + lrow, bv);
          }
        }
        mbar_arrive(&rb_full[wg * 2 + rb]);
        if (!mbar_wait(&rb_full[wg * 2 + rb], (rb_iter >> 1) & 1, abort, p.status)) break;
        ++rb_iter;
        const int pos = it.tile * BM + lrow;
        const bool pos_valid = (pos >= it.pad) && (pos < p.T);
        const bool fast = __all_sync(0xffffffffu, pos_valid && (pos <= p.T - p.W));
        const int jmin = pos - (p.T - p.W);  // rows with j >= jmin see pos
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        int l = 0;
        for (int ch = first; ch < it.n_ch; ch += 2, ++l) {
          if (!epi_wait(&accfull[wg], k_iter & 1, abort, p.status, lane)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int bt = 0; bt < BN / 32; ++bt) {
            uint32_t v[32];
            __syncwarp();
            tmem_ld32(t_acc + bt * 32, v);
            tmem_ld_wait();
            const float* rbb = row_b + l * BN + bt * 32;
            if (fast) {
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 bb = lds128(rbb + i);
                a0 += ex2(fmaf(__uint_as_float(v[i]), c, -bb.x));
                a1 += ex2(fmaf(__uint_as_float(v[i + 1]), c, -bb.y));
                a2 += ex2(fmaf(__uint_as_float(v[i + 2]), c, -bb.z));
                a3 += ex2(fmaf(__uint_as_float(v[i + 3]), c, -bb.w));
              }
            } else if (pos_valid) {
              const int r0 = ch * BN + bt * 32;
              int j = r0 % p.W;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                if (j >= jmin && r0 + i < p.R)
                  a0 += ex2(fmaf(__uint_as_float(v[i]), c, -lds32(rbb + i)));
                j = (j + 1 == p.W) ? 0 : j + 1;
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[wg]);
          ++k_iter;
        }
        if (!ok) break;
        if (pos_valid)
          p.usage[(static_cast<size_t>(wg) * p.U + it.u) * p.T + pos] = (a0 + a1) + (a2 + a3);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kAccCols);
#endif
}

// ------------------------------------------------------------------ host ----

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode(std::string* err) {
  static EncodeTiledFn fn = nullptr;
  if (fn) return fn;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr,
                                                   12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr) {
    if (err) *err = "cuTensorMapEncodeTiled not available from the driver";
    return nullptr;
  }
  fn = reinterpret_cast<EncodeTiledFn>(ptr);
  return fn;
}

// 2-D view [rows][d] of a bf16 tensor, boxes of 64 x 128 elements, 128 B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, int d,
              std::string* err) {
  EncodeTiledFn enc = get_encode(err);
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                   dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")";
    return false;
  }
  return true;
}

template <int D>
cudaError_t launch_d(const kvc_handle* h, const UsageArgs& a, int pass, cudaStream_t s,
                     std::string* err) {
  const Dims& dm = h->dims;
  CUtensorMap map_q, map_k;
  if (!make_map(&map_q, a.q, static_cast<uint64_t>(dm.U) * dm.R, D, err) ||
      !make_map(&map_k, a.k, static_cast<uint64_t>(dm.U) * a.T, D, err))
    return cudaErrorInvalidValue;

  Params p;
  p.U = dm.U;
  p.T = a.T;
  p.R = dm.R;
  p.W = dm.W;
  p.B = dm.B;
  p.H = dm.H;
  p.scale_log2 = a.scale_log2;
  p.pad = a.pad;
  p.rowpart = h->ws.rowstat;
  p.usage = h->ws.usage;
  p.r_local = rows_local(dm.R);
  p.status = h->ws.status;

  cudaError_t e;
  if (pass == 1) {
    // items = (unit, 128-row tile)
    const size_t smem = Layout<D>::bytes(0);
    e = cudaFuncSetAttribute(usage_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    p.n_tiles = (dm.R + BM - 1) / BM;
    p.n_items = dm.U * p.n_tiles;
    const int grid = p.n_items < h->num_sms ? p.n_items : h->num_sms;
    usage_kernel<D, 1><<<grid, kThreads, smem, s>>>(map_q, map_k, p);
  } else {
    // items = (unit, 128-slot tile)
    const size_t smem = Layout<D>::bytes(p.r_local);
    e = cudaFuncSetAttribute(usage_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    p.n_tiles = (a.T + BM - 1) / BM;
    p.n_items = dm.U * p.n_tiles;
    const int grid = p.n_items < h->num_sms ? p.n_items : h->num_sms;
    usage_kernel<D, 2><<<grid, kThreads, smem, s>>>(map_k, map_q, p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_usage(const kvc_handle* h, const UsageArgs& a, int pass,
                                   cudaStream_t s, std::string* err) {
  switch (h->dims.d) {
    case 64:
      return launch_d<64>(h, a, pass, s, err);
    case 128:
      return launch_d<128>(h, a, pass, s, err);
    default:
      if (err) *err = "head_dim must be 64 or 128";
      return cudaErrorInvalidValue;
  }
}

size_t attention_usage_smem_bytes(int d, int R) {
  const int rl = rows_local(R);
  return d == 64 ? Layout<64>::bytes(rl) : Layout<128>::bytes(rl);
}

}  // namespace kvc
