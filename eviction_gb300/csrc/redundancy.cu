// redundancy.cu -- SkipKV key-redundancy score mixed into the selection score.
//
// "SkipKV: Selective Skipping of KV Generation and Storage for Efficient
// Inference with Large Reasoning Models", A2 Method details, 4.1: the token
// redundancy score (after R-KV) and the final eviction score: per KV head, r_i = the mean cosine similarity of key i to the other
// valid keys, R = softmax of r over the valid slots, I = score / (sum of the
// score over the valid slots), and selection runs on f = sigma*I - (1-sigma)*R
// (more redundant -> evicted earlier).  Padding slots never count and get
// f = -inf.
//
// The mean cosine needs no n x n similarity matrix.  With k^_j = k_j / |k_j|
// (the zero vector for a zero key) and S = sum over the valid j of k^_j,
//     sum over j != i of cos(k_i, k_j) = k^_i . S - [k_i != 0]
// exactly, so a unit costs O(n d).
//
// Work layout: persistent CTAs, one unit at a time each.  A producer warp
// streams the unit's valid key rows through a ring of 24 KB shared-memory
// chunks by 1-D bulk async copies, twice: pass A (row norms, S) and pass B
// (k^_i . S, chunks newest first).  It runs ahead across passes and units, so
// the ring never drains; the second read of a unit comes a few hundred KB
// after the first and is served mostly by L2 (the first read is tagged
// evict-last, the second evict-first).  Twelve consumer warps take a chunk
// when its copy lands and free it with one arrival per warp.  Per row, 1/|k|
// and e^r (and the scores, copied in asynchronously while the passes run)
// stay in shared memory for units up to 2048 slots, else they use device
// scratch; the sums over the unit (S, sum e^r, sum score) are fixed-order
// trees, so repeated calls give the same bits.  Every wait is bounded and
// reports through the status word.
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kConsumerWarps = 12;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;  // + the producer warp
constexpr int kChunkBytes = 24576;         // 96 rows of d 128, 192 of d 64: two consumer steps
constexpr int kStages = 3;
constexpr int kRowsCap = 2048;             // units up to this many slots keep per-row values in smem
constexpr int kEpl = 16;                   // key elements per lane and row (two 16-byte loads)
constexpr int kBarConsumers = 1;           // named barrier of the consumer warps

struct RedArgs {
  const uint16_t* k;
  const float* score;
  const int32_t* pad;
  float* sel;     // may alias score
  float* red;     // optional R output
  float* rinv;    // [U][T] scratch: 1/|k| per slot
  float* rexp;    // [U][T] scratch: e^r per slot
  int T, B, H, U;
  float sigma;
  uint32_t* status;
};

template <int D>
struct Geo {
  static constexpr int kLpr = D / kEpl;                    // lanes per row: 8 (d 128), 4 (d 64)
  static constexpr int kRpw = 32 / kLpr;                   // rows per warp and step
  static constexpr int kRowsStep = kConsumerWarps * kRpw;  // rows per consumer step
  static constexpr int kChunkRows = kChunkBytes / (D * 2);
  static constexpr int kSteps = kChunkRows / kRowsStep;    // 2
  static constexpr int kGroups = kRpw / 4;                 // row groups per warp after two folds
  static_assert(kChunkRows % kRowsStep == 0, "a chunk is a whole number of consumer steps");
};

struct RedSmem {
  static constexpr size_t ring = 0;
  static constexpr size_t sacc = ring + static_cast<size_t>(kStages) * kChunkBytes;  // [12][128]
  static constexpr size_t stot = sacc + kConsumerWarps * 128 * 4;                     // [128]
  static constexpr size_t wsum = stot + 128 * 4;                                      // [12][2]
  static constexpr size_t full = wsum + kConsumerWarps * 2 * 4;
  static constexpr size_t empty = full + kStages * 8;
  static constexpr size_t abort_flag = empty + kStages * 8;
  static constexpr size_t rows = abort_flag + 16;  // [3][kRowsCap] 1/|k|, e^r, score (short units)
  static constexpr size_t bytes(bool rows_in_smem) {
    return rows + (rows_in_smem ? 3 * kRowsCap * 4 : 0);
  }
};

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16),
// with an L2 cache policy.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 4-byte asynchronous global -> shared copies (the unit's scores, landing
// while the passes run).
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kBarConsumers), "n"(kConsumers) : "memory");
}

// The valid rows [pad, T) of unit u.
__device__ __forceinline__ int unit_pad(const RedArgs& a, int u) {
  return min(max(a.pad[(u / a.H) % a.B], 0), a.T);
}

// 16 bf16 of one row held by one lane as 8 fp32 pairs: elements [8 sub, 8 sub + 8)
// and [D/2 + 8 sub, D/2 + 8 sub + 8).
__device__ __forceinline__ void unpack16(const uint4 w0, const uint4 w1, float2 (&x)[8]) {
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j)
    x[j] = make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
}

__device__ __forceinline__ uint4 lds4(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }

// Pass A, one row: acc += k / |k|; returns 1/|k| (0 for a zero key).
template <int D>
__device__ __forceinline__ float pass_a_row(const uint4 w0, const uint4 w1, float2 (&acc)[8]) {
  float2 x[8];
  unpack16(w0, w1, x);
  float2 sa = make_float2(0.f, 0.f), sb = sa;  // two chains: half the latency
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    sa = fma2(x[j], x[j], sa);
    sb = fma2(x[j + 1], x[j + 1], sb);
  }
  const float2 s2 = add2(sa, sb);
  float ss = s2.x + s2.y;
#pragma unroll
  for (int o = Geo<D>::kLpr / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
  const float2 iv = make_float2(inv, inv);
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = fma2(x[j], iv, acc[j]);
  return inv;
}

// Pass B, one row: k . S.
template <int D>
__device__ __forceinline__ float pass_b_row(const uint4 w0, const uint4 w1, const float2 (&sv)[8]) {
  float2 x[8];
  unpack16(w0, w1, x);
  float2 da = make_float2(0.f, 0.f), db = da;
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    da = fma2(x[j], sv[j], da);
    db = fma2(x[j + 1], sv[j + 1], db);
  }
  const float2 d2 = add2(da, db);
  float dot = d2.x + d2.y;
#pragma unroll
  for (int o = Geo<D>::kLpr / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  return dot;
}

// Rows of one chunk for this lane: calls f(row_in_chunk, w0, w1, ok) per
// consumer step; a full chunk is unrolled without row guards.
template <int D, typename F>
__device__ __forceinline__ void for_chunk_rows(const uint16_t* buf, int rows, int grp, int sub,
                                               F&& f) {
  using G = Geo<D>;
  if (rows == G::kChunkRows) {
    uint4 w[G::kSteps][2];
#pragma unroll
    for (int st = 0; st < G::kSteps; ++st) {
      const uint16_t* row = buf + (st * G::kRowsStep + grp) * D;
      w[st][0] = lds4(row + sub * 8);
      w[st][1] = lds4(row + D / 2 + sub * 8);
    }
#pragma unroll
    for (int st = 0; st < G::kSteps; ++st) f(st * G::kRowsStep + grp, w[st][0], w[st][1], true);
    return;
  }
  for (int base = 0; base < rows; base += G::kRowsStep) {
    const int r = base + grp;
    const bool ok = r < rows;
    uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
    if (ok) {
      w0 = lds4(buf + r * D + sub * 8);
      w1 = lds4(buf + r * D + D / 2 + sub * 8);
    }
    f(r, w0, w1, ok);
  }
}

// ROWS: units of up to kRowsCap slots keep 1/|k| and e^r in shared memory,
// longer ones in the device scratch.
template <int D, bool ROWS>
__global__ void __launch_bounds__(kThreads) redundancy_kernel(const RedArgs a) {
  using G = Geo<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem + RedSmem::ring;
  float* sacc = reinterpret_cast<float*>(smem + RedSmem::sacc);
  float* stot = reinterpret_cast<float*>(smem + RedSmem::stot);
  float* wsum = reinterpret_cast<float*>(smem + RedSmem::wsum);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RedSmem::full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + RedSmem::empty);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + RedSmem::abort_flag);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    // A timeout already recorded (by this launch or an unread earlier failure)
    // stops the CTA before it issues any copy: the result is invalid anyway.
    *abort_flag =
        (*reinterpret_cast<const volatile uint32_t*>(a.status) & KVC_STATUS_WAIT_TIMEOUT) ? 1 : 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---- producer: for every unit of this CTA, its chunks twice -------------
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
      int seq = 0;  // ring items issued
      for (int u = blockIdx.x; u < a.U && !*abort_flag; u += gridDim.x) {
        const int pad = unit_pad(a, u);
        const int n = a.T - pad;
        const int nch = (n + G::kChunkRows - 1) / G::kChunkRows;
        const uint16_t* src = a.k + (static_cast<size_t>(u) * a.T + pad) * D;
        for (int g = 0; g < 2 * nch && !*abort_flag; ++g, ++seq) {
          // pass B takes the chunks newest first: the most recently read are
          // the likeliest to still be in L2
          const int c = g < nch ? g : 2 * nch - 1 - g;
          const int s = seq % kStages;
          if (seq >= kStages &&
              !mbar_wait(&empty[s], static_cast<uint32_t>(seq / kStages - 1) & 1u, abort_flag,
                         a.status))
            break;
          const uint32_t bytes =
              static_cast<uint32_t>(min(G::kChunkRows, n - c * G::kChunkRows)) * D * 2;
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_copy(ring + static_cast<size_t>(s) * kChunkBytes,
                    src + static_cast<size_t>(c) * G::kChunkRows * D, bytes, &full[s],
                    g < nch ? keep : drop);
        }
      }
      // After an abort, let the copies in flight land before the shared memory
      // is released: only the last item of each slot can be outstanding.
      if (*abort_flag) {
        const uint64_t t0 = global_timer_ns();
        for (int s = 0; s < kStages && s < seq; ++s) {
          const int last = s + kStages * ((seq - 1 - s) / kStages);
          while (!mbar_test_sleep(&full[s], static_cast<uint32_t>(last / kStages) & 1u,
                                  kWaitSleepNs) &&
                 global_timer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    return;
  }

  // ---- consumers --------------------------------------------------------------
  const int grp = warp * G::kRpw + lane / G::kLpr;  // row group within a step
  const int sub = lane % G::kLpr;                   // dims [8 sub, +8) and [D/2 + 8 sub, +8)
  int slot = 0;                                     // ring slot of the next item
  uint32_t phase = 0;                               // its full-barrier phase parity
  // Wait for the next ring item, hand its buffer to f, free the slot.  The
  // first probe suspends until the copy lands (the usual case); the bounded
  // wait is the fallback.
  auto take = [&](auto&& f) {
    if (!mbar_test_sleep(&full[slot], phase, kWaitSleepNs))
      mbar_wait(&full[slot], phase, abort_flag, a.status);
    f(reinterpret_cast<const uint16_t*>(ring + static_cast<size_t>(slot) * kChunkBytes));
    __syncwarp();
    if (lane == 0 && !*abort_flag) mbar_arrive(&empty[slot]);
    if (++slot == kStages) {
      slot = 0;
      phase ^= 1u;
    }
  };

  int pad = blockIdx.x < a.U ? unit_pad(a, blockIdx.x) : 0;
  for (int u = blockIdx.x; u < a.U; u += gridDim.x) {
    // the next unit's padding, loaded now and used one unit later
    const int pad_next = u + static_cast<int>(gridDim.x) < a.U ? unit_pad(a, u + gridDim.x) : 0;
    const int n = a.T - pad;
    const int nch = (n + G::kChunkRows - 1) / G::kChunkRows;
    const size_t base = static_cast<size_t>(u) * a.T;
    float* rinv = ROWS ? reinterpret_cast<float*>(smem + RedSmem::rows) : a.rinv + base + pad;
    float* rexp = ROWS ? rinv + kRowsCap : a.rexp + base + pad;
    const float* srow = a.score + base + pad;
    float* sscore = rinv + 2 * kRowsCap;  // ROWS only
    if (ROWS)
      for (int i = tid; i < n; i += kConsumers) cp_async4(sscore + i, srow + i);

    // pass A: row norms and the per-lane sums of k^
    float2 acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = make_float2(0.f, 0.f);
    for (int c = 0; c < nch; ++c) {
      const int rows = min(G::kChunkRows, n - c * G::kChunkRows);
      take([&](const uint16_t* buf) {
        for_chunk_rows<D>(buf, rows, grp, sub, [&](int r, uint4 w0, uint4 w1, bool ok) {
          const float inv = pass_a_row<D>(w0, w1, acc);
          if (ok && sub == 0) rinv[c * G::kChunkRows + r] = inv;
        });
      });
    }
    // S: fold the row groups of each warp twice, then the warps in order
#pragma unroll
    for (int o = 16; o >= 8; o >>= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[j].x += __shfl_xor_sync(0xffffffffu, acc[j].x, o);
        acc[j].y += __shfl_xor_sync(0xffffffffu, acc[j].y, o);
      }
    if (lane < 8) {
      float* dst = sacc + (warp * G::kGroups + lane / G::kLpr) * D;
      *reinterpret_cast<float4*>(dst + sub * 8) = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
      *reinterpret_cast<float4*>(dst + sub * 8 + 4) = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
      *reinterpret_cast<float4*>(dst + D / 2 + sub * 8) =
          make_float4(acc[4].x, acc[4].y, acc[5].x, acc[5].y);
      *reinterpret_cast<float4*>(dst + D / 2 + sub * 8 + 4) =
          make_float4(acc[6].x, acc[6].y, acc[7].x, acc[7].y);
    }
    consumer_sync();
    if (tid < D) {
      float v = 0.f;
      for (int g = 0; g < kConsumerWarps * G::kGroups; ++g) v += sacc[g * D + tid];
      stot[tid] = v;
    }
    consumer_sync();
    float2 sv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = (j < 4 ? sub * 8 : D / 2 + sub * 8) + 2 * (j % 4);
      sv[j] = make_float2(stot[e], stot[e + 1]);
    }

    // pass B: e^{r_i}, r_i = (k_i . S / |k_i| - 1) / (n - 1)
    const float inv_nm1 = n >= 2 ? 1.0f / static_cast<float>(n - 1) : 0.f;
    float pe = 0.f;
    for (int cc = 0; cc < nch; ++cc) {
      const int c = nch - 1 - cc;  // the producer's pass-B order
      const int rows = min(G::kChunkRows, n - c * G::kChunkRows);
      take([&](const uint16_t* buf) {
        for_chunk_rows<D>(buf, rows, grp, sub, [&](int r, uint4 w0, uint4 w1, bool ok) {
          const float dot = pass_b_row<D>(w0, w1, sv);
          if (ok && sub == 0) {
            const int i = c * G::kChunkRows + r;
            const float inv = rinv[i];
            const float e = __expf(inv > 0.f ? fmaf(dot, inv, -1.0f) * inv_nm1 : 0.f);
            rexp[i] = e;
            pe += e;
          }
        });
      });
    }

    // sums of e^r and of the score over the unit (lanes, warps in order)
    const float* sc = srow;
    if (ROWS) {
      cp_async_wait_all();  // this thread's score copies (it reads only its own rows)
      sc = sscore;
    }
    float ps = 0.f;
    for (int i = tid; i < n; i += kConsumers) ps += sc[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      pe += __shfl_xor_sync(0xffffffffu, pe, o);
      ps += __shfl_xor_sync(0xffffffffu, ps, o);
    }
    if (lane == 0) {
      wsum[2 * warp] = pe;
      wsum[2 * warp + 1] = ps;
    }
    consumer_sync();  // also: every rexp store of the unit is visible below
    float z = 0.f, s_tot = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) {
      z += wsum[2 * w];
      s_tot += wsum[2 * w + 1];
    }
    const float inv_z = z > 0.f ? 1.0f / z : 0.f;
    const float w_i = a.sigma * (s_tot > 0.f ? 1.0f / s_tot : 0.f);
    const float w_r = (1.0f - a.sigma) * inv_z;
    float* sel = a.sel + base;
    float* red = a.red ? a.red + base : nullptr;
    for (int i = tid; i < n; i += kConsumers) {
      const float e = rexp[i];
      sel[pad + i] = fmaf(w_i, sc[i], -(w_r * e));
      if (red) red[pad + i] = e * inv_z;
    }
    for (int i = tid; i < pad; i += kConsumers) {
      sel[i] = -INFINITY;
      if (red) red[i] = 0.f;
    }
    consumer_sync();  // sacc, stot, wsum and the row values are rewritten by the next unit
    pad = pad_next;
  }
}

}  // namespace

cudaError_t launch_redundancy(const kvc_handle* h, const uint16_t* k, const float* score, int T,
                              const int32_t* pad, float* sel, float* red, cudaStream_t s) {
  const int D = h->dims.d;
  // scratch: the workspace's raw-usage and mass arrays, free once the segments
  // are cut (neither is read after step 4 of the event)
  RedArgs a{k, score, pad, sel, red, h->ws.usage, h->ws.mass, T, h->dims.B, h->dims.H,
            h->dims.U, h->cfg.redundancy_sigma, h->ws.status};
  const bool rows = T <= kRowsCap;
  const int smem = static_cast<int>(RedSmem::bytes(rows));
  void (*kern)(const RedArgs) =
      D == 64 ? (rows ? redundancy_kernel<64, true> : redundancy_kernel<64, false>)
              : (rows ? redundancy_kernel<128, true> : redundancy_kernel<128, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int fit = per_sm * h->num_sms;
  const int grid = fit < h->dims.U ? fit : h->dims.U;
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

size_t redundancy_smem_bytes(int, int T) { return RedSmem::bytes(T <= kRowsCap); }

}  // namespace kvc
