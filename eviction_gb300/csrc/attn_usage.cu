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
//   pass 1: rows on TMEM lanes (A = query rows, B = 256-slot chunks of K);
//           each epilogue thread owns one row and keeps an online max / sum;
//           out: -b_r (b_r = log2 of the row normaliser in the scaled log2
//           domain) and 1/Z'_r (the row's largest probability).
//   pass 2: slots on TMEM lanes (A = cached keys, B = 256-row chunks of Q);
//           each epilogue thread owns one slot and sums
//           exp2(scale*log2e*z - b_r) over the rows.
// Work item = one unit and a PAIR of 128-row A tiles: every 256-row B chunk
// that TMA brings in feeds one M128 x N256 MMA group per tile, which halves
// the operand traffic per FLOP.  Each tile has one 256-column TMEM
// accumulator; the two tiles alternate, so one tile's accumulator drains
// while the other's MMAs run.
//
// Persistent warp-specialised CTAs: warp 0 streams B chunks through a ring
// (TMA), warp 18 loads each tile slot's A tile (reloaded as soon as the slot's
// last MMA of an item completes) and, in pass 2, the item's row constants (one
// bulk copy), warp 1 issues tcgen05.mma, and 16 epilogue warps (warps 2-17:
// tile slot x column half x lane quarter) drain the accumulators, 64 columns
// at a time, releasing an accumulator once its last columns are in registers.
// At the end of an item the two column halves of a row (pass 1) or slot
// (pass 2) leave their partials in shared memory and go straight on; warp 19
// combines them and writes the results, so that the combination is not on the
// accumulator hand-off path.  Every wait is bounded.
#include <cmath>
#include <cstdio>

#include "attn_common.cuh"

namespace kvc {
namespace {

using namespace attn;

constexpr int kEpiWarps = 16;                     // tile slot x column half x lane quarter
constexpr int kLoaderWarp = 2 + kEpiWarps;        // A tiles / row constants
constexpr int kMergeWarp = kLoaderWarp + 1;       // combines the two column halves
constexpr int kThreads = 32 * (kMergeWarp + 1);   // B, MMA, epilogue, loader, merge
constexpr int BM = 128;         // A-operand rows per tile (TMEM lanes)
constexpr int BN = 256;         // B-operand rows per chunk (accumulator columns)
constexpr int kHalf = BN / 2;   // accumulator columns per epilogue column half
constexpr int kTiles = 2;       // A tiles per work item
constexpr int kMaxStages = 6;   // B ring depth limit
constexpr int kAccCols = kTiles * BN;  // one accumulator per tile slot: 512 columns
constexpr int kBarriers = 48;          // mbarrier slots in shared memory
// Shared memory of the per-item partials handed to the merge warp, two
// buffers (item parity) of pass 1 [tile slot][half][128 rows][max, sum] or
// pass 2 [tile slot][half][128 slots].
__host__ __device__ constexpr int part_bytes(int pass) {
  return 2 * kTiles * 2 * BM * (pass == 1 ? 8 : 4);
}

struct Params {
  int U, T, R, Rp, W, B, H;
  int n_items, n_tiles, n_pairs, n_stages, unit_major;
  int rb_shift;  // log2 of the pass-2 row-constant buffers (2, or 1 for the largest R)
  float scale_log2;
  const int32_t* pad;
  float* negb;    // [U][Rp] -b_r (pass 1 writes, pass 2 reads by bulk copy)
  float* pmax;    // [U][Rp] 1/Z'_r
  float* usage;   // [U][T]
  uint32_t* status;
};

struct Item {
  int u, pad, n_ch, c_start, c_end;  // chunks cover [c_start, c_end) of the B rows
  int tile[kTiles];   // tile index within the unit, -1 if absent
  int a_row[kTiles];  // first A row of the tile in the 2-D tensor view
  int b_row0;         // first B row of chunk 0
};

template <int PASS>
__device__ __forceinline__ Item decode(const Params& p, int item) {
  Item it;
  it.u = item / p.n_pairs;
  const int pair = item - it.u * p.n_pairs;
  const int b = (it.u / p.H) % p.B;
  it.pad = min(max(p.pad[b], 0), p.T);
  int n_present = 0;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    const int tile = pair * kTiles + t;
    bool present = tile < p.n_tiles;
    if (PASS == 2) present = present && (tile * BM + BM > it.pad);  // not all padding
    it.tile[t] = present ? tile : -1;
    it.a_row[t] = (PASS == 1) ? it.u * p.R + tile * BM : it.u * p.T + tile * BM;
    n_present += present ? 1 : 0;
  }
  if (PASS == 1) {
    it.c_start = (it.pad / BN) * BN;
    it.c_end = p.T;
    it.b_row0 = it.u * p.T + it.c_start;
  } else {
    it.c_start = 0;
    it.c_end = p.R;
    it.b_row0 = it.u * p.R;
  }
  it.n_ch = (it.pad < p.T && n_present) ? (it.c_end - it.c_start + BN - 1) / BN : 0;
  return it;
}

// Accumulator columns (= MMA N) of chunk ch: the rows left, rounded up to the
// 32-column block of the epilogue (a multiple of 16, as the MMA needs).
__device__ __forceinline__ int chunk_cols(const Item& it, int ch) {
  const int left = it.c_end - (it.c_start + ch * BN);
  return left >= BN ? BN : ((left + 31) & ~31);
}

// Shared-memory layout (byte offsets from the 1024-aligned base).
struct Layout {
  int a_bytes, b_bytes;  // per tile / per stage
  int off_b, off_bars, off_misc, off_rowb, off_part, total;
  __host__ __device__ Layout(int D, int n_stages, int rowb_bytes, int part_bytes) {
    a_bytes = BM * D * 2;
    b_bytes = BN * D * 2;
    off_b = kTiles * a_bytes;  // A: one buffer per tile slot
    off_bars = off_b + n_stages * b_bytes;
    off_misc = off_bars + kBarriers * 8;
    off_rowb = off_misc + 16;
    off_part = off_rowb + rowb_bytes;
    total = 1024 + off_part + part_bytes;
  }
};

// The k-th work item of this CTA, or -1 past the end.  With many units per SM
// each CTA takes whole units (all tile pairs of a unit back to back): no two SMs
// then fetch the same operand lines at the same moment, and the unit's operands
// stay in L2 for the CTA's next items.  With few units, items are interleaved
// across CTAs so that every SM has work.
__device__ __forceinline__ int cta_item(const Params& p, int k) {
  if (p.unit_major) {
    const int unit = blockIdx.x + (k / p.n_pairs) * gridDim.x;
    return unit < p.U ? unit * p.n_pairs + (k % p.n_pairs) : -1;
  }
  const int item = blockIdx.x + k * gridDim.x;
  return item < p.n_items ? item : -1;
}

template <int D, int PASS>
__global__ void __launch_bounds__(kThreads, 1)
    usage_kernel(const __grid_constant__ CUtensorMap map_a,
                 const __grid_constant__ CUtensorMap map_b, Params p) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
  const int rbf = (PASS == 2) ? rowb_floats(p.R) : 0;
  const Layout ly(D, p.n_stages, (rbf * 4) << p.rb_shift, part_bytes(PASS));
  const int NS = p.n_stages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle, as an offset from the shared
  // array so that the compiler keeps the shared address space
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* smem = smem_raw + ((1024u - mis) & 1023u);
  uint8_t* a_buf = smem;
  uint8_t* b_buf = smem + ly.off_b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ly.off_bars);
  uint64_t* full = bars;                      // [kMaxStages] B stage landed
  uint64_t* empty = bars + kMaxStages;        // [kMaxStages] B stage consumed
  uint64_t* afull = bars + 2 * kMaxStages;    // [kTiles] tile slot's A landed
  uint64_t* aempty = afull + kTiles;          // [kTiles] tile slot's A consumed
  uint64_t* accfull = aempty + kTiles;        // [kTiles] tile slot's accumulator written
  uint64_t* accempty = accfull + kTiles;      // [kTiles] ... drained (its 8 epilogue warps)
  uint64_t* done = accempty + kTiles;         // [1]
  uint64_t* rbfull = done + 1;                // [2] pass 2 row constants landed
  uint64_t* rbempty = rbfull + 2;             // [2] ... consumed (all epilogue warps)
  uint64_t* part_full = rbempty + 2;          // [2][kTiles] both halves' partials stored
  uint64_t* part_empty = part_full + 2 * kTiles;  // [2][kTiles] ... read by the merge warp
  static_assert(2 * kMaxStages + 4 * kTiles + 1 + 2 + 2 + 4 * kTiles <= kBarriers,
                "barrier area too small");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + ly.off_misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + ly.off_misc + 4);
  float* row_b_all = reinterpret_cast<float*>(smem + ly.off_rowb);
  float* part = reinterpret_cast<float*>(smem + ly.off_part);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&afull[t], 1);
      mbar_init(&aempty[t], 1);
      mbar_init(&accfull[t], 1);
      mbar_init(&accempty[t], 8);  // 4 lane quarters x 2 column halves
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&rbfull[b], 1);
      mbar_init(&rbempty[b], kEpiWarps);
    }
    for (int m = 0; m < 2 * kTiles; ++m) {
      mbar_init(&part_full[m], 8);  // 4 lane quarters x 2 column halves
      mbar_init(&part_empty[m], 1);
    }
    mbar_init(done, 1);
    *abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
  }
  if constexpr (PASS == 2) {
    // rows past the unit's constants never get copied: they must contribute 0
    for (int i = threadIdx.x; i < (rbf << p.rb_shift); i += kThreads) {
      const int r = i % rbf;
      if (r >= p.Rp) row_b_all[i] = -INFINITY;
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, kAccCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ B producer
    // (all lanes run the loop and wait converged; lane 0 issues the copies)
    {
      int b_iter = 0;
      bool ok = true;
      for (int kk = 0, item = cta_item(p, 0); ok && item >= 0; item = cta_item(p, ++kk)) {
        const Item it = decode<PASS>(p, item);
        for (int c = 0; c < it.n_ch; ++c) {
          const int s = b_iter % NS;
          if (!warp_wait(&empty[s], ((b_iter / NS) & 1) ^ 1, abort, p.status)) {
            ok = false;
            break;
          }
          ++b_iter;
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], ly.b_bytes);
            tma_load_3d(b_buf + s * ly.b_bytes, &map_b, 0, it.b_row0 + c * BN, 0, &full[s]);
          }
        }
      }
      // drain: every issued copy must land before the CTA may exit
      for (int i = (b_iter > NS ? b_iter - NS : 0); i < b_iter; ++i)
        drain_wait(&full[i % NS], (i / NS) & 1, p.status);
    }
    __syncwarp();
  } else if (warp == kLoaderWarp) {
    // ------------------------------------------- A tiles and row constants
    // A tile slot t is reloaded as soon as the slot's last MMA of the previous
    // item has completed, while the other slot's MMAs still run.  (All lanes
    // run the loop; lane 0 issues the copies.)
    {
      int a_cnt[kTiles] = {0, 0};
      int rb_iter = 0;
      bool ok = true;
      for (int kk = 0, item = cta_item(p, 0); ok && item >= 0; item = cta_item(p, ++kk)) {
        const Item it = decode<PASS>(p, item);
        if (it.n_ch == 0) continue;
#pragma unroll
        for (int t = 0; t < kTiles; ++t) {
          if (!ok || it.tile[t] < 0) continue;
          if (!warp_wait(&aempty[t], (a_cnt[t] & 1) ^ 1, abort, p.status)) {
            ok = false;
            continue;
          }
          ++a_cnt[t];
          if (lane == 0) {
            mbar_arrive_expect_tx(&afull[t], ly.a_bytes);
            // one box: 128 rows x all 64-element K blocks, K block outermost
            tma_load_3d(a_buf + t * ly.a_bytes, &map_a, 0, it.a_row[t], 0, &afull[t]);
          }
        }
        if (ok && PASS == 2) {
          const int rb = rb_iter & p.rb_shift;
          if (!warp_wait(&rbempty[rb], ((rb_iter >> p.rb_shift) & 1) ^ 1, abort, p.status)) break;
          ++rb_iter;
          if (lane == 0) {
            mbar_arrive_expect_tx(&rbfull[rb], p.Rp * 4);
            bulk_load(row_b_all + rb * rbf, p.negb + static_cast<size_t>(it.u) * p.Rp,
                      p.Rp * 4, &rbfull[rb]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kTiles; ++t)
        if (a_cnt[t] > 0) drain_wait(&afull[t], (a_cnt[t] - 1) & 1, p.status);
      const int n_rb = 1 << p.rb_shift;
      for (int i = (rb_iter > n_rb ? rb_iter - n_rb : 0); i < rb_iter; ++i)
        drain_wait(&rbfull[i & p.rb_shift], (i >> p.rb_shift) & 1, p.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (all lanes run the loop and wait converged; lane 0 issues MMAs and commits)
    {
      const uint32_t a_base = smem_u32(a_buf), b_base = smem_u32(b_buf);
      int a_cnt[kTiles] = {0, 0};  // A loads consumed per tile slot
      int kt[kTiles] = {0, 0};     // accumulator fills per tile slot
      int b_iter = 0;
      bool ok = true;
      for (int kk = 0, item = cta_item(p, 0); ok && item >= 0; item = cta_item(p, ++kk)) {
        const Item it = decode<PASS>(p, item);
        for (int c = 0; ok && c < it.n_ch; ++c) {
          const int s = b_iter % NS;
          if (!warp_wait(&full[s], (b_iter / NS) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          const uint32_t idesc = idesc_bf16_f32(BM, chunk_cols(it, c));
          const uint32_t b_tile = b_base + s * ly.b_bytes;
#pragma unroll
          for (int t = 0; t < kTiles; ++t) {
            if (!ok || it.tile[t] < 0) continue;
            if (c == 0) {
              if (!warp_wait(&afull[t], a_cnt[t] & 1, abort, p.status)) {
                ok = false;
                continue;
              }
              ++a_cnt[t];
            }
            if (!warp_wait(&accempty[t], (kt[t] & 1) ^ 1, abort, p.status)) {
              ok = false;
              continue;
            }
            tc_fence_after();
            const uint32_t a_tile = a_base + t * ly.a_bytes;
            if (lane == 0) {
#pragma unroll
              for (int k = 0; k < D / 16; ++k) {
                const int kb = k / 4, kq = k % 4;
                const uint64_t ad = sw128_desc(a_tile + kb * BM * 128 + kq * 32);
                const uint64_t bd = sw128_desc(b_tile + kb * BN * 128 + kq * 32);
                mma_bf16(tmem + t * BN, ad, bd, idesc, k > 0 ? 1u : 0u);
              }
              mma_commit(&accfull[t]);
              if (c == it.n_ch - 1) mma_commit(&aempty[t]);  // slot's A free for the next item
            }
            __syncwarp();
            ++kt[t];
          }
          if (!ok) break;
          if (lane == 0) mma_commit(&empty[s]);
          ++b_iter;
        }
      }
      if (lane == 0) mma_commit(done);
      __syncwarp();
      drain_wait(done, 0, p.status);
    }
    __syncwarp();
  } else if (warp == kMergeWarp) {
    // ------------------------------------------------------------ merge
    // Combines the two column halves' partials of every item and tile slot
    // (handed over in shared memory) and writes the results, off the
    // epilogue's path: lane i takes rows (pass 1) or slots (pass 2) i + 32j.
    const float c = p.scale_log2;
    int n_merge[kTiles] = {0, 0};
    bool ok = true;
    for (int kk = 0, item = cta_item(p, 0); ok && item >= 0; item = cta_item(p, ++kk)) {
      const Item it = decode<PASS>(p, item);
      if (PASS == 2 && it.n_ch == 0) continue;  // the epilogue skips these items
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        const int tile = it.tile[t];
        if (!ok || tile < 0) continue;
        const int pb = (n_merge[t] & 1) * kTiles + t;
        if (!warp_wait(&part_full[pb], (n_merge[t] >> 1) & 1, abort, p.status)) {
          ok = false;
          continue;
        }
        ++n_merge[t];
        float a0[4], a1[4], b0[4], b1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int lrow = lane + 32 * j;
          if (PASS == 1) {
            const float* h0 = part + (pb * 2 + 0) * BM * 2;
            const float* h1 = part + (pb * 2 + 1) * BM * 2;
            a0[j] = h0[2 * lrow];
            b0[j] = h0[2 * lrow + 1];
            a1[j] = h1[2 * lrow];
            b1[j] = h1[2 * lrow + 1];
          } else {
            a0[j] = part[(pb * 2 + 0) * BM + lrow];
            a1[j] = part[(pb * 2 + 1) * BM + lrow];
            b0[j] = b1[j] = 0.f;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&part_empty[pb]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int lrow = lane + 32 * j;
          if (PASS == 1) {
            const int r = tile * BM + lrow;
            const int qpos = p.T - p.W + (r % p.W);
            const bool row_valid = (r < p.R) && (qpos >= it.pad) && (it.n_ch > 0);
            if (r < p.Rp) {
              // (max, sum) of columns [0, 128) and [128, 256) of every chunk
              const float mz = a0[j], sum = b0[j], m2 = a1[j], s2 = b1[j];
              const float M = fmaxf(mz, m2);
              const float S = (M == -INFINITY)
                                  ? 0.f
                                  : sum * ex2((mz - M) * c) + s2 * ex2((m2 - M) * c);
              const bool has = row_valid && S > 0.f;
              const size_t o = static_cast<size_t>(it.u) * p.Rp + r;
              p.negb[o] = has ? -(M * c + log2f(S)) : -INFINITY;
              p.pmax[o] = has ? 1.0f / S : 0.f;
            }
          } else {
            const int pos = tile * BM + lrow;
            if (pos >= it.pad && pos < p.T)
              p.usage[static_cast<size_t>(it.u) * p.T + pos] = a0[j] + a1[j];
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp 2 + 4g + i (g = 0..3): tile slot g & 1, column half g >> 1 of the
    // slot's accumulator; lane quarter warp % 4 (the TMEM lanes a warp may
    // access).  Four epilogue warps per SM sub-partition hide each other's
    // TMEM-load and barrier latency.  At the end of an item both halves store
    // their partial of each row (pass 1) or slot (pass 2) in shared memory for
    // the merge warp and go on with the next item.
    const int grp = (warp - 2) >> 2;
    const int wg = grp & 1;            // tile slot
    const int half = grp >> 1;         // accumulator columns [128 half, 128 half + 128)
    const int quarter = warp & 3;
    const int lrow = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                            static_cast<uint32_t>(wg * BN + half * kHalf);
    const float c = p.scale_log2;
    int k = 0;        // accumulator fills of this tile slot consumed
    int n_merge = 0;  // items of this tile slot handed to the merge warp
    int rb_iter = 0;
    bool ok = true;
    auto release = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[wg]);
    };
    for (int kk = 0, item = cta_item(p, 0); ok && item >= 0; item = cta_item(p, ++kk)) {
      const Item it = decode<PASS>(p, item);
      const int tile = wg == 0 ? it.tile[0] : it.tile[1];
      if (PASS == 1) {
        const int r = (tile >= 0 ? tile : 0) * BM + lrow;
        const int qpos = p.T - p.W + (r % p.W);
        const bool row_valid = tile >= 0 && (r < p.R) && (qpos >= it.pad) && (it.n_ch > 0);
        // once per item: every row valid, and the warp's smallest query slot
        // (a chunk's half is all visible to every row when it lies in
        // [pad, qmin]: the per-fill test is then a few uniform compares)
        const bool all_valid = __all_sync(0xffffffffu, row_valid);
        const int qmin = __reduce_min_sync(0xffffffffu, qpos);
        const int n_full = (it.c_end - it.c_start) / BN;  // chunks of BN columns
        float mz = -INFINITY, sum = 0.f;  // max in raw logit units, sum rel. to it
        for (int ch = 0; tile >= 0 && ch < it.n_ch; ++ch) {
          if (!warp_wait(&accfull[wg], k & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int c0 = it.c_start + ch * BN;
          const int p0 = c0 + half * kHalf;
          // every row of the warp sees all of this warp's 128 columns
          const bool fast = all_valid && it.pad <= p0 && qmin >= p0 + kHalf - 1 &&
                            (ch < n_full || chunk_cols(it, ch) - half * kHalf >= kHalf);
          uint32_t v[2][32];
          float bmx[2];
          __syncwarp();
          if (fast) {
            // whole half, every row sees every column: two 64-column steps,
            // release after the second load
            load2(t_lane, true, v, bmx);
            tmem_ld_wait();
            row_pair(v, bmx, c, mz, sum);
            __syncwarp();
            load2(t_lane + 64, true, v, bmx);
            tmem_ld_wait();
            release();
            row_pair(v, bmx, c, mz, sum);
          } else {
            // masked or partial chunk, one 32-column block at a time: a block
            // that no row of the warp sees is skipped, one that every row sees
            // in full takes the unmasked arithmetic
            const int n_cols = chunk_cols(it, ch);
            const int nb = max(0, min(4, (n_cols - half * kHalf) / 32));  // this warp's blocks
            const int lo = max(it.pad, c0), hi = min(qpos, c0 + n_cols - 1);
            for (int b = 0; b < nb; ++b) {
              const int pb0 = p0 + 32 * b;
              const bool all = __all_sync(0xffffffffu, lo <= pb0 && hi >= pb0 + 31);
              const bool some = __any_sync(0xffffffffu, min(hi, pb0 + 31) >= max(lo, pb0));
              __syncwarp();
              if (all) {
                tmem_ld32_max(t_lane + 32 * b, v[0], bmx[0]);
                tmem_ld_wait();
                if (b == nb - 1) release();
                row_block<true>(v[0], bmx[0], pb0, lo, hi, c, mz, sum);
              } else if (some) {
                tmem_ld32(t_lane + 32 * b, v[0]);
                tmem_ld_wait();
                if (b == nb - 1) release();
                row_block<false>(v[0], -INFINITY, pb0, lo, hi, c, mz, sum);
              } else if (b == nb - 1) {
                release();
              }
            }
            if (nb == 0) release();
          }
          ++k;
        }
        if (!ok) break;
        if (tile < 0) continue;
        // partial (max, sum) of this half's columns of every chunk
        const int pb = (n_merge & 1) * kTiles + wg;
        if (!warp_wait(&part_empty[pb], ((n_merge >> 1) & 1) ^ 1, abort, p.status)) break;
        *reinterpret_cast<float2*>(part + ((pb * 2 + half) * BM + lrow) * 2) = make_float2(mz, sum);
        __syncwarp();
        if (lane == 0) mbar_arrive(&part_full[pb]);
        ++n_merge;
      } else {
        if (it.n_ch == 0) continue;
        // the unit's negated row constants (bulk copy by the loader warp)
        const int rb = rb_iter & p.rb_shift;
        if (!warp_wait(&rbfull[rb], (rb_iter >> p.rb_shift) & 1, abort, p.status)) break;
        ++rb_iter;
        const float* row_b = row_b_all + rb * rbf;
        const int pos = (tile >= 0 ? tile : 0) * BM + lrow;
        const bool pos_valid = tile >= 0 && (pos >= it.pad) && (pos < p.T);
        const bool fast = __all_sync(0xffffffffu, pos_valid && (pos <= p.T - p.W));
        const int jmin = pos - (p.T - p.W);  // rows with j >= jmin see pos
        const int n_full = (it.c_end - it.c_start) / BN;  // chunks of BN query rows
        float2 acc = make_float2(0.f, 0.f);
        for (int ch = 0; tile >= 0 && ch < it.n_ch; ++ch) {
          if (!warp_wait(&accfull[wg], k & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int r0 = ch * BN + half * kHalf;  // first query row of this warp's columns
          uint32_t v[2][32];
          float bmx[2];
          __syncwarp();
          if (fast && (ch < n_full || chunk_cols(it, ch) - half * kHalf >= kHalf)) {
            // whole half, every query row sees the slot
            load2(t_lane, false, v, bmx);
            tmem_ld_wait();
            slot_pair(v, row_b + r0, c, acc);
            __syncwarp();
            load2(t_lane + 64, false, v, bmx);
            tmem_ld_wait();
            release();
            slot_pair(v, row_b + r0 + 64, c, acc);
          } else {
            // one 32-row block at a time; with windows of whole blocks, a block
            // of rows that no slot of the warp is seen by is skipped and one
            // whose rows see every slot takes the unmasked arithmetic
            const int n_cols = chunk_cols(it, ch);
            const int nb = max(0, min(4, (n_cols - half * kHalf) / 32));
            for (int b = 0; b < nb; ++b) {
              const int rb0 = r0 + 32 * b;
              bool all = false, some = true;
              if (p.W % 32 == 0) {
                const int j0 = rb0 % p.W;  // the block's window indices j0 .. j0+31
                all = __all_sync(0xffffffffu, j0 >= jmin);
                some = __any_sync(0xffffffffu, j0 + 31 >= jmin);
              }
              __syncwarp();
              if (all) {
                tmem_ld32(t_lane + 32 * b, v[0]);
                tmem_ld_wait();
                if (b == nb - 1) release();
                slot_block<true>(v[0], row_b + rb0, rb0, p.W, jmin, c, acc);
              } else if (some) {
                tmem_ld32(t_lane + 32 * b, v[0]);
                tmem_ld_wait();
                if (b == nb - 1) release();
                slot_block<false>(v[0], row_b + rb0, rb0, p.W, jmin, c, acc);
              } else if (b == nb - 1) {
                release();
              }
            }
            if (nb == 0) release();
          }
          ++k;
        }
        // every epilogue warp releases the row constants, tile or no tile
        __syncwarp();
        if (lane == 0) mbar_arrive(&rbempty[rb]);
        if (!ok) break;
        if (tile < 0) continue;
        // partial usage over the query rows of this half's columns of every chunk
        const int pb = (n_merge & 1) * kTiles + wg;
        if (!warp_wait(&part_empty[pb], ((n_merge >> 1) & 1) ^ 1, abort, p.status)) break;
        part[(pb * 2 + half) * BM + lrow] = acc.x + acc.y;
        __syncwarp();
        if (lane == 0) mbar_arrive(&part_full[pb]);
        ++n_merge;
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

// 3-D view of a [rows][d] bf16 tensor: x = 64 elements of a K block (128 B),
// y = row (stride d*2 B), z = K block (stride 128 B).  A box of
// 64 x box_rows x d/64 lands in shared memory as d/64 consecutive
// [box_rows][128 B] blocks, each with the 128-byte swizzle -- the K-major
// layout the MMA descriptors expect -- in a single TMA operation.  Rows past
// the end of the tensor read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows,
              std::string* err) {
  EncodeTiledFn enc = get_encode(err);
  if (!enc) return false;
  cuuint64_t dims[3] = {64, rows, static_cast<cuuint64_t>(d / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(d / 64)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) *err = "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")";
    return false;
  }
  return true;
}

}  // namespace

// The usage kernels' 3-D tensor-map view (shared with the CTA-pair kernel).
bool make_usage_map(CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows,
                    std::string* err) {
  return make_map(m, base, rows, d, box_rows, err);
}

namespace {

int smem_optin() {
  static int v = 0;
  if (!v) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      v = 227 * 1024;
  }
  return v;
}

// The deepest B ring (at least 2 stages) that fits next to the A tiles.
int pick_stages(int D, int rowb_bytes, int part_bytes) {
  for (int s = kMaxStages; s >= 2; --s)
    if (Layout(D, s, rowb_bytes, part_bytes).total <= smem_optin()) return s;
  return 0;
}

template <int D>
cudaError_t launch_d(const kvc_handle* h, const UsageArgs& a, int pass, cudaStream_t s,
                     std::string* err) {
  const Dims& dm = h->dims;
  const uint64_t q_rows = static_cast<uint64_t>(dm.U) * dm.R;
  const uint64_t k_rows = static_cast<uint64_t>(dm.U) * a.T;
  // pass 1: A = query tiles (128 rows), B = key chunks (256 rows);
  // pass 2: A = key tiles, B = query chunks
  CUtensorMap map_a, map_b;
  if (!make_map(&map_a, pass == 1 ? a.q : a.k, pass == 1 ? q_rows : k_rows, D, BM, err) ||
      !make_map(&map_b, pass == 1 ? a.k : a.q, pass == 1 ? k_rows : q_rows, D, BN, err))
    return cudaErrorInvalidValue;

  Params p;
  p.U = dm.U;
  p.T = a.T;
  p.R = dm.R;
  p.Rp = round4(dm.R);
  p.W = dm.W;
  p.B = dm.B;
  p.H = dm.H;
  p.scale_log2 = a.scale_log2;
  p.pad = a.pad;
  p.negb = h->ws.negb;
  p.pmax = h->ws.pmax;
  p.usage = h->ws.usage;
  p.status = h->ws.status;

  const int rbf = (pass == 2) ? rowb_floats(dm.R) : 0;
  p.rb_shift = Layout(D, 2, 2 * rbf * 4, part_bytes(pass)).total <= smem_optin() ? 1 : 0;
  p.n_stages = pick_stages(D, (rbf * 4) << p.rb_shift, part_bytes(pass));
  if (p.n_stages == 0) {
    if (err) *err = "attention kernel does not fit in shared memory";
    return cudaErrorInvalidValue;
  }
  const size_t smem = Layout(D, p.n_stages, (rbf * 4) << p.rb_shift, part_bytes(pass)).total;
  p.n_tiles = (pass == 1) ? (dm.R + BM - 1) / BM : (a.T + BM - 1) / BM;
  p.n_pairs = (p.n_tiles + kTiles - 1) / kTiles;
  p.n_items = dm.U * p.n_pairs;
  p.unit_major = dm.U >= 2 * h->num_sms ? 1 : 0;
  const int grid = p.n_items < h->num_sms ? p.n_items : h->num_sms;
  cudaError_t e;
  if (pass == 1) {
    e = cudaFuncSetAttribute(usage_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    usage_kernel<D, 1><<<grid, kThreads, smem, s>>>(map_a, map_b, p);
  } else {
    e = cudaFuncSetAttribute(usage_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    usage_kernel<D, 2><<<grid, kThreads, smem, s>>>(map_a, map_b, p);
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

// Shared memory the attention kernels need with their shallowest ring (2 stages)
// and a single row-constant buffer.
size_t attention_usage_smem_bytes(int d, int R) {
  const int p1 = Layout(d, 2, 0, part_bytes(1)).total;
  const int p2 = Layout(d, 2, rowb_floats(R) * 4, part_bytes(2)).total;
  return static_cast<size_t>(p1 > p2 ? p1 : p2);
}

int attention_row_stride(int R) { return round4(R); }

}  // namespace kvc
