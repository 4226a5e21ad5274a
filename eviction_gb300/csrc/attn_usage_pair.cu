// attn_usage_pair.cu -- the window attention usage on CTA pairs (cta_group::2).
//
// Computes exactly what attn_usage.cu computes ("Adaptive Mass-Segmented KV
// Compression for Long-Form Reasoning", Method, Key design 1; "SkipKV: ...", A2
// token importance score): pass 1 the per-row softmax normalisers of the window
// queries' QK^T, pass 2 the per-slot sums of the normalised probabilities.
//
// Why pairs: on one SM the M128 x N256 accumulators fill all 512 TMEM columns
// twice over (two tile slots), so only one accumulator can drain while the
// other fills, and the drain (about as long as one fill's MMAs plus the
// hand-off) leaves the tensor pipe idle.  Two SMs sharing one M256 x N128 MMA
// read the same operand bytes per FLOP as one SM's M128 x N256 (each SM holds
// its 128 A rows and half of the 128 B rows), while each SM's accumulator is
// only 128 columns wide: four accumulators per SM, three fills of slack for
// each drain.
//
// A cluster of two CTAs on one TPC; rank 0 leads.  Per CTA:
//   warp 0      loader: per item this CTA's 128-row A tile (two buffers, so
//               that the next item's tile lands while this item's MMAs run)
//               and, in pass 2, the item's row constants, then its 64 rows of
//               each 128-row B chunk; the completions of A and B are counted
//               on the leader's barriers;
//   warps 1, 18 TMEM allocation (warp 1 of both CTAs, 512 columns at the same
//               address); MMA issue in the leader only (tcgen05.mma.cta_group::2,
//               M256 N128), warp 1 the even fills and warp 18 the odd ones: one
//               thread alone cannot issue a fill's eight MMAs, test its barriers
//               and commit within the 700 cycles the fill takes; commits
//               multicast to both CTAs;
//   warps 2-17  epilogue: group g = 0..3 drains accumulator g (fills g, g+4,
//               ...), lane quarter q = warp % 4; releases on the leader's
//               `accempty` (a cluster-scope arrive);
//   warp 19     merge: combines the four groups' partials of each row (pass 1)
//               or slot (pass 2) and writes the results.
// Work item = one unit and one PAIR of 128-row A tiles (rank r owns tile
// 2*pair + r).  An absent tile (past the unit's rows, or all padding) is still
// loaded (the MMA covers both halves) and drained, never used.  Every wait is
// bounded; every thread of both CTAs meets at the final cluster barrier, so no
// CTA exits while its peer may still signal it.
#include <cmath>
#include <cstdio>

#include "attn_common.cuh"

namespace kvc {
namespace {

using namespace attn;

constexpr int kGroups = 4;                        // epilogue groups = accumulators
constexpr int kEpiWarps = 4 * kGroups;            // group x lane quarter
constexpr int kMma2Warp = 2 + kEpiWarps;  // issues the odd fills (warp 1 the even ones)
constexpr int kMergeWarp = kMma2Warp + 1;
constexpr int kThreads = 32 * (kMergeWarp + 1);
constexpr int BM = 128;           // A rows per CTA (TMEM lanes); the pair's MMA has M = 256
constexpr int BN = 128;           // B rows per fill (MMA N = accumulator columns)
constexpr int BNH = BN / 2;       // B rows each CTA of the pair holds per fill
constexpr int kAccCols = kGroups * BN;  // 512
constexpr int kABufs = 2;
constexpr int kMaxStages = 8;
constexpr int kBarriers = 64;
constexpr uint16_t kBoth = 0x3;   // multicast mask: ranks 0 and 1
// B stages: kGroups (a stage is released by its fill's accumulator commit) or
// 2 * kGroups (released by a commit of its own, one more per fill).
#ifndef KVC_PAIR_STAGES
#define KVC_PAIR_STAGES 4
#endif
constexpr int kStages = KVC_PAIR_STAGES;
static_assert(kStages == 4 || kStages == 8, "4 or 8 B stages");

// Which waits poll instead of suspending: 0 none, 1 the MMA issuer, 2 also
// the producers, 3 every role.
#ifndef KVC_PAIR_POLL
#define KVC_PAIR_POLL 0
#endif
constexpr int kPoll = KVC_PAIR_POLL;

template <int LEVEL>
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                      uint32_t* status) {
  return kPoll >= LEVEL ? mbar_wait_poll(bar, parity, abort, status)
                        : mbar_wait(bar, parity, abort, status);
}

// Warp-uniform wait of the epilogue and merge warps: all lanes wait converged
// and vote on the outcome.
__device__ __forceinline__ bool pwait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           uint32_t* status) {
  const bool ok = pwait<3>(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

// Per-item partials of the four groups handed to the merge warp, two buffers
// (item parity): pass 1 [parity][group][128 rows][max, sum], pass 2
// [parity][group][128 slots].
__host__ __device__ constexpr int pair_part_bytes(int pass) {
  return 2 * kGroups * BM * (pass == 1 ? 8 : 4);
}

struct PairParams {
  int U, T, R, Rp, W, B, H;
  int n_items, n_tiles, n_pairs, n_stages, unit_major;
  int rb_shift;
  float scale_log2;
  const int32_t* pad;
  float* negb;
  float* pmax;
  float* usage;
  uint32_t* status;
};

struct PairLayout {
  int a_bytes, b_bytes;
  int off_b, off_bars, off_misc, off_rowb, off_part, total;
  __host__ __device__ PairLayout(int D, int n_stages, int rowb_bytes, int part_bytes) {
    a_bytes = BM * D * 2;
    b_bytes = BNH * D * 2;
    off_b = kABufs * a_bytes;
    off_bars = off_b + n_stages * b_bytes;
    off_misc = off_bars + kBarriers * 8;
    off_rowb = off_misc + 16;
    off_part = off_rowb + rowb_bytes;
    total = 1024 + off_part + part_bytes;
  }
};

struct PairItem {
  int u, pad, n_ch, c_start, c_end;
  int tile;    // this CTA's tile within the unit, -1 if absent
  int a_row;   // first A row of this CTA's tile in the 2-D view (a real row range even
               // when absent: loaded, never used)
  int b_row0;  // first B row of chunk 0
};

template <int PASS>
__device__ __forceinline__ PairItem decode_pair(const PairParams& p, int item, int rank) {
  PairItem it;
  it.u = item / p.n_pairs;
  const int pair = item - it.u * p.n_pairs;
  const int b = (it.u / p.H) % p.B;
  it.pad = min(max(p.pad[b], 0), p.T);
  bool any = false;
  it.tile = -1;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int tile = pair * 2 + t;
    bool present = tile < p.n_tiles;
    if (PASS == 2) present = present && (tile * BM + BM > it.pad);
    any = any || present;
    if (t == rank && present) it.tile = tile;
  }
  it.a_row = (PASS == 1 ? it.u * p.R : it.u * p.T) + (pair * 2 + rank) * BM;
  if (PASS == 1) {
    it.c_start = (it.pad / BN) * BN;
    it.c_end = p.T;
    it.b_row0 = it.u * p.T + it.c_start;
  } else {
    it.c_start = 0;
    it.c_end = p.R;
    it.b_row0 = it.u * p.R;
  }
  it.n_ch = (it.pad < p.T && any) ? (it.c_end - it.c_start + BN - 1) / BN : 0;
  return it;
}

// Valid B rows of chunk ch rounded up to the 32-column block of the epilogue.
__device__ __forceinline__ int pair_chunk_cols(const PairItem& it, int ch) {
  const int left = it.c_end - (it.c_start + ch * BN);
  return left >= BN ? BN : ((left + 31) & ~31);
}

// The k-th work item of this CTA pair, or -1 past the end (both CTAs of a pair
// walk the same items).
__device__ __forceinline__ int pair_item(const PairParams& p, int k) {
  const int cid = blockIdx.x / 2, nc = gridDim.x / 2;
  if (p.unit_major) {
    const int unit = cid + (k / p.n_pairs) * nc;
    return unit < p.U ? unit * p.n_pairs + (k % p.n_pairs) : -1;
  }
  const int item = cid + k * nc;
  return item < p.n_items ? item : -1;
}

template <int D, int PASS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    usage_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b, PairParams p) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
  const int rbf = (PASS == 2) ? rowb_floats(p.R) : 0;
  const PairLayout ly(D, p.n_stages, (rbf * 4) << p.rb_shift, pair_part_bytes(PASS));
  const int NS = p.n_stages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* smem = smem_raw + ((1024u - mis) & 1023u);
  uint8_t* a_buf = smem;
  uint8_t* b_buf = smem + ly.off_b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ly.off_bars);
  uint64_t* full = bars;                          // [kMaxStages] leader: both B halves landed
  uint64_t* empty = full + kMaxStages;            // [kMaxStages] B stage consumed (8 stages)
  uint64_t* afull = empty + kMaxStages;           // [kABufs] leader: both A tiles landed
  uint64_t* aempty = afull + kABufs;              // [kABufs] this CTA's A tile consumed
  uint64_t* accfull = aempty + kABufs;            // [kGroups] accumulator written
  uint64_t* accempty = accfull + kGroups;         // [kGroups] leader: drained in both CTAs
  uint64_t* done = accempty + kGroups;            // [1] leader: every MMA finished
  uint64_t* rbfull = done + 1;                    // [2] pass 2 row constants landed
  uint64_t* rbempty = rbfull + 2;                 // [2] ... consumed (all epilogue warps)
  uint64_t* part_full = rbempty + 2;              // [2] all groups' partials stored
  uint64_t* part_empty = part_full + 2;           // [2] ... read by the merge warp
  static_assert(2 * kMaxStages + 2 * kABufs + 2 * kGroups + 1 + 2 + 2 + 2 + 2 <= kBarriers,
                "barrier area too small");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + ly.off_misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + ly.off_misc + 4);
  float* row_b_all = reinterpret_cast<float*>(smem + ly.off_rowb);
  float* part = reinterpret_cast<float*>(smem + ly.off_part);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);   // the leader's producer arrives (and expects both halves)
      mbar_init(&empty[s], 1);  // one multicast commit
    }
    for (int b = 0; b < kABufs; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 2);  // one multicast commit from each MMA thread
    }
    for (int g = 0; g < kGroups; ++g) {
      mbar_init(&accfull[g], 1);
      mbar_init(&accempty[g], 2 * 4);  // 4 lane quarters x 2 CTAs
    }
    mbar_init(done, 2);  // each MMA thread
    for (int b = 0; b < 2; ++b) {
      mbar_init(&rbfull[b], 1);
      mbar_init(&rbempty[b], kEpiWarps);
      mbar_init(&part_full[b], kEpiWarps);
      mbar_init(&part_empty[b], 1);
    }
    *abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
  }
  if constexpr (PASS == 2) {
    for (int i = threadIdx.x; i < (rbf << p.rb_shift); i += kThreads) {
      const int r = i % rbf;
      if (r >= p.Rp) row_b_all[i] = -INFINITY;
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kAccCols);  // warp 1 of BOTH CTAs
  tc_fence_before();
  cluster_sync();  // barrier inits and the allocation visible to both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the leader's barriers as shared::cluster addresses
  const uint32_t full_l = map_to_rank(smem_u32(full), 0);
  const uint32_t afull_l = map_to_rank(smem_u32(afull), 0);
  const uint32_t accempty_l = map_to_rank(smem_u32(accempty), 0);

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      int b_iter = 0;  // = the fill a B load feeds
      int a_cnt = 0, rb_iter = 0;
      bool ok = true;
      for (int kk = 0, item = pair_item(p, 0); ok && item >= 0; item = pair_item(p, ++kk)) {
        const PairItem it = decode_pair<PASS>(p, item, rank);
        if (it.n_ch == 0) continue;
        // this CTA's A tile into buffer a_cnt % 2, free once both MMA threads'
        // work on the item two before is done
        const int ab = a_cnt % kABufs;
        if (!pwait<2>(&aempty[ab], ((a_cnt / kABufs) & 1) ^ 1, abort, p.status)) break;
        ++a_cnt;
        if (leader) mbar_arrive_expect_tx(&afull[ab], 2 * ly.a_bytes);
        tma_load_3d_pair(a_buf + ab * ly.a_bytes, &map_a, 0, it.a_row, 0, afull_l + 8u * ab);
        if (PASS == 2) {
          const int rb = rb_iter & p.rb_shift;
          if (!pwait<2>(&rbempty[rb], ((rb_iter >> p.rb_shift) & 1) ^ 1, abort, p.status))
            break;
          ++rb_iter;
          mbar_arrive_expect_tx(&rbfull[rb], p.Rp * 4);
          bulk_load(row_b_all + rb * rbf, p.negb + static_cast<size_t>(it.u) * p.Rp, p.Rp * 4,
                    &rbfull[rb]);
        }
        for (int c = 0; c < it.n_ch; ++c) {
          // stage s is free once the fill 4 earlier (same stage, same
          // accumulator) has completed: that fill's accfull phase
          const int s = b_iter % NS;
          if (!pwait<2>(kStages == kGroups ? &accfull[s] : &empty[s], ((b_iter / NS) & 1) ^ 1,
                        abort, p.status)) {
            ok = false;
            break;
          }
          ++b_iter;
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * ly.b_bytes);
          tma_load_3d_pair(b_buf + s * ly.b_bytes, &map_b, 0,
                           it.b_row0 + c * BN + static_cast<int>(rank) * BNH, 0,
                           full_l + 8u * s);
        }
      }
      // drain: both halves of every copy in flight land before either CTA may
      // exit (the peer waits at the final cluster barrier)
      if (leader) {
        for (int i = (b_iter > NS ? b_iter - NS : 0); i < b_iter; ++i)
          drain_wait(&full[i % NS], (i / NS) & 1, p.status);
        for (int i = (a_cnt > kABufs ? a_cnt - kABufs : 0); i < a_cnt; ++i)
          drain_wait(&afull[i % kABufs], (i / kABufs) & 1, p.status);
      }
      const int n_rb = 1 << p.rb_shift;
      for (int i = (rb_iter > n_rb ? rb_iter - n_rb : 0); i < rb_iter; ++i)
        drain_wait(&rbfull[i & p.rb_shift], (i >> p.rb_shift) & 1, p.status);
    }
    __syncwarp();
  } else if (warp == 1 || warp == kMma2Warp) {
    // ------------------------------------------------ MMA issuers (leader only)
    // Thread `me` issues the fills f with f % 2 == me; fill f uses accumulator
    // and B stage f % 4, so each thread owns two of them and commits them.
    if (leader && lane == 0) {
      const int me = warp == 1 ? 0 : 1;
      const uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
      // descriptors of the first A and B buffers; another buffer or K slice
      // adds its byte offset / 16 to the address field (shared addresses stay
      // below 2^18, so the field does not overflow)
      const uint64_t a_desc0 = sw128_desc(smem_u32(a_buf));
      const uint64_t b_desc0 = sw128_desc(smem_u32(b_buf));
      int a_cnt = 0, f_base = 0;
      bool ok = true;
      for (int kk = 0, item = pair_item(p, 0); ok && item >= 0; item = pair_item(p, ++kk)) {
        const PairItem it = decode_pair<PASS>(p, item, rank);
        if (it.n_ch == 0) continue;
        const int ab = a_cnt % kABufs;
        bool have_a = false;
        for (int c = (f_base + me) % 2 == 0 ? 0 : 1; ok && c < it.n_ch; c += 2) {
          const int f = f_base + c;
          const int g = f % kGroups;  // accumulator
          const int st = f % NS;      // B stage
          if (!pwait<1>(&full[st], (f / NS) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          if (!have_a) {
            if (!pwait<1>(&afull[ab], (a_cnt / kABufs) & 1, abort, p.status)) {
              ok = false;
              break;
            }
            have_a = true;
          }
          if (!pwait<1>(&accempty[g], ((f / kGroups) & 1) ^ 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const int kb = k / 4, kq = k % 4;
            mma_bf16_pair(tmem + g * BN,
                          a_desc0 + ((ab * ly.a_bytes + kb * BM * 128 + kq * 32) >> 4),
                          b_desc0 + ((st * ly.b_bytes + kb * BNH * 128 + kq * 32) >> 4), idesc,
                          k > 0 ? 1u : 0u);
          }
          // one commit per fill: the accumulator is written and, with it, B
          // stage g is free again in both CTAs
          mma_commit_pair_multicast(&accfull[g], kBoth);
          if (kStages != kGroups) mma_commit_pair_multicast(&empty[st], kBoth);
        }
        if (!ok) break;
        // the A buffer is free once both threads' MMAs of this item are done
        mma_commit_pair_multicast(&aempty[ab], kBoth);
        f_base += it.n_ch;
        ++a_cnt;
      }
      mma_commit_pair(done);
      drain_wait(done, 0, p.status);
    }
    __syncwarp();
  } else if (warp == kMergeWarp) {
    // ------------------------------------------------------------ merge
    const float c = p.scale_log2;
    int n_merge = 0;
    bool ok = true;
    for (int kk = 0, item = pair_item(p, 0); ok && item >= 0; item = pair_item(p, ++kk)) {
      const PairItem it = decode_pair<PASS>(p, item, rank);
      if (PASS == 2 && it.n_ch == 0) continue;
      if (it.tile < 0) continue;
      const int pb = n_merge & 1;
      if (!pwait_warp(&part_full[pb], (n_merge >> 1) & 1, abort, p.status)) {
        ok = false;
        break;
      }
      ++n_merge;
      float a[kGroups][4], b[kGroups][4];
#pragma unroll
      for (int g = 0; g < kGroups; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int lrow = lane + 32 * j;
          if (PASS == 1) {
            const float* h = part + ((pb * kGroups + g) * BM + lrow) * 2;
            a[g][j] = h[0];
            b[g][j] = h[1];
          } else {
            a[g][j] = part[(pb * kGroups + g) * BM + lrow];
            b[g][j] = 0.f;
          }
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(&part_empty[pb]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int lrow = lane + 32 * j;
        if (PASS == 1) {
          const int r = it.tile * BM + lrow;
          const int qpos = p.T - p.W + (r % p.W);
          const bool row_valid = (r < p.R) && (qpos >= it.pad) && (it.n_ch > 0);
          if (r < p.Rp) {
            float M = -INFINITY;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) M = fmaxf(M, a[g][j]);
            float S = 0.f;
            if (M != -INFINITY) {
#pragma unroll
              for (int g = 0; g < kGroups; ++g)
                S += (a[g][j] == -INFINITY) ? 0.f : b[g][j] * ex2((a[g][j] - M) * c);
            }
            const bool has = row_valid && S > 0.f;
            const size_t o = static_cast<size_t>(it.u) * p.Rp + r;
            p.negb[o] = has ? -(M * c + log2f(S)) : -INFINITY;
            p.pmax[o] = has ? 1.0f / S : 0.f;
          }
        } else {
          const int pos = it.tile * BM + lrow;
          if (pos >= it.pad && pos < p.T) {
            float s = 0.f;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) s += a[g][j];
            p.usage[static_cast<size_t>(it.u) * p.T + pos] = s;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp 2 + 4g + i: group g drains accumulator g (the item's fills f with
    // f % 4 == g), all 128 of its columns; lane quarter warp % 4.
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int lrow = quarter * 32 + lane;
    const uint32_t t_lane =
        tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(grp * BN);
    const float c = p.scale_log2;
    int f_base = 0;   // fills of the items before this one
    int n_merge = 0;  // items handed to the merge warp
    int rb_iter = 0;
    bool ok = true;
    auto release = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(accempty_l + 8u * grp);
    };
    for (int kk = 0, item = pair_item(p, 0); ok && item >= 0; item = pair_item(p, ++kk)) {
      const PairItem it = decode_pair<PASS>(p, item, rank);
      const int tile = it.tile;
      if (PASS == 1) {
        const int r = (tile >= 0 ? tile : 0) * BM + lrow;
        const int qpos = p.T - p.W + (r % p.W);
        const bool row_valid = tile >= 0 && (r < p.R) && (qpos >= it.pad) && (it.n_ch > 0);
        float mz = -INFINITY, sum = 0.f;
        // this group's chunks: ch with (f_base + ch) % 4 == grp
        for (int ch = (grp - f_base % kGroups + kGroups) % kGroups; ch < it.n_ch; ch += kGroups) {
          const int kf = (f_base + ch) / kGroups;  // fill count of this accumulator
          if (!pwait_warp(&accfull[grp], kf & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (tile < 0) {  // the MMA filled this CTA's half for the peer's tile only
            release();
            continue;
          }
          const int c0 = it.c_start + ch * BN;
          const int n_cols = pair_chunk_cols(it, ch);
          const int nb = n_cols / 32;
          const int lo = max(it.pad, c0), hi = min(qpos, c0 + n_cols - 1);
          const bool fast =
              __all_sync(0xffffffffu, row_valid && nb == 4 && lo <= c0 && hi >= c0 + BN - 1);
          uint32_t v[2][32];
          float bmx[2];
          __syncwarp();
          if (fast) {
            load2(t_lane, true, v, bmx);
            tmem_ld_wait();
            row_pair(v, bmx, c, mz, sum);
            __syncwarp();
            load2(t_lane + 64, true, v, bmx);
            tmem_ld_wait();
            release();
            row_pair(v, bmx, c, mz, sum);
          } else {
            for (int b = 0; b < nb; ++b) {
              __syncwarp();
              tmem_ld32(t_lane + 32 * b, v[0]);
              tmem_ld_wait();
              if (b == nb - 1) release();
              row_block<false>(v[0], -INFINITY, c0 + 32 * b, lo, hi, c, mz, sum);
            }
            if (nb == 0) release();
          }
        }
        f_base += it.n_ch;
        if (!ok) break;
        if (tile < 0) continue;
        const int pb = n_merge & 1;
        if (!pwait_warp(&part_empty[pb], ((n_merge >> 1) & 1) ^ 1, abort, p.status)) break;
        *reinterpret_cast<float2*>(part + ((pb * kGroups + grp) * BM + lrow) * 2) =
            make_float2(mz, sum);
        __syncwarp();
        if (lane == 0) mbar_arrive(&part_full[pb]);
        ++n_merge;
      } else {
        if (it.n_ch == 0) continue;
        const int rb = rb_iter & p.rb_shift;
        if (!pwait_warp(&rbfull[rb], (rb_iter >> p.rb_shift) & 1, abort, p.status)) break;
        ++rb_iter;
        const float* row_b = row_b_all + rb * rbf;
        const int pos = (tile >= 0 ? tile : 0) * BM + lrow;
        const bool pos_valid = tile >= 0 && (pos >= it.pad) && (pos < p.T);
        const bool fast = __all_sync(0xffffffffu, pos_valid && (pos <= p.T - p.W));
        const int jmin = pos - (p.T - p.W);
        float2 acc = make_float2(0.f, 0.f);
        for (int ch = (grp - f_base % kGroups + kGroups) % kGroups; ch < it.n_ch; ch += kGroups) {
          const int kf = (f_base + ch) / kGroups;
          if (!pwait_warp(&accfull[grp], kf & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (tile < 0) {
            release();
            continue;
          }
          const int n_cols = pair_chunk_cols(it, ch);
          const int nb = n_cols / 32;
          const int r0 = ch * BN;  // first query row of the fill's columns
          uint32_t v[2][32];
          float bmx[2];
          __syncwarp();
          if (nb == 4 && fast) {
            load2(t_lane, false, v, bmx);
            tmem_ld_wait();
            slot_pair(v, row_b + r0, c, acc);
            __syncwarp();
            load2(t_lane + 64, false, v, bmx);
            tmem_ld_wait();
            release();
            slot_pair(v, row_b + r0 + 64, c, acc);
          } else {
            for (int b = 0; b < nb; ++b) {
              __syncwarp();
              tmem_ld32(t_lane + 32 * b, v[0]);
              tmem_ld_wait();
              if (b == nb - 1) release();
              slot_block<false>(v[0], row_b + r0 + 32 * b, r0 + 32 * b, p.W, jmin, c, acc);
            }
            if (nb == 0) release();
          }
        }
        f_base += it.n_ch;
        __syncwarp();
        if (lane == 0) mbar_arrive(&rbempty[rb]);
        if (!ok) break;
        if (tile < 0) continue;
        const int pb = n_merge & 1;
        if (!pwait_warp(&part_empty[pb], ((n_merge >> 1) & 1) ^ 1, abort, p.status)) break;
        part[(pb * kGroups + grp) * BM + lrow] = acc.x + acc.y;
        __syncwarp();
        if (lane == 0) mbar_arrive(&part_full[pb]);
        ++n_merge;
      }
    }
  }

  // every thread of both CTAs: no CTA leaves while the other may still write
  // its shared memory, arrive on its barriers or read its tensor memory
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kAccCols);  // warp 1 of BOTH CTAs
#endif
}

int pair_smem_optin() {
  static int v = 0;
  if (!v) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      v = 227 * 1024;
  }
  return v;
}

}  // namespace

bool make_usage_map(CUtensorMap* m, const void* base, uint64_t rows, int d, int box_rows,
                    std::string* err);

template <int D>
cudaError_t launch_pair_d(const kvc_handle* h, const UsageArgs& a, int pass, cudaStream_t s,
                          std::string* err) {
  const Dims& dm = h->dims;
  const uint64_t q_rows = static_cast<uint64_t>(dm.U) * dm.R;
  const uint64_t k_rows = static_cast<uint64_t>(dm.U) * a.T;
  CUtensorMap map_a, map_b;
  if (!make_usage_map(&map_a, pass == 1 ? a.q : a.k, pass == 1 ? q_rows : k_rows, D, BM, err) ||
      !make_usage_map(&map_b, pass == 1 ? a.k : a.q, pass == 1 ? k_rows : q_rows, D, BNH, err))
    return cudaErrorInvalidValue;
  PairParams p;
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
  const int part = pair_part_bytes(pass);
  p.rb_shift = PairLayout(D, 2, 2 * rbf * 4, part).total <= pair_smem_optin() ? 1 : 0;
  p.n_stages = PairLayout(D, kStages, (rbf * 4) << p.rb_shift, part).total <= pair_smem_optin()
                   ? kStages
                   : 0;
  if (p.n_stages == 0) {
    if (err) *err = "paired attention kernel does not fit in shared memory";
    return cudaErrorInvalidValue;
  }
  const size_t smem = PairLayout(D, p.n_stages, (rbf * 4) << p.rb_shift, part).total;
  p.n_tiles = (pass == 1) ? (dm.R + BM - 1) / BM : (a.T + BM - 1) / BM;
  p.n_pairs = (p.n_tiles + 1) / 2;
  p.n_items = dm.U * p.n_pairs;
  auto kern = pass == 1 ? usage_pair_kernel<D, 1> : usage_pair_kernel<D, 2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // Persistent pairs, one per pair of SMs that can hold one at the same time:
  // a cluster must sit inside one GPC, so fewer than num_sms / 2 pairs may fit,
  // and a pair left for a second wave would double the time.
  int pairs_max = h->num_sms / 2;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2 * pairs_max);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = smem;
  int fit = 0;
  if (cudaOccupancyMaxActiveClusters(&fit, kern, &lc) == cudaSuccess && fit > 0) {
    if (fit < pairs_max) pairs_max = fit;
  } else {
    cudaGetLastError();
  }
  p.unit_major = dm.U >= 2 * pairs_max ? 1 : 0;
  const int clusters = p.n_items < pairs_max ? p.n_items : pairs_max;
  kern<<<2 * clusters, kThreads, smem, s>>>(map_a, map_b, p);
  return cudaGetLastError();
}

cudaError_t launch_attention_usage_pair(const kvc_handle* h, const UsageArgs& a, int pass,
                                        cudaStream_t s, std::string* err) {
  switch (h->dims.d) {
    case 64:
      return launch_pair_d<64>(h, a, pass, s, err);
    case 128:
      return launch_pair_d<128>(h, a, pass, s, err);
    default:
      if (err) *err = "head_dim must be 64 or 128";
      return cudaErrorInvalidValue;
  }
}

}  // namespace kvc
