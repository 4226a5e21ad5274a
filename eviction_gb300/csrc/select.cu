// select.cu -- segment-local top-k with must-keep and budget fix-up, one CTA per
// unit; emits the kept slots in ascending order.
//
// "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Method:
//  Key design 3: must-keep = 4 sinks and the recent suffix, inserted first; if
//                the budget left is negative the suffix is shortened, sinks
//                protected.  (The worked example counts the must-keep start and
//                end inside the first and last segments' quotas.)
//  Key design 4: top-q_i inside each segment on the base score, union with the
//                must-keep set, over budget -> drop low-score non-must-keep
//                picks; the kept indices are sorted.
// Rules (shared with any exact implementation of the same reading):
//   * B = min(T_keep, n); n_s = min(n_sink, B); n_r = min(n_recent, B - n_s);
//   * segment i picks max(0, q_i - |MK in i|) of its non-must-keep slots;
//   * order: score descending, ties -> lower slot; removal of the excess picks
//     in the exact reverse order (score ascending, ties -> higher slot).
// Scores are compared through an order-preserving 32-bit key.  Each warp takes
// whole segments: a bitwise search finds the want-th largest key among the
// segment's candidates, then one ordered ballot pass takes the ties at that key
// lowest slot first.  The global excess is removed the same way across the CTA
// (bitwise search for the excess-th smallest pick key, ties highest slot first).
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;  // units up to 4096 slots (see select_kernel)
constexpr int kRegPer = 8;  // slots per thread up to which the excess search keeps keys in registers
constexpr int kKeyPer = 16;  // longer units: gathered pick keys per thread held in registers

enum : uint8_t { kOut = 0, kMust = 1, kPick = 2 };

__device__ __forceinline__ uint32_t score_key(const float* sc, int v) {
  return float_order_key(__ldg(sc + v));
}

template <int NT>
__device__ __forceinline__ int block_count(int v, int* red) {
  constexpr int kWarps = NT / 32;
  v = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(v)));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += red[w];
  return t;
}

struct SelParams {
  int T, B, H, S_max, budget, n_sink, n_recent;
  const float* score;
  const int32_t* pad;
  const int32_t* seg_start;
  const int32_t* seg_len;
  const int32_t* quota;
  const int32_t* n_seg;
  int32_t* kept_idx;
  int32_t* n_kept;
};

// One warp: mark the `want` best candidates (flag == kOut) of [st, en).
__device__ __forceinline__ void pick_segment(const float* sc, uint8_t* flag, int st, int en,
                                             int want, int lane) {
  // largest x with #(candidates with key >= x) >= want: the want-th largest key
  uint32_t x = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t t = x | (1u << bit);
    unsigned cnt = 0;
    for (int v = st + lane; v < en; v += 32)
      cnt += (flag[v] == kOut && score_key(sc, v) >= t) ? 1u : 0u;
    if (static_cast<int>(__reduce_add_sync(0xffffffffu, cnt)) >= want) x = t;
  }
  unsigned gt = 0;
  for (int v = st + lane; v < en; v += 32)
    gt += (flag[v] == kOut && score_key(sc, v) > x) ? 1u : 0u;
  int ties_left = want - static_cast<int>(__reduce_add_sync(0xffffffffu, gt));
  const uint32_t below = (1u << lane) - 1u;
  for (int base = st; base < en; base += 32) {
    const int v = base + lane;
    const bool cand = v < en && flag[v] == kOut;
    const uint32_t k = cand ? score_key(sc, v) : 0u;
    const bool tie = cand && k == x;
    const uint32_t ball = __ballot_sync(0xffffffffu, tie);
    const bool take = (cand && k > x) ||
                      (tie && static_cast<int>(__popc(ball & below)) < ties_left);
    ties_left -= __popc(ball);
    __syncwarp();
    if (take) flag[v] = kPick;
  }
}

// As pick_segment for segments of at most 32*PER slots, with the candidates'
// keys held in registers across the search.
template <int PER>
__device__ __forceinline__ void pick_segment_reg(const float* sc, uint8_t* flag, int st, int en,
                                                 int want, int lane) {
  uint32_t key[PER];
  bool cand[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int v = st + lane + 32 * i;
    cand[i] = v < en && flag[v] == kOut;
    key[i] = cand[i] ? score_key(sc, v) : 0u;
  }
  uint32_t x = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t t = x | (1u << bit);
    unsigned cnt = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) cnt += (cand[i] && key[i] >= t) ? 1u : 0u;
    if (static_cast<int>(__reduce_add_sync(0xffffffffu, cnt)) >= want) x = t;
  }
  unsigned gt = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) gt += (cand[i] && key[i] > x) ? 1u : 0u;
  int ties_left = want - static_cast<int>(__reduce_add_sync(0xffffffffu, gt));
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < PER; ++i) {  // 32-slot groups in slot order
    const bool tie = cand[i] && key[i] == x;
    const uint32_t ball = __ballot_sync(0xffffffffu, tie);
    const bool take = (cand[i] && key[i] > x) ||
                      (tie && static_cast<int>(__popc(ball & below)) < ties_left);
    ties_left -= __popc(ball);
    if (take) flag[st + lane + 32 * i] = kPick;
  }
  __syncwarp();
}

// NT = 256 threads; units longer than 4096 slots (few, with many segments)
// take NT = 1024: four times the warps for the per-segment searches.  The
// selection compares keys only, so the result is the same for any NT.
template <int NT>
__global__ void __launch_bounds__(NT)
    select_kernel(SelParams p) {
  constexpr int kThreads = NT, kWarps = NT / 32;
  extern __shared__ uint8_t sm[];
  int32_t* s_start = reinterpret_cast<int32_t*>(sm);             // [S_max] valid offset
  int32_t* s_want = s_start + p.S_max;                            // [S_max]
  uint8_t* flag = reinterpret_cast<uint8_t*>(s_want + p.S_max);  // [T]
  // [budget] pick keys of the excess search of long units (T > kRegPer * kThreads)
  uint32_t* s_key = reinterpret_cast<uint32_t*>(flag + ((p.T + 15) & ~15));
  __shared__ int red[kWarps];
  __shared__ int red2[2 * kWarps];
  __shared__ int s_scan[kWarps];

  const int u = blockIdx.x;
  const int T = p.T;
  const int b = (u / p.H) % p.B;
  const int pad = min(max(p.pad[b], 0), T);
  const int n = T - pad;
  const float* sc = p.score + static_cast<size_t>(u) * T + pad;
  int32_t* out = p.kept_idx + static_cast<size_t>(u) * p.budget;
  const int ns = (n > 0) ? min(max(p.n_seg[u], 0), p.S_max) : 0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int Bk = min(p.budget, max(n, 0));
  const int n_s = min(p.n_sink, Bk);
  const int n_r = min(p.n_recent, Bk - n_s);

  // segment starts (valid offsets) and picks wanted per segment
  int want_sum = 0;
  for (int s = threadIdx.x; s < ns; s += kThreads) {
    const int st = min(max(p.seg_start[static_cast<size_t>(u) * p.S_max + s] - pad, 0), n);
    const int L = p.seg_len[static_cast<size_t>(u) * p.S_max + s];
    const int q = p.quota[static_cast<size_t>(u) * p.S_max + s];
    const int mk = max(0, min(st + L, n_s) - st) + max(0, st + L - max(st, n - n_r));
    const int want = max(0, min(q - mk, L - mk));
    s_start[s] = st;
    s_want[s] = want;
    want_sum += want;
  }
  for (int v = threadIdx.x; v < n; v += kThreads)
    flag[v] = (v < n_s || v >= n - n_r) ? kMust : kOut;
  const int total_picks = block_count<NT>(want_sum, red);  // (also orders the writes above)

  // segment-local picks, one warp per segment
  for (int s = warp; s < ns; s += kWarps) {
    const int st = s_start[s];
    const int en = (s + 1 < ns) ? max(st, s_start[s + 1]) : n;
    const int want = s_want[s];
    if (want <= 0) continue;
    if (en - st <= 32 * 8)
      pick_segment_reg<8>(sc, flag, st, en, want, lane);
    else
      pick_segment(sc, flag, st, en, want, lane);
  }
  __syncthreads();

  // over budget: drop the `excess` worst picks (score ascending, ties: higher slot)
  const int excess = n_s + n_r + total_picks - Bk;
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(n, static_cast<int>(threadIdx.x) * per);
  const int hi = min(n, lo + per);
  if (excess > 0) {
    // x = the excess-th smallest pick key: largest x with #(pick key < x) < excess
    uint32_t x = 0;
    if (per <= kRegPer) {  // CTA-uniform: every thread takes the same branch (barriers inside)
      uint32_t key[kRegPer];
      bool pk[kRegPer];
#pragma unroll
      for (int i = 0; i < kRegPer; ++i) {
        const int v = lo + i;
        pk[i] = v < hi && flag[v] == kPick;
        key[i] = pk[i] ? score_key(sc, v) : 0u;
      }
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t t = x | (1u << bit);
        unsigned cnt = 0;
#pragma unroll
        for (int i = 0; i < kRegPer; ++i) cnt += (pk[i] && key[i] < t) ? 1u : 0u;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        // alternate buffers: one barrier per step
        int* rb = red2 + (bit & 1) * kWarps;
        if (lane == 0) rb[warp] = static_cast<int>(cnt);
        __syncthreads();
        int total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) total += rb[w];
        if (total < excess) x = t;
      }
    } else {
      // long units: the picks' keys (at most the budget) gathered once into
      // shared memory in slot order, then searched there -- in registers when
      // there are at most kKeyPer per thread -- instead of every step
      // re-reading all of this thread's slots from global memory
      int cnt = 0;
      for (int v = lo; v < hi; ++v) cnt += flag[v] == kPick ? 1 : 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) s_scan[warp] = incl;
      __syncthreads();
      int pos = incl - cnt;
      for (int w = 0; w < warp; ++w) pos += s_scan[w];
      int n_pick = 0;
      for (int w = 0; w < kWarps; ++w) n_pick += s_scan[w];
      for (int v = lo; v < hi; ++v)
        if (flag[v] == kPick) s_key[pos++] = score_key(sc, v);
      __syncthreads();
      if (n_pick <= kKeyPer * kThreads) {  // CTA-uniform
        uint32_t key[kKeyPer];
#pragma unroll
        for (int i = 0; i < kKeyPer; ++i) {
          const int j = threadIdx.x + i * kThreads;
          key[i] = j < n_pick ? s_key[j] : 0xffffffffu;  // never below a threshold
        }
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t t = x | (1u << bit);
          unsigned c2 = 0;
#pragma unroll
          for (int i = 0; i < kKeyPer; ++i) c2 += key[i] < t ? 1u : 0u;
          c2 = __reduce_add_sync(0xffffffffu, c2);
          int* rb = red2 + (bit & 1) * kWarps;
          if (lane == 0) rb[warp] = static_cast<int>(c2);
          __syncthreads();
          int total = 0;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) total += rb[w];
          if (total < excess) x = t;
        }
      } else {
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t t = x | (1u << bit);
          int c2 = 0;
          for (int j = threadIdx.x; j < n_pick; j += kThreads) c2 += s_key[j] < t ? 1 : 0;
          if (block_count<NT>(c2, red) < excess) x = t;
        }
      }
      __syncthreads();  // s_scan is reused below
    }
    int lt = 0, ties = 0;
    for (int v = lo; v < hi; ++v) {
      if (flag[v] != kPick) continue;
      const uint32_t k = score_key(sc, v);
      lt += (k < x) ? 1 : 0;
      ties += (k == x) ? 1 : 0;
    }
    const int drop_ties = excess - block_count<NT>(lt, red);
    // ties above this thread's range (higher slots are dropped first)
    int incl = ties;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += t;
    }
    if (lane == 0) s_scan[warp] = incl;
    __syncthreads();
    int after = incl - ties;  // ties in higher lanes of this warp
    for (int w = warp + 1; w < kWarps; ++w) after += s_scan[w];
    for (int v = hi - 1; v >= lo; --v) {
      if (flag[v] != kPick) continue;
      const uint32_t k = score_key(sc, v);
      if (k < x) {
        flag[v] = kOut;
      } else if (k == x) {
        if (after < drop_ties) flag[v] = kOut;
        ++after;
      }
    }
    __syncthreads();
  }

  // ordered write-out: contiguous ranges per thread + block exclusive scan
  int cnt = 0;
  for (int v = lo; v < hi; ++v) cnt += flag[v] != kOut ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();  // s_scan may still be read by the excess pass
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_scan[w];
  int pos = wbase + incl - cnt;
  for (int v = lo; v < hi; ++v)
    if (flag[v] != kOut && pos < p.budget) out[pos++] = pad + v;
  int total = 0;
  for (int w = 0; w < kWarps; ++w) total += s_scan[w];
  for (int r = total + threadIdx.x; r < p.budget; r += kThreads) out[r] = -1;
  if (threadIdx.x == 0) p.n_kept[u] = min(total, p.budget);
}

}  // namespace

size_t select_smem_bytes(const kvc_config& c, int T) {
  const size_t base = static_cast<size_t>(s_max_of(c, T)) * 8 + ((static_cast<size_t>(T) + 15) & ~size_t(15));
  return base + (T > kRegPer * kThreads ? static_cast<size_t>(c.budget) * 4 : 0) + 16;
}

cudaError_t launch_select(const kvc_handle* h, const float* score, int T,
                          const int32_t* pad, const int32_t* seg_start,
                          const int32_t* seg_len, const int32_t* quota,
                          const int32_t* n_seg, int32_t* kept_idx,
                          int32_t* n_kept, cudaStream_t s) {
  const kvc_config& c = h->cfg;
  SelParams p;
  p.T = T;
  p.B = h->dims.B;
  p.H = h->dims.H;
  p.S_max = s_max_of(c, T);
  p.budget = c.budget;
  p.n_sink = c.n_sink;
  p.n_recent = c.n_recent;
  p.score = score;
  p.pad = pad;
  p.seg_start = seg_start;
  p.seg_len = seg_len;
  p.quota = quota;
  p.n_seg = n_seg;
  p.kept_idx = kept_idx;
  p.n_kept = n_kept;
  const size_t smem = select_smem_bytes(c, T);
  const bool wide = T > 4096;
  auto kern = wide ? select_kernel<1024> : select_kernel<kThreads>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<h->dims.U, wide ? 1024 : kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvc
