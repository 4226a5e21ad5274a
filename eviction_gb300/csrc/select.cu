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
//     in the exact reverse order.
// Keys are 64-bit: (order-preserving score bits << 32) | ~slot, so "best
// first" is descending key and every key is unique.  In-segment ranks are
// counted directly (segments are at most seg_max long); the global excess is
// removed with a bitwise search for the excess-th smallest pick key.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint64_t sel_key(float score, int v) {
  return (static_cast<uint64_t>(float_order_key(score)) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(v));
}

__device__ __forceinline__ int block_count(int v, int* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) t += red[w];
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

// flags: 0 = out, 1 = must-keep, 2 = pick
__global__ void __launch_bounds__(kThreads)
    select_kernel(SelParams p) {
  extern __shared__ uint8_t sm[];
  int32_t* s_start = reinterpret_cast<int32_t*>(sm);        // [S_max] valid offset
  int32_t* s_want = s_start + p.S_max;                       // [S_max]
  uint8_t* flag = reinterpret_cast<uint8_t*>(s_want + p.S_max);  // [T]
  __shared__ int red[kThreads / 32];
  __shared__ int s_scan[kThreads / 32];

  const int u = blockIdx.x;
  const int T = p.T;
  const int b = (u / p.H) % p.B;
  const int pad = min(max(p.pad[b], 0), T);
  const int n = T - pad;
  const float* sc = p.score + static_cast<size_t>(u) * T + pad;
  int32_t* out = p.kept_idx + static_cast<size_t>(u) * p.budget;
  const int ns = (n > 0) ? min(max(p.n_seg[u], 0), p.S_max) : 0;

  const int Bk = min(p.budget, max(n, 0));
  const int n_s = min(p.n_sink, Bk);
  const int n_r = min(p.n_recent, Bk - n_s);

  // segment starts (valid offsets) and picks wanted per segment
  for (int s = threadIdx.x; s < ns; s += kThreads) {
    const int st = min(max(p.seg_start[static_cast<size_t>(u) * p.S_max + s] - pad, 0), n);
    const int L = p.seg_len[static_cast<size_t>(u) * p.S_max + s];
    const int q = p.quota[static_cast<size_t>(u) * p.S_max + s];
    const int mk = max(0, min(st + L, n_s) - st) +
                   max(0, st + L - max(st, n - n_r));
    s_start[s] = st;
    s_want[s] = min(max(0, q - mk), L - mk);
  }
  __syncthreads();

  // ranks inside segments
  int picks = 0;
  for (int v = threadIdx.x; v < n; v += kThreads) {
    const bool must = (v < n_s) || (v >= n - n_r);
    uint8_t f = must ? 1 : 0;
    if (!must && ns > 0) {
      int lo = 0, hi = ns - 1;  // last segment with start <= v
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (s_start[mid] <= v) lo = mid; else hi = mid - 1;
      }
      const int st = s_start[lo];
      const int en = (lo + 1 < ns) ? max(st, s_start[lo + 1]) : n;
      const int want = s_want[lo];
      if (want > 0) {
        const uint64_t key = sel_key(sc[v], v);
        int rank = 0;
        for (int w = st; w < en && rank < want; ++w) {
          if (w < n_s || w >= n - n_r) continue;
          rank += (sel_key(sc[w], w) > key) ? 1 : 0;
        }
        if (rank < want) {
          f = 2;
          ++picks;
        }
      }
    }
    flag[v] = f;
  }
  const int total_picks = block_count(picks, red);
  const int excess = n_s + n_r + total_picks - Bk;

  if (excess > 0) {
    // the excess-th smallest pick key: largest x with #{picks with key < x} < excess
    uint64_t x = 0;
    for (int bit = 63; bit >= 0; --bit) {
      const uint64_t trial = x | (1ull << bit);
      int cnt = 0;
      for (int v = threadIdx.x; v < n; v += kThreads)
        if (flag[v] == 2 && sel_key(sc[v], v) < trial) ++cnt;
      if (block_count(cnt, red) < excess) x = trial;
    }
    for (int v = threadIdx.x; v < n; v += kThreads)
      if (flag[v] == 2 && sel_key(sc[v], v) <= x) flag[v] = 0;
    __syncthreads();
  }

  // ordered write-out: contiguous ranges per thread + block exclusive scan
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(n, static_cast<int>(threadIdx.x) * per);
  const int hi = min(n, lo + per);
  int cnt = 0;
  for (int v = lo; v < hi; ++v) cnt += flag[v] ? 1 : 0;
  int incl = cnt;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_scan[w];
  int pos = wbase + incl - cnt;
  for (int v = lo; v < hi; ++v)
    if (flag[v] && pos < p.budget) out[pos++] = pad + v;
  int total = 0;
  for (int w = 0; w < kThreads / 32; ++w) total += s_scan[w];
  for (int r = total + threadIdx.x; r < p.budget; r += kThreads) out[r] = -1;
  if (threadIdx.x == 0) p.n_kept[u] = min(total, p.budget);
}

}  // namespace

size_t select_smem_bytes(const kvc_config& c, int T) {
  return static_cast<size_t>(s_max_of(c, T)) * 8 + static_cast<size_t>(T) + 16;
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
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  select_kernel<<<h->dims.U, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvc
