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
// The step is unit::select_phase (unit_phases.cuh, with its rules and search),
// which the fused per-unit kernel also runs; this file holds the stand-alone
// kernel of the kvc_select entry point and of units past 4096 slots.
#include "unit_phases.cuh"

namespace kvc {
namespace {

using unit::SelParams;
using unit::kRegPer;

constexpr int kThreads = 256;  // units up to 4096 slots (see select_kernel)

// Dynamic shared memory: start, want [S_max] | flags [T] | the radix
// histograms [warps][256] of the picks, reused by the pick keys [budget] of the
// excess search (units past kRegPer * kThreads slots; a barrier separates the
// two uses) | with 32 warps, the CTA-wide histogram [256 + 4] of that search.
struct SelLayout {
  int off_flag, off_key, off_hist, off_xhist, total;
};
__host__ __device__ inline SelLayout sel_layout(int S_max, int T, int budget, int warps) {
  SelLayout l;
  l.off_flag = 8 * S_max;
  l.off_key = (l.off_flag + ((T + 15) & ~15) + 15) & ~15;
  l.off_hist = l.off_key;
  const int keys = T > kRegPer * kThreads ? 4 * budget : 0;
  const int hist = 1024 * warps;
  l.total = l.off_key + (keys > hist ? keys : hist);
  l.off_xhist = (l.total + 15) & ~15;
  if (warps >= 32) l.total = l.off_xhist + 4 * (256 + 4);
  return l;
}

// NT = 256 threads, held to 40 registers so that six CTAs share an SM (the
// kernel is latency-bound per unit); units longer than 4096 slots (few, with
// many segments) take NT = 1024: four times the warps for the per-segment
// searches.  The selection compares keys only, so the result is the same for
// any NT.
template <int NT>
__global__ void __launch_bounds__(NT, NT == kThreads ? 6 : 1)
    select_kernel(SelParams p) {
  constexpr int kWarps = NT / 32;
  extern __shared__ uint8_t sm[];
  __shared__ int red[kWarps];
  __shared__ int red2[2 * kWarps];
  __shared__ int s_scan[kWarps];
  unit::SelSmem ss;
  const SelLayout ly = sel_layout(p.S_max, p.T, p.budget, kWarps);
  ss.start = reinterpret_cast<int32_t*>(sm);                  // [S_max] valid offset
  ss.want = ss.start + p.S_max;                               // [S_max]
  ss.flag = sm + ly.off_flag;                                 // [T]
  // [budget] pick keys of the excess search of long units (T > kRegPer * 256)
  ss.key = reinterpret_cast<uint32_t*>(sm + ly.off_key);
  ss.hist = reinterpret_cast<int*>(sm + ly.off_hist);         // [NT/32][256]
  ss.xhist = NT >= 1024 ? reinterpret_cast<int*>(sm + ly.off_xhist) : nullptr;  // [256 + 4]
  ss.red = red;
  ss.red2 = red2;
  ss.scan = s_scan;
  const int u = blockIdx.x;
  const int T = p.T;
  const int b = (u / p.H) % p.B;
  const int pad = min(max(p.pad[b], 0), T);
  const int n = T - pad;
  const int ns = (n > 0) ? min(max(p.n_seg[u], 0), p.S_max) : 0;
  const size_t so = static_cast<size_t>(u) * p.S_max;
  const unit::SegsGlobal segs{p.seg_start + so, p.seg_len + so, p.quota + so, pad};
  unit::select_phase<NT, true>(p, u, p.score + static_cast<size_t>(u) * T + pad, pad, n, ns,
                               segs, ss);
}

}  // namespace

size_t select_smem_bytes(const kvc_config& c, int T) {
  const int warps = (T > 4096 ? 1024 : kThreads) / 32;
  return static_cast<size_t>(sel_layout(s_max_of(c, T), T, c.budget, warps).total) + 16;
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
