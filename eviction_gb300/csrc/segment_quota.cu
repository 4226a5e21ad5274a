// segment_quota.cu -- cumulative-mass segmentation and segment quotas, one CTA
// per unit, in exact integer arithmetic.
//
// "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Method:
//  Key design 2:  C(t) = sum_{u<=t} m_u,  b_k = min{t | C(t) >= k*Delta};
//                 segments longer than the maximum are split into near-equal
//                 parts, short adjacent ones merged (16..256), masses recounted.
//  Key design 3:  q_i^min = min(q_min, L_i), T_rem = T_keep - sum q_i^min,
//                 q_i = q_i^min + round(T_rem M_i / sum M), clipped to L_i and
//                 corrected to the exact budget.
//
// The step is unit::segment_phase (unit_phases.cuh, with its exactness rules),
// which the fused per-unit kernel also runs; this file holds the stand-alone
// kernel of the kvc_segment_quota entry point and of units past 4096 slots.
#include <cmath>

#include "unit_phases.cuh"

namespace kvc {
namespace {

using unit::SegParams;
using unit::kMaxK;

constexpr int kThreads = 128;  // per-unit latency chains: more CTAs in flight beat wider ones
// Units longer than 4096 slots: 8 sub-range prefixes per thread range (64 slots
// of a 32768-slot unit each), so warp 0's scans of the mass in global memory
// (cut points, segment masses) cover 8 slots instead of 64.
constexpr int kLongSub = 8;

// NT = 128: 12 CTAs per SM (40 registers) rather than 10 at the natural 48:
// the kernel is latency-bound per unit, and more units in flight shorten the
// launch.  Units longer than 4096 slots are few, and each takes NT = 512
// threads: a quarter of the slots per thread in the scan and the searches.
// Every result is exact integer arithmetic, the same for any NT.
template <int NT>
__global__ void __launch_bounds__(NT, NT == 128 ? 12 : 3)
    segment_quota_kernel(SegParams p) {
  extern __shared__ uint8_t sm[];
  // dynamic shared layout: seg mass (u64) | rem (i64) | start | len | quota |
  // q_floor (i32) x S_cap
  __shared__ int32_t s_b[kMaxK];
  __shared__ uint64_t s_warp[NT / 32];
  __shared__ uint64_t s_pre[NT];
  __shared__ uint64_t s_sub[NT == 512 ? NT * kLongSub : 1];
  __shared__ uint64_t s_total;
  __shared__ int s_nseg;
  unit::SegSmem ss;
  ss.mass = reinterpret_cast<uint64_t*>(sm);
  ss.rem = reinterpret_cast<int64_t*>(ss.mass + p.S_cap);
  ss.start = reinterpret_cast<int32_t*>(ss.rem + p.S_cap);
  ss.len = ss.start + p.S_cap;
  ss.q = ss.len + p.S_cap;
  ss.floor = ss.q + p.S_cap;
  ss.b = s_b;
  ss.part = s_warp;
  ss.pre = s_pre;
  ss.sub = s_sub;
  ss.total = &s_total;
  ss.nseg = &s_nseg;
  const int u = blockIdx.x;
  const int T = p.T;
  const int b = (u / p.H) % p.B;
  const int pad = min(max(p.pad[b], 0), T);
  unit::segment_phase<NT, NT == 512 ? kLongSub : 1>(p, u, p.mass + static_cast<size_t>(u) * T + pad,
                                                    pad, T - pad, ss, true);
}

}  // namespace

int segment_threshold_count(double delta) {
  int K = 0;
  for (int k = 1; k <= kMaxK + 1; ++k) {
    if (!(static_cast<double>(k) * delta < 1.0)) break;
    ++K;
  }
  return K;
}

// Delta (a positive finite fp32) as m * 2^e with m odd: fl(k * Delta) in the
// thresholds is then (k * m) * 2^e exactly (k * m < 2^35).
void segment_delta_parts(float delta, uint64_t* m, int* e) {
  int ex = 0;
  const double f = std::frexp(static_cast<double>(delta), &ex);  // delta = f * 2^ex
  uint64_t mm = static_cast<uint64_t>(std::ldexp(f, 24));  // f has 24 significant bits
  int ee = ex - 24;
  while (mm != 0 && (mm & 1ull) == 0) {
    mm >>= 1;
    ++ee;
  }
  *m = mm;
  *e = ee;
}

int segment_capacity(const kvc_config& c, int T) {
  const int K = segment_threshold_count(static_cast<double>(c.delta));
  // raw segments (before merging) number at most K+1; after split/merge at
  // most min(S_max, K + 1 + ceil(T/seg_max)).
  const int bound = K + 1 + (T + c.seg_max - 1) / c.seg_max;
  const int smax = s_max_of(c, T);
  int cap = bound < smax ? bound : smax;
  if (cap < K + 1) cap = K + 1;
  // fixed-length ablation: at most T / seg_fixed (<= T / seg_min) segments
  if (c.seg_fixed > 0 && T / c.seg_fixed > cap) cap = T / c.seg_fixed;
  return cap;
}

size_t segment_smem_bytes(const kvc_config& c, int T) {
  return static_cast<size_t>(segment_capacity(c, T)) * (8 + 8 + 4 * 4);
}

cudaError_t launch_segment_quota(const kvc_handle* h, const float* mass, int T,
                                 const int32_t* pad, int32_t* seg_start,
                                 int32_t* seg_len, int32_t* quota,
                                 int32_t* n_seg, cudaStream_t s) {
  const kvc_config& c = h->cfg;
  SegParams p;
  p.T = T;
  p.B = h->dims.B;
  p.H = h->dims.H;
  p.S_max = s_max_of(c, T);
  p.S_cap = segment_capacity(c, T);
  p.budget = c.budget;
  p.q_min = c.q_min;
  p.seg_min = c.seg_min;
  p.seg_max = c.seg_max;
  p.seg_fixed = c.seg_fixed;
  p.quota_by_len = c.quota_by_len;
  p.global_topk = c.global_topk;
  segment_delta_parts(c.delta, &p.delta_m, &p.delta_e);
  p.K = segment_threshold_count(static_cast<double>(c.delta));
  p.mass = mass;
  p.pad = pad;
  p.seg_start = seg_start;
  p.seg_len = seg_len;
  p.quota = quota;
  p.n_seg = n_seg;
  const size_t smem = segment_smem_bytes(c, T);
  const bool wide = T > 4096;
  auto kern = wide ? segment_quota_kernel<512> : segment_quota_kernel<kThreads>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<h->dims.U, wide ? 512 : kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvc
