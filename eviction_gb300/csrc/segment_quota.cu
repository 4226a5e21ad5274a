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
// Exactness: the fp32 mass becomes 40-bit fixed point (mu = trunc(m * 2^40),
// exact), prefix sums are uint64, the thresholds are
// tau_k = ceil(fl(fl(k*Delta) * S)) in IEEE double with round-to-nearest and no
// fused operations, the split/merge and quota rules are integer only.  The
// same definitions with the same tie rules give the same bits on any machine.
//   * empty raw segments are dropped; merge left to right until >= seg_min,
//     a short tail joins its predecessor; then split L > seg_max into
//     c = ceil(L/seg_max) parts, the first L mod c one longer;
//   * budget = min(T_keep, n); infeasible minimums go to the heaviest segments
//     (ties: lower index); round = half up; correction one unit at a time on the
//     exact remainder (short: largest remainder among q < L, ties lower index;
//     over: smallest remainder among q > q^min, ties higher index).
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 128;  // per-unit latency chains: more CTAs in flight beat wider ones
constexpr int kMaxK = 1024;  // thresholds: delta >= 1/1024
constexpr int kFastSegs = 256;  // segment count up to which the quota correction ranks directly

__device__ __forceinline__ uint64_t fixed_mass(float m) {
  // m * 2^40 is exact in fp32 (an exponent shift); truncation toward zero.
  const float scaled = m * 1099511627776.0f;
  return scaled > 0.f ? __float2ull_rz(scaled) : 0ull;
}

__device__ __forceinline__ uint64_t warp_incl_scan(uint64_t v) {
  const int lane = threadIdx.x % 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

struct SegParams {
  int T, B, H, S_max, S_cap;
  int budget, q_min, seg_min, seg_max;
  int seg_fixed, quota_by_len, global_topk;  // ablation switches (0 = the method)
  double delta;
  int K;  // number of thresholds
  const float* mass;
  const int32_t* pad;
  int32_t* seg_start;
  int32_t* seg_len;
  int32_t* quota;
  int32_t* n_seg;
};

// The correction steps of the quota rule, in bulk.  Each step gives (or takes)
// one unit to the segment with the best current remainder, and a segment's
// remainder moves by the mass total Mt per unit, so the steps taken are exactly
// the D best "bids" b_s(k) = rem_s -/+ k*Mt over k < cap_s, ordered by value and
// then by segment index.  A search for the D-th bid value followed by an ordered
// pass over the ties reproduces the sequential result.
//   short (negate = false): bids rem_s - k*Mt, cap_s = len_s - q_s; q_s += taken
//   over  (negate = true):  bids -rem_s - k*Mt, cap_s = q_s - floor_s; q_s -= taken
__device__ __forceinline__ int64_t bids_ge(int64_t b0, int64_t M, int64_t cap, int64_t v) {
  if (cap <= 0 || b0 < v) return 0;
  const int64_t k = (b0 - v) / M + 1;
  return k < cap ? k : cap;
}

__device__ void take_best_bids(const int64_t* rem, const int32_t* ref, int32_t* q, int ns,
                               int64_t M, int64_t D, bool negate, bool low_first, int lane,
                               int32_t* scratch) {
  auto b0_of = [&](int s) { return negate ? -rem[s] : rem[s]; };
  auto cap_of = [&](int s) -> int64_t {
    return negate ? static_cast<int64_t>(q[s]) - ref[s] : static_cast<int64_t>(ref[s]) - q[s];
  };
  // Fast exact path.  Round-half-up leaves every first bid of a segment with
  // spare capacity in (-M/2, M/2] (short) or [-M/2, M/2) (over), so bids of
  // round r (k = r) all lie below every bid of round r-1: the D best bids are
  // whole rounds (one unit to every segment with capacity left) plus the D'
  // best first bids of the next round, in (bid, index) order.  No division.
  bool in_range = ns <= kFastSegs;
  for (int s = lane; s < ns; s += 32) {
    if (cap_of(s) <= 0) continue;
    const int64_t twice = 2 * b0_of(s);
    in_range = in_range && (negate ? (twice >= -M && twice < M) : (twice > -M && twice <= M));
  }
  if (__all_sync(0xffffffffu, in_range)) {
    // complete rounds r: the largest r with sum_s min(cap_s, r) <= D
    auto given = [&](int64_t r) {
      int64_t g = 0;
      for (int s = lane; s < ns; s += 32) {
        const int64_t cap = cap_of(s);
        g += cap <= 0 ? 0 : (cap < r ? cap : r);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
      return g;
    };
    int64_t rmax = 0;
    for (int s = lane; s < ns; s += 32) {
      const int64_t cap = cap_of(s);
      rmax = cap > rmax ? cap : rmax;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const int64_t t = __shfl_xor_sync(0xffffffffu, rmax, o);
      rmax = t > rmax ? t : rmax;
    }
    int64_t r = 0, r_hi = rmax;  // given(0) = 0 <= D
    while (r < r_hi) {
      const int64_t mid = r + (r_hi - r + 1) / 2;
      if (given(mid) <= D) r = mid; else r_hi = mid - 1;
    }
    D -= given(r);
    // round r: the D best first bids among the segments with capacity > r
    for (int s = lane; s < ns; s += 32) {
      const int64_t cap = cap_of(s);
      int64_t t = cap < r ? cap : r;
      if (cap > r && D > 0) {
        const int64_t b0 = b0_of(s);
        int64_t rank = 0;
        for (int j = 0; j < ns; ++j) {
          if (j == s || cap_of(j) <= r) continue;
          const int64_t bj = b0_of(j);
          rank += (bj > b0 || (bj == b0 && (low_first ? j < s : j > s))) ? 1 : 0;
        }
        if (rank < D) t += 1;
      }
      scratch[s] = static_cast<int32_t>(t);
    }
    __syncwarp();
    for (int s = lane; s < ns; s += 32) q[s] = negate ? q[s] - scratch[s] : q[s] + scratch[s];
    __syncwarp();
    return;
  }
  // General path (bids outside that range cannot arise from the rounding rule;
  // kept so that the routine is exact for any input).
  // search range: every bid lies in [lo, hi]
  int64_t lo = INT64_MAX, hi = INT64_MIN;
  for (int s = lane; s < ns; s += 32) {
    const int64_t cap = cap_of(s);
    if (cap <= 0) continue;
    const int64_t b0 = b0_of(s);
    hi = b0 > hi ? b0 : hi;
    const int64_t last = b0 - (cap - 1) * M;
    lo = last < lo ? last : lo;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int64_t ol = __shfl_xor_sync(0xffffffffu, lo, o);
    const int64_t oh = __shfl_xor_sync(0xffffffffu, hi, o);
    lo = ol < lo ? ol : lo;
    hi = oh > hi ? oh : hi;
  }
  if (lo > hi) return;  // no bids (cannot happen for a consistent input)
  auto count_ge = [&](int64_t v) {
    int64_t c = 0;
    for (int s = lane; s < ns; s += 32) c += bids_ge(b0_of(s), M, cap_of(s), v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
  };
  // v* = largest v with count_ge(v) >= D
  if (count_ge(lo) < D) D = count_ge(lo);  // cannot happen: total bids >= D
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo + 1) / 2;
    if (count_ge(mid) >= D) lo = mid; else hi = mid - 1;
  }
  const int64_t vstar = lo;
  // bids strictly above v*, then the ties at v* in index order
  int64_t above = 0;
  for (int s = lane; s < ns; s += 32) above += bids_ge(b0_of(s), M, cap_of(s), vstar + 1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
  int64_t ties_left = D - above;
  const int n_chunks = (ns + 31) / 32;
  for (int cc = 0; cc < n_chunks; ++cc) {
    const int chunk = low_first ? cc : n_chunks - 1 - cc;
    const int s = chunk * 32 + lane;
    int64_t t = 0;
    bool tie = false;
    if (s < ns) {
      const int64_t b0 = b0_of(s), cap = cap_of(s);
      t = bids_ge(b0, M, cap, vstar + 1);
      tie = bids_ge(b0, M, cap, vstar) > t;
    }
    const uint32_t ball = __ballot_sync(0xffffffffu, tie);
    const uint32_t before = low_first ? (ball & ((1u << lane) - 1u))
                                      : (lane == 31 ? 0u : (ball & ~((2u << lane) - 1u)));
    if (tie && static_cast<int64_t>(__popc(before)) < ties_left) t += 1;
    ties_left -= __popc(ball);
    if (s < ns) q[s] = static_cast<int32_t>(negate ? q[s] - t : q[s] + t);
    __syncwarp();
  }
}

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
  uint64_t* s_mass = reinterpret_cast<uint64_t*>(sm);
  int64_t* s_rem = reinterpret_cast<int64_t*>(s_mass + p.S_cap);
  int32_t* s_start = reinterpret_cast<int32_t*>(s_rem + p.S_cap);
  int32_t* s_len = s_start + p.S_cap;
  int32_t* s_q = s_len + p.S_cap;
  int32_t* s_floor = s_q + p.S_cap;
  __shared__ int32_t s_b[kMaxK];
  __shared__ uint64_t s_tau[kMaxK];
  __shared__ uint64_t s_warp[NT / 32];
  __shared__ uint64_t s_total;
  __shared__ int s_nseg;

  const int u = blockIdx.x;
  const int T = p.T;
  const int b = (u / p.H) % p.B;
  const int pad = min(max(p.pad[b], 0), T);
  const int n = T - pad;
  const float* m = p.mass + static_cast<size_t>(u) * T + pad;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  int32_t* o_start = p.seg_start + static_cast<size_t>(u) * p.S_max;
  int32_t* o_len = p.seg_len + static_cast<size_t>(u) * p.S_max;
  int32_t* o_q = p.quota + static_cast<size_t>(u) * p.S_max;

  if (n <= 0) {
    for (int s = threadIdx.x; s < p.S_max; s += NT) {
      o_start[s] = 0;
      o_len[s] = 0;
      o_q[s] = 0;
    }
    if (threadIdx.x == 0) p.n_seg[u] = 0;
    return;
  }

  // ---- 1. prefix sums of the fixed-point mass over contiguous thread ranges
  const int per = (n + NT - 1) / NT;
  const int lo = min(n, threadIdx.x * per), hi = min(n, lo + per);
  uint64_t local = 0;
  for (int v = lo; v < hi; ++v) local += fixed_mass(m[v]);
  const uint64_t incl = warp_incl_scan(local);
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t run = 0;
    for (int w = 0; w < NT / 32; ++w) {
      const uint64_t t = s_warp[w];
      s_warp[w] = run;
      run += t;
    }
    s_total = run;
  }
  __syncthreads();
  const uint64_t before = s_warp[warp] + incl - local;  // prefix before `lo`
  const uint64_t S = s_total;

  // ---- 2. cut points: b_k = min{t in [1,n] : C(t) >= tau_k}; each threshold
  // is computed once (fp64 is slow on this part), then found by the thread
  // whose range holds it
  const double S_d = __ull2double_rn(S);
  for (int k = threadIdx.x; k < p.K; k += NT) {
    const double frac = __dmul_rn(static_cast<double>(k + 1), p.delta);
    s_tau[k] = static_cast<uint64_t>(ceil(__dmul_rn(frac, S_d)));
  }
  __syncthreads();
  for (int k = 0; k < p.K; ++k) {
    const uint64_t tau = s_tau[k];
    if (tau == 0) {
      if (threadIdx.x == 0) s_b[k] = 1;
    } else if (before < tau && tau <= before + local) {
      uint64_t c = before;
      for (int v = lo; v < hi; ++v) {
        c += fixed_mass(m[v]);
        if (c >= tau) {
          s_b[k] = v + 1;
          break;
        }
      }
    }
  }
  __syncthreads();

  // ---- 3. raw segments, merge, split (serial: at most K+1 raw segments)
  if (threadIdx.x == 0 && (p.global_topk || p.seg_fixed > 0)) {
    // ablations: one segment over everything, or fixed-length segments whose
    // shorter tail joins the segment before it
    int ns_ab = 1;
    if (p.global_topk) {
      s_start[0] = 0;
      s_len[0] = n;
    } else {
      ns_ab = max(1, n / p.seg_fixed);
      for (int s = 0; s < ns_ab; ++s) {
        s_start[s] = s * p.seg_fixed;
        s_len[s] = (s + 1 < ns_ab) ? p.seg_fixed : n - s * p.seg_fixed;
      }
    }
    s_nseg = ns_ab;
  } else if (threadIdx.x == 0) {
    // raw segments into s_start/s_len (drop empty)
    int n_raw = 0, prev = 0;
    for (int k = 0; k < p.K; ++k) {
      const int bk = s_b[k];
      if (bk > prev) {
        s_start[n_raw] = prev;
        s_len[n_raw] = bk - prev;
        ++n_raw;
        prev = bk;
      }
    }
    if (prev < n) {
      s_start[n_raw] = prev;
      s_len[n_raw] = n - prev;
      ++n_raw;
    }
    // merge in place
    int n_mer = 0;
    int cur_s = s_start[0], cur_l = s_len[0];
    for (int r = 1; r < n_raw; ++r) {
      if (cur_l < p.seg_min) {
        cur_l += s_len[r];
      } else {
        s_start[n_mer] = cur_s;
        s_len[n_mer] = cur_l;
        ++n_mer;
        cur_s = s_start[r];
        cur_l = s_len[r];
      }
    }
    if (cur_l < p.seg_min && n_mer > 0) {
      s_len[n_mer - 1] += cur_l;
    } else {
      s_start[n_mer] = cur_s;
      s_len[n_mer] = cur_l;
      ++n_mer;
    }
    // split, back to front so that the merged list is read before overwritten
    int n_out = 0;
    for (int r = 0; r < n_mer; ++r) {
      const int L = s_len[r];
      n_out += (L <= p.seg_max) ? 1 : (L + p.seg_max - 1) / p.seg_max;
    }
    int w = n_out;
    for (int r = n_mer - 1; r >= 0; --r) {
      const int L = s_len[r], st = s_start[r];
      if (L <= p.seg_max) {
        --w;
        s_start[w] = st;
        s_len[w] = L;
        continue;
      }
      const int c = (L + p.seg_max - 1) / p.seg_max;
      const int base = L / c, extra = L % c;
      // part j starts at st + j*base + min(j, extra)
      for (int j = c - 1; j >= 0; --j) {
        --w;
        s_start[w] = st + j * base + min(j, extra);
        s_len[w] = base + (j < extra ? 1 : 0);
      }
    }
    s_nseg = n_out;
  }
  __syncthreads();
  const int ns = s_nseg;

  // ---- 4. segment masses (one warp per segment)
  for (int s = warp; s < ns; s += NT / 32) {
    uint64_t acc = 0;
    for (int v = s_start[s] + lane; v < s_start[s] + s_len[s]; v += 32)
      acc += fixed_mass(m[v]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) s_mass[s] = acc;
  }
  __syncthreads();

  // ablation: quotas in proportion to segment length (lengths replace masses)
  if (p.quota_by_len)
    for (int s = threadIdx.x; s < ns; s += NT) s_mass[s] = static_cast<uint64_t>(s_len[s]);
  __syncthreads();

  // ---- 5. quotas (warp 0)
  if (warp == 0) {
    const int budget = min(p.budget, n);
    uint64_t Mt = 0;
    int64_t floor_tot = 0;
    for (int s = lane; s < ns; s += 32) {
      s_floor[s] = min(p.q_min, s_len[s]);
      Mt += s_mass[s];
      floor_tot += s_floor[s];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Mt += __shfl_xor_sync(0xffffffffu, Mt, o);
      floor_tot += __shfl_xor_sync(0xffffffffu, floor_tot, o);
    }
    __syncwarp();
    if (floor_tot > budget) {
      // heaviest segments first (ties: lower index) while budget remains
      for (int s = lane; s < ns; s += 32) {
        int64_t before_s = 0;
        for (int j = 0; j < ns; ++j) {
          const bool ahead = (s_mass[j] > s_mass[s]) || (s_mass[j] == s_mass[s] && j < s);
          if (ahead) before_s += s_floor[j];
        }
        const int64_t left = budget - before_s;
        s_q[s] = static_cast<int32_t>(left <= 0 ? 0 : (left < s_floor[s] ? left : s_floor[s]));
      }
      __syncwarp();
      for (int s = lane; s < ns; s += 32) s_floor[s] = s_q[s];
      __syncwarp();
      floor_tot = budget;
    }
    const int64_t t_rem = budget - floor_tot;
    int64_t qtot = 0;
    for (int s = lane; s < ns; s += 32) {
      int64_t share = 0;
      if (Mt > 0) {
        const uint64_t num = 2ull * static_cast<uint64_t>(t_rem) * s_mass[s] + Mt;
        share = static_cast<int64_t>(num / (2ull * Mt));
      }
      int64_t q = s_floor[s] + share;
      if (q > s_len[s]) q = s_len[s];
      s_q[s] = static_cast<int32_t>(q);
      s_rem[s] = (static_cast<int64_t>(s_floor[s]) * static_cast<int64_t>(Mt) +
                  t_rem * static_cast<int64_t>(s_mass[s])) -
                 q * static_cast<int64_t>(Mt);
      qtot += q;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qtot += __shfl_xor_sync(0xffffffffu, qtot, o);
    __syncwarp();
    // correction to the exact budget (bulk form of the one-unit-at-a-time rule)
    if (qtot < budget) {
      // segment s bids rem_s - k*Mt for k < L_s - q_s; take the D largest,
      // ties between segments -> lower index first.
      take_best_bids(s_rem, s_len, s_q, ns, static_cast<int64_t>(Mt),
                     budget - qtot, /*negate=*/false, /*low_first=*/true, lane,
                     reinterpret_cast<int32_t*>(s_mass));
    } else if (qtot > budget) {
      // segment s bids rem_s + k*Mt for k < q_s - floor_s; take the D smallest,
      // ties -> higher index first (the negated bids, largest first).
      take_best_bids(s_rem, s_floor, s_q, ns, static_cast<int64_t>(Mt),
                     qtot - budget, /*negate=*/true, /*low_first=*/false, lane,
                     reinterpret_cast<int32_t*>(s_mass));
    }
  }
  __syncthreads();

  // ---- 6. outputs (absolute starts), zero past n_seg
  for (int s = threadIdx.x; s < p.S_max; s += NT) {
    if (s < ns) {
      o_start[s] = pad + s_start[s];
      o_len[s] = s_len[s];
      o_q[s] = s_q[s];
    } else {
      o_start[s] = 0;
      o_len[s] = 0;
      o_q[s] = 0;
    }
  }
  if (threadIdx.x == 0) p.n_seg[u] = ns;
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
  p.delta = static_cast<double>(c.delta);
  p.K = segment_threshold_count(p.delta);
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
