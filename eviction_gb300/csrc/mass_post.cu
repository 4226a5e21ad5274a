// mass_post.cu -- from raw usage to score, mass and credit, one CTA per unit.
//
// "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Method,
// Key design 1:
//   * entries a window query cannot see (causal suffix) are filled with the
//     window's maximum score: the largest softmax probability of the unit,
//     max_r 1/Z'_r, taken from pass 1 of the attention kernel;
//   * u = average pool (kernel avg_pool, zero outside the valid slots, divided
//     by the kernel size);  m_i = (max(u_i,0)+eps) / sum_v (max(u_v,0)+eps);
//   * c = lambda*c_in + (1-lambda)*m with c_in := m on slots that are new since
//     the last event;  m_used = normalize(beta*m + (1-beta)*normalize(c)).
// The base score ("RefreshKV: ...", A2: max pooling of neighbouring attention
// scores; A6: kernel 7) is the filled usage max-pooled over valid neighbours.
//
// Reading of the normalisations: m sums to one, so the credit total is
// 1 + lambda * (sum over carried slots of (c_in - m)), and the mix
// beta*m + (1-beta)*c/sum(c) already sums to one; one block reduction of three
// totals (all of m, the carried slots' c_in and m) gives every value, and the
// last normalize() is a division by one, left out.
//
// Units up to 4096 slots take one pass with the filled usage in shared memory
// and per-slot values in registers; longer ones sweep global memory (the
// unit's data stays in L1/L2 between sweeps).  Every sum is a strided
// per-thread pass plus one fixed-order block reduction, so repeated runs give
// identical bits.
#include <cmath>

#include "unit_phases.cuh"

namespace kvc {
int attention_row_stride(int R);
namespace {

using unit::PostParams;
using unit::block_max;

// Units longer than kSmemT slots sweep global memory.  They are few (a long
// cache holds few sequences), so each takes a CTA of NT = 1024 threads: four
// times the loads in flight per unit of a 256-thread CTA.
template <int NT>
__global__ void __launch_bounds__(NT)
    mass_post_kernel(PostParams p) {
  __shared__ float red[3 * (NT / 32 + 1)];
  const int u = blockIdx.x;
  const int b = (u / p.H) % p.B;
  const int T = p.T;
  const int pad = min(max(p.pad[b], 0), T);
  const size_t base = static_cast<size_t>(u) * T;
  float* a = p.usage + base;
  float* mass = p.mass + base;
  float* score = p.score + base;
  float* cpost = p.credit_post + base;
  const float* cin = p.credit_in + base;

  if (pad >= T) {
    for (int i = threadIdx.x; i < T; i += NT) {
      mass[i] = 0.f;
      score[i] = -INFINITY;
      cpost[i] = 0.f;
    }
    return;
  }

  // fill value = largest probability of any present row (absent rows hold 0)
  float pm = 0.f;
  for (int r = threadIdx.x; r < p.R; r += NT)
    pm = fmaxf(pm, p.pmax[static_cast<size_t>(u) * p.Rp + r]);
  const float fill = block_max<NT>(pm, red);

  // a'(i) = a(i) + fill * (#present (head, query) pairs that cannot see i)
  const int j_lo = max(0, pad - (T - p.W));  // first present window query
  for (int i = pad + threadIdx.x; i < T; i += NT) {
    const int unseen = max(0, min(p.W, i - T + p.W) - j_lo) * p.G;
    a[i] += fill * static_cast<float>(unseen);
  }
  __syncthreads();

  // score = max-pooled usage; the mass totals (as in unit::mass_phase: one
  // reduction of the up total and the carried slots' credit-in and up)
  const int n_carry = min(max(p.n_carry[b], 0), T - pad);
  const int ra = p.avg_pool / 2, rm = p.max_pool / 2;
  const float inv_k = 1.0f / static_cast<float>(p.avg_pool);
  const bool pools75 = ra == 2 && rm == 3;
  float tot = 0.f, cin_c = 0.f, up_c = 0.f;
  for (int i = threadIdx.x; i < T; i += NT) {
    if (i < pad) {
      score[i] = -INFINITY;
      continue;
    }
    float mx, s;
    if (pools75 && i - 3 >= pad && i + 3 < T) {  // interior slot, default pools: unrolled
      const float w0 = a[i - 3], w1 = a[i - 2], w2 = a[i - 1], w3 = a[i], w4 = a[i + 1],
                  w5 = a[i + 2], w6 = a[i + 3];
      mx = fmaxf(fmaxf(fmaxf(w0, w1), fmaxf(w2, w3)), fmaxf(fmaxf(w4, w5), w6));
      s = (((w1 + w2) + w3) + w4) + w5;  // the loop's order
    } else {
      mx = -INFINITY;
      for (int t = max(pad, i - rm); t <= min(T - 1, i + rm); ++t) mx = fmaxf(mx, a[t]);
      s = 0.f;
      for (int t = max(pad, i - ra); t <= min(T - 1, i + ra); ++t) s += a[t];
    }
    score[i] = mx;
    const float up = fmaxf(s * inv_k, 0.f) + p.eps;
    mass[i] = up;  // kept for the second sweep, which overwrites it
    tot += up;
    if (i < pad + n_carry) {
      cin_c += cin[i];
      up_c += up;
    }
  }
  const float3 tt = unit::block_sum3<NT>(make_float3(tot, cin_c, up_c), red);
  const float total1 = tt.x;
  const float lam = p.lambda, beta = p.beta;
  const float c_total = 1.0f + lam * (tt.y - tt.z / total1);
  // the two normalisations as products with reciprocals taken once per unit
  const float inv_total = 1.0f / total1;
  const float inv_ct = c_total > 0.f ? 1.0f / c_total : 0.f;

  // mass (m_used) and credit
  for (int i = threadIdx.x; i < T; i += NT) {
    float mu = 0.f, c = 0.f;
    if (i >= pad) {
      const float m = mass[i] * inv_total;  // the first sweep's up
      c = (i < pad + n_carry) ? lam * cin[i] + (1.0f - lam) * m : m;
      const float cn = (c_total > 0.f) ? c * inv_ct : m;
      mu = beta * m + (1.0f - beta) * cn;
    }
    mass[i] = mu;
    cpost[i] = c;
  }
}

// Units of up to kSmemT slots: one pass (unit::mass_phase; the fused per-unit
// kernel runs the same function with the same CTA shape, unit::mass_shape).
// The filled usage of the unit sits in shared memory (the pooling windows read
// it there), each thread keeps its slots' values in registers across the
// three totals, and score, mass and credit are written once.
// Latency-bound: one CTA per unit, so the more CTAs an SM holds the better.
// 32 registers: 16 CTAs of 128 threads per SM, or up to 6 slots per thread 8
// CTAs of 256 (units past 2048 slots).
template <int NT, int kEpt>  // T <= kEpt * NT
__global__ void __launch_bounds__(NT, NT == 128 ? 16 : (kEpt <= 6 ? 8 : (kEpt <= 8 ? 6 : 4)))
    mass_post_smem_kernel(PostParams p) {
  __shared__ float red[3 * (NT / 32 + 1)];
  __shared__ float a[kEpt * NT];
  unit::mass_phase<kEpt, NT>(p, blockIdx.x, a, red, nullptr, nullptr);
}

}  // namespace

cudaError_t launch_mass_post(const kvc_handle* h, int T, const int32_t* pad,
                             const int32_t* n_carry, const float* credit_in,
                             float* credit_post, float* mass, float* score,
                             cudaStream_t s) {
  const Dims& dm = h->dims;
  PostParams p;
  p.T = T;
  p.R = dm.R;
  p.W = dm.W;
  p.G = dm.G;
  p.B = dm.B;
  p.H = dm.H;
  p.avg_pool = h->cfg.avg_pool;
  p.max_pool = h->cfg.max_pool;
  p.eps = h->cfg.eps;
  p.lambda = h->cfg.lambda;
  p.beta = h->cfg.beta;
  p.Rp = attention_row_stride(dm.R);
  p.pmax = h->ws.pmax;
  p.usage = h->ws.usage;
  p.pad = pad;
  p.n_carry = n_carry;
  p.credit_in = credit_in;
  p.credit_post = credit_post;
  p.mass = mass;
  p.score = score;
  if (T <= unit::kSmemT) {
    int nt, ept;
    unit::mass_shape(T, &nt, &ept);
    auto k = nt == 256    ? mass_post_smem_kernel<256, 16>
             : ept == 4  ? mass_post_smem_kernel<128, 4>
             : ept == 6  ? mass_post_smem_kernel<128, 6>
             : ept == 8  ? mass_post_smem_kernel<128, 8>
             : ept == 12 ? mass_post_smem_kernel<128, 12>
                         : mass_post_smem_kernel<128, 16>;
    k<<<dm.U, nt, 0, s>>>(p);
  } else {
    mass_post_kernel<1024><<<dm.U, 1024, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kvc
