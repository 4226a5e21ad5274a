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
// Units up to 4096 slots take one pass with the filled usage in shared memory
// and per-slot values in registers; longer ones sweep global memory (the
// unit's data stays in L1/L2 between sweeps).  Every sum is a strided
// per-thread pass plus one fixed-order block reduction, so repeated runs give
// identical bits.
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
int attention_row_stride(int R);
namespace {

constexpr int kThreads = 256;

template <int NT = kThreads>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();  // red may still be read by a previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = (lane < NT / 32) ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) red[NT / 32] = t;
  }
  __syncthreads();
  return red[NT / 32];
}

template <int NT = kThreads>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = (lane < NT / 32) ? red[lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (lane == 0) red[NT / 32] = t;
  }
  __syncthreads();
  return red[NT / 32];
}

struct PostParams {
  int T, R, W, G, B, H;
  int avg_pool, max_pool;
  float eps, lambda, beta;
  int Rp;
  const float* pmax;  // [U][Rp] largest probability of each row (0 if absent)
  float* usage;       // [U][T] raw usage, filled in place
  const int32_t* pad;
  const int32_t* n_carry;
  const float* credit_in;
  float* credit_post;
  float* mass;
  float* score;
};

// Units longer than kSmemT slots sweep global memory.  They are few (a long
// cache holds few sequences), so each takes a CTA of NT = 1024 threads: four
// times the loads in flight per unit of a 256-thread CTA.
template <int NT>
__global__ void __launch_bounds__(NT)
    mass_post_kernel(PostParams p) {
  __shared__ float red[NT / 32 + 1];
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

  // score = max-pooled usage; first mass total
  const int ra = p.avg_pool / 2, rm = p.max_pool / 2;
  const float inv_k = 1.0f / static_cast<float>(p.avg_pool);
  float tot = 0.f;
  for (int i = threadIdx.x; i < T; i += NT) {
    if (i < pad) {
      score[i] = -INFINITY;
      continue;
    }
    float mx = -INFINITY;
    for (int t = max(pad, i - rm); t <= min(T - 1, i + rm); ++t) mx = fmaxf(mx, a[t]);
    score[i] = mx;
    float s = 0.f;
    for (int t = max(pad, i - ra); t <= min(T - 1, i + ra); ++t) s += a[t];
    tot += fmaxf(s * inv_k, 0.f) + p.eps;
  }
  const float total1 = block_sum<NT>(tot, red);

  // mass and credit
  const int n_carry = min(max(p.n_carry[b], 0), T - pad);
  const float lam = p.lambda;
  float ctot = 0.f;
  for (int i = threadIdx.x; i < T; i += NT) {
    if (i < pad) {
      mass[i] = 0.f;
      cpost[i] = 0.f;
      continue;
    }
    float s = 0.f;
    for (int t = max(pad, i - ra); t <= min(T - 1, i + ra); ++t) s += a[t];
    const float m = (fmaxf(s * inv_k, 0.f) + p.eps) / total1;
    const float prior = (i < pad + n_carry) ? cin[i] : m;
    const float c = lam * prior + (1.0f - lam) * m;
    mass[i] = m;
    cpost[i] = c;
    ctot += c;
  }
  const float c_total = block_sum<NT>(ctot, red);

  // mix and normalise
  const float beta = p.beta;
  float mtot = 0.f;
  for (int i = pad + threadIdx.x; i < T; i += NT) {
    const float m = mass[i];
    const float cn = (c_total > 0.f) ? cpost[i] / c_total : m;
    const float mix = beta * m + (1.0f - beta) * cn;
    mass[i] = mix;
    mtot += mix;
  }
  const float mix_total = block_sum<NT>(mtot, red);
  for (int i = pad + threadIdx.x; i < T; i += NT) mass[i] = mass[i] / mix_total;
}

// Units of up to kSmemT slots: one pass.  The filled usage of the unit sits in
// shared memory (the pooling windows read it there), each thread keeps its
// slots' values in registers across the normalisations, and score, mass and
// credit are written once.  The arithmetic and the summation order (per thread
// over its slots, then block_sum) are those of the general kernel below.
constexpr int kSmemT = 4096;

// Latency-bound: one CTA per unit, so the more CTAs an SM holds the better.
// Up to 8 slots per thread the kernel fits in 32 registers without spilling,
// which lets 8 CTAs share an SM (5 at its natural 47 registers).
template <int kEpt>  // slots per thread: T <= kEpt * kThreads
__global__ void __launch_bounds__(kThreads, kEpt <= 8 ? 8 : 4)
    mass_post_smem_kernel(PostParams p) {
  __shared__ float red[kThreads / 32 + 1];
  __shared__ float a[kEpt * kThreads];
  const int u = blockIdx.x;
  const int b = (u / p.H) % p.B;
  const int T = p.T;
  const int pad = min(max(p.pad[b], 0), T);
  const size_t base = static_cast<size_t>(u) * T;
  float* mass = p.mass + base;
  float* score = p.score + base;
  float* cpost = p.credit_post + base;
  const float* cin = p.credit_in + base;
  const float* usage = p.usage + base;

  if (pad >= T) {
    for (int i = threadIdx.x; i < T; i += kThreads) {
      mass[i] = 0.f;
      score[i] = -INFINITY;
      cpost[i] = 0.f;
    }
    return;
  }
  const int n_carry = min(max(p.n_carry[b], 0), T - pad);
  // this thread's credit-in values, loaded early (used after two reductions)
  float cprior[kEpt];
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = threadIdx.x + k * kThreads;
    cprior[k] = (i >= pad && i < pad + n_carry) ? cin[i] : 0.f;
  }

  float pm = 0.f;
  for (int r = threadIdx.x; r < p.R; r += kThreads)
    pm = fmaxf(pm, p.pmax[static_cast<size_t>(u) * p.Rp + r]);
  const float fill = block_max(pm, red);

  const int j_lo = max(0, pad - (T - p.W));
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = threadIdx.x + k * kThreads;
    if (i < T) {
      const int unseen = max(0, min(p.W, i - T + p.W) - j_lo) * p.G;
      a[i] = i >= pad ? usage[i] + fill * static_cast<float>(unseen) : 0.f;
    }
  }
  __syncthreads();

  const int ra = p.avg_pool / 2, rm = p.max_pool / 2;
  const float inv_k = 1.0f / static_cast<float>(p.avg_pool);
  float up[kEpt];  // max(avg pool, 0) + eps
  float tot = 0.f;
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = threadIdx.x + k * kThreads;
    up[k] = 0.f;
    if (i >= T) continue;
    if (i < pad) {
      score[i] = -INFINITY;
      continue;
    }
    float mx = -INFINITY;
    for (int t = max(pad, i - rm); t <= min(T - 1, i + rm); ++t) mx = fmaxf(mx, a[t]);
    score[i] = mx;
    float sm = 0.f;
    for (int t = max(pad, i - ra); t <= min(T - 1, i + ra); ++t) sm += a[t];
    up[k] = fmaxf(sm * inv_k, 0.f) + p.eps;
    tot += up[k];
  }
  const float total1 = block_sum(tot, red);

  const float lam = p.lambda;
  float ctot = 0.f;
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = threadIdx.x + k * kThreads;
    if (i < pad || i >= T) continue;
    const float m = up[k] / total1;
    const float prior = (i < pad + n_carry) ? cprior[k] : m;
    const float c = lam * prior + (1.0f - lam) * m;
    up[k] = m;
    cprior[k] = c;
    ctot += c;
  }
  const float c_total = block_sum(ctot, red);

  const float beta = p.beta;
  float mtot = 0.f;
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = threadIdx.x + k * kThreads;
    if (i < pad || i >= T) continue;
    const float m = up[k];
    const float cn = (c_total > 0.f) ? cprior[k] / c_total : m;
    const float mix = beta * m + (1.0f - beta) * cn;
    up[k] = mix;
    mtot += mix;
  }
  const float mix_total = block_sum(mtot, red);
#pragma unroll
  for (int k = 0; k < kEpt; ++k) {
    const int i = threadIdx.x + k * kThreads;
    if (i >= T) continue;
    if (i < pad) {
      mass[i] = 0.f;
      cpost[i] = 0.f;
    } else {
      mass[i] = up[k] / mix_total;
      cpost[i] = cprior[k];
    }
  }
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
  if (T <= 4 * kThreads)
    mass_post_smem_kernel<4><<<dm.U, kThreads, 0, s>>>(p);
  else if (T <= 8 * kThreads)
    mass_post_smem_kernel<8><<<dm.U, kThreads, 0, s>>>(p);
  else if (T <= kSmemT)
    mass_post_smem_kernel<kSmemT / kThreads><<<dm.U, kThreads, 0, s>>>(p);
  else
    mass_post_kernel<1024><<<dm.U, 1024, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvc
