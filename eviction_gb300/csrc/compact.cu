// compact.cu -- physical gather-compaction of K, V and the credit.
//
// "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Method,
// Key design 4: the sorted kept indices gather K and V into a fixed-length
// per-head cache (a real copy, not a mask); Key design 1: the credit follows
// the same indices.  Rows past n_kept are written as zeros.
//
// HBM-bound bit copy.  A row of d bf16 is d/8 16-byte vectors; consecutive
// threads take consecutive vectors, so a warp moves 512 contiguous bytes per
// instruction for K and again for V.  Grid: units x row blocks, sized to fill
// every SM several times over.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 128;

// gridDim.y is at most 65535: larger unit counts launch in chunks of units
constexpr int kMaxGridY = 65535;

struct CompactParams {
  int T, budget, vecs;  // vecs = 16-byte vectors per row
  int unit0;            // first unit of this launch
  const uint4* k;
  const uint4* v;
  const float* credit;
  const int32_t* kept_idx;
  const int32_t* n_kept;
  uint4* k_out;
  uint4* v_out;
  float* credit_out;
  uint32_t* status;
};

__global__ void __launch_bounds__(kThreads)
    compact_kernel(CompactParams p) {
  __shared__ int32_t s_src[kRowsPerBlock];
  const int u = p.unit0 + static_cast<int>(blockIdx.y);
  const int r0 = blockIdx.x * kRowsPerBlock;
  const int rows = min(kRowsPerBlock, p.budget - r0);
  const int nk = p.n_kept[u];
  for (int r = threadIdx.x; r < rows; r += kThreads) {
    const int rr = r0 + r;
    int src = (rr < nk) ? p.kept_idx[static_cast<size_t>(u) * p.budget + rr] : -1;
    if (src >= p.T || src < -1 || (rr < nk && src < 0)) {  // not a slot: zero row
      atomicOr(p.status, KVC_STATUS_BAD_INDEX);
      src = -1;
    }
    s_src[r] = src;
    p.credit_out[static_cast<size_t>(u) * p.budget + rr] =
        (src >= 0) ? p.credit[static_cast<size_t>(u) * p.T + src] : 0.f;
  }
  __syncthreads();
  const size_t in_base = static_cast<size_t>(u) * p.T * p.vecs;
  const size_t out_base = (static_cast<size_t>(u) * p.budget + r0) * p.vecs;
  const int total = rows * p.vecs;
  constexpr int kUnroll = 4;
  for (int x0 = threadIdx.x; x0 < total; x0 += kThreads * kUnroll) {
    uint4 kv[kUnroll], vv[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int x = x0 + j * kThreads;
      kv[j] = make_uint4(0, 0, 0, 0);
      vv[j] = make_uint4(0, 0, 0, 0);
      if (x < total) {
        const int r = x / p.vecs, c = x - r * p.vecs;
        const int src = s_src[r];
        if (src >= 0) {
          const size_t off = in_base + static_cast<size_t>(src) * p.vecs + c;
          kv[j] = __ldg(p.k + off);
          vv[j] = __ldg(p.v + off);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int x = x0 + j * kThreads;
      if (x < total) {
        p.k_out[out_base + x] = kv[j];
        p.v_out[out_base + x] = vv[j];
      }
    }
  }
}

}  // namespace

cudaError_t launch_compact(const kvc_handle* h, const uint16_t* k,
                           const uint16_t* v, const float* credit_post, int T,
                           const int32_t* kept_idx, const int32_t* n_kept,
                           uint16_t* k_out, uint16_t* v_out,
                           float* credit_out, cudaStream_t s) {
  CompactParams p;
  p.T = T;
  p.budget = h->cfg.budget;
  p.vecs = h->dims.d * 2 / 16;
  p.k = reinterpret_cast<const uint4*>(k);
  p.v = reinterpret_cast<const uint4*>(v);
  p.credit = credit_post;
  p.kept_idx = kept_idx;
  p.n_kept = n_kept;
  p.k_out = reinterpret_cast<uint4*>(k_out);
  p.v_out = reinterpret_cast<uint4*>(v_out);
  p.credit_out = credit_out;
  p.status = h->ws.status;
  const int U = h->dims.U;
  for (int u0 = 0; u0 < U; u0 += kMaxGridY) {
    p.unit0 = u0;
    dim3 grid((p.budget + kRowsPerBlock - 1) / kRowsPerBlock, min(kMaxGridY, U - u0));
    compact_kernel<<<grid, kThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kvc
