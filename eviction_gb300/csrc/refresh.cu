// refresh.cu -- query-similarity refresh trigger, one warp per (layer, sequence).
//
// "RefreshKV: Updating Small KV Cache During Long-form Generation", dynamic
// scheduling: every S-th decode step each layer compares the current token's
// query, averaged over all query heads, with the averaged query of its most
// recent full-attention step by cosine similarity; below the threshold s it
// takes a full step, and that query becomes the reference.  A zero reference
// (no full step yet) or a zero query (cosine undefined) decides a refresh.
// Sums run in fp32 in a fixed order (heads in order per element, then a fixed
// butterfly over the warp), so repeated calls give the same bits.
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kRowsPerBlock = 4;  // one warp per (layer, sequence) row

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__global__ void __launch_bounds__(32 * kRowsPerBlock)
    refresh_kernel(const uint16_t* __restrict__ q, float* __restrict__ q_ref, int rows, int Hq,
                   int d, float threshold, int32_t* __restrict__ flag, float* __restrict__ sim) {
  const int row = blockIdx.x * kRowsPerBlock + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;  // warp-uniform
  const uint16_t* qr = q + static_cast<size_t>(row) * Hq * d;
  float* ref = q_ref + static_cast<size_t>(row) * d;
  const float inv_h = 1.0f / static_cast<float>(Hq);
  float dot = 0.f, nq = 0.f, nr = 0.f;
  for (int i = lane; i < d; i += 32) {
    float m = 0.f;
    for (int hq = 0; hq < Hq; ++hq) m += bf16_bits_to_float(qr[static_cast<size_t>(hq) * d + i]);
    m *= inv_h;
    const float r = ref[i];
    dot = fmaf(m, r, dot);
    nq = fmaf(m, m, nq);
    nr = fmaf(r, r, nr);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
    nq += __shfl_xor_sync(0xffffffffu, nq, o);
    nr += __shfl_xor_sync(0xffffffffu, nr, o);
  }
  const bool defined = nq > 0.f && nr > 0.f;
  const float c = defined ? dot / (sqrtf(nq) * sqrtf(nr)) : -2.f;
  const bool refresh = !defined || c < threshold;
  if (lane == 0) {
    sim[row] = c;
    flag[row] = refresh ? 1 : 0;
  }
  if (refresh) {
    __syncwarp();
    for (int i = lane; i < d; i += 32) {
      float m = 0.f;
      for (int hq = 0; hq < Hq; ++hq) m += bf16_bits_to_float(qr[static_cast<size_t>(hq) * d + i]);
      ref[i] = m * inv_h;
    }
  }
}

}  // namespace

cudaError_t launch_refresh(const kvc_handle* h, const uint16_t* q, float* q_ref,
                           float threshold, int32_t* flag, float* sim, cudaStream_t s) {
  const int rows = h->dims.L * h->dims.B;
  const int Hq = h->dims.H * h->dims.G;
  const int grid = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  refresh_kernel<<<grid, 32 * kRowsPerBlock, 0, s>>>(q, q_ref, rows, Hq, h->dims.d, threshold,
                                                      flag, sim);
  return cudaGetLastError();
}

}  // namespace kvc
