// kvc_noalloc.cu -- kvc_mass for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they compress the
// cache: an inference engine that reserved all free device memory for its KV
// pool up front, or code running where allocation is not allowed.  For them
// kvc_mass_noalloc runs the same kernels as kvc_mass without a handle: its
// scratch (per-query softmax statistics and raw usage) lives in a fixed
// file-scope device array that every GPU loading this library holds until the
// process exits.  The caller passes every input and output.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it (one atomic
// slot per device, so two host threads making their first call at once both
// store the same address); make that first call before any stream capture.  The
// cached address belongs to the device's primary context: after
// cudaDeviceReset on that device it is stale, and this entry point must not be
// used on that device again in the process.  All calls share the array, so
// calls that overlap on the GPU (two streams, two threads) race and must not be
// issued; the array keeps the last call's contents, and nothing in it needs to
// start at zero (every scratch value is written before it is read).
#include <atomic>
#include <cmath>
#include <cstdio>
#include <string>

#include "kvc_internal.cuh"

namespace kvc {
size_t attention_usage_smem_bytes(int d, int R);
int attention_row_stride(int R);
}  // namespace kvc

namespace {

// 4 MiB of scratch (KVC_NOALLOC_SCRATCH_FLOATS floats), 256-byte aligned.
static __device__ __align__(256) float g_noalloc_scratch[KVC_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
std::atomic<float*> g_scratch_ptr[kMaxDevices] = {};

size_t align_floats(size_t n) { return (n + 63) & ~size_t(63); }  // 256-byte steps

int config_error(const char* why) {
  std::fprintf(stderr, "kvc_mass_noalloc: %s\n", why);
  return KVC_ERR_ARG;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int kvc_mass_noalloc(const kvc_config* cfg, const uint16_t* q, const uint16_t* k,
                                int T, const int32_t* pad, const int32_t* n_carry,
                                const float* credit_in, float* credit_post, float* mass,
                                float* score, uint32_t* status, void* stream) {
  std::string why;
  const int vrc = kvc::validate_config(cfg, &why);
  if (vrc != KVC_OK) {
    std::fprintf(stderr, "kvc_mass_noalloc: %s\n", why.c_str());
    return vrc;
  }
  if (T < 1 || T > cfg->max_T) {
    std::fprintf(stderr, "kvc_mass_noalloc: T must lie in [1, max_T]\n");
    return KVC_ERR_SHAPE;
  }
  if (!status)
    return config_error("status is null: device failure reports (a bounded wait that ran "
                        "out, a bad index) have nowhere else to go");
  if (!q || !k || !pad || !n_carry || !credit_in || !credit_post || !mass || !score)
    return config_error("null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(pad) || !aligned16(n_carry) ||
      !aligned16(credit_in) || !aligned16(credit_post) || !aligned16(mass) ||
      !aligned16(score) || (reinterpret_cast<uintptr_t>(status) & 3u)) {
    std::fprintf(stderr, "kvc_mass_noalloc: pointer not 16-byte aligned\n");
    return KVC_ERR_ALIGN;
  }

  // device and its scratch address (set-up on the first call per device)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return KVC_ERR_DEVICE;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return KVC_ERR_DEVICE;
  }
  if (major != 10 || minor != 3) return KVC_ERR_DEVICE;
  float* base = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!base) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&base), g_noalloc_scratch);
    if (e != cudaSuccess || !base) {
      std::fprintf(stderr, "kvc_mass_noalloc: cudaGetSymbolAddress failed: %s\n",
                   cudaGetErrorString(e));
      cudaGetLastError();
      return KVC_ERR_CUDA;
    }
    g_scratch_ptr[dev].store(base, std::memory_order_release);
  }

  // a handle on the stack: same kernels and launch shapes as kvc_mass
  kvc_handle h;
  h.cfg = *cfg;
  h.device = dev;
  h.num_sms = sms;
  kvc::Dims& d = h.dims;
  d.L = cfg->n_layers;
  d.B = cfg->batch;
  d.H = cfg->n_kv_heads;
  d.G = cfg->group;
  d.W = cfg->window;
  d.d = cfg->head_dim;
  d.R = d.G * d.W;  // both products bounded by the validation above
  d.U = d.L * d.B * d.H;
  int smem_optin = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (kvc::attention_usage_smem_bytes(d.d, d.R) > static_cast<size_t>(smem_optin))
    return KVC_ERR_UNSUPPORTED;

  const size_t U = d.U, Rp = kvc::attention_row_stride(d.R);
  const size_t n_negb = align_floats(U * Rp), n_pmax = align_floats(U * Rp);
  const size_t n_use = align_floats(U * static_cast<size_t>(T));
  const size_t need = n_negb + n_pmax + n_use;
  if (need > KVC_NOALLOC_SCRATCH_FLOATS) {
    std::fprintf(stderr,
                 "kvc_mass_noalloc: needs %zu scratch floats (units * (2*rows + T)), the "
                 "fixed maximum is %u; call it per layer or on fewer sequences\n",
                 need, KVC_NOALLOC_SCRATCH_FLOATS);
    return KVC_ERR_SHAPE;
  }
  h.ws.negb = base;
  h.ws.pmax = base + n_negb;
  h.ws.usage = base + n_negb + n_pmax;
  h.ws.status = status;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  const double sc = cfg->softmax_scale > 0.f ? static_cast<double>(cfg->softmax_scale)
                                             : 1.0 / std::sqrt(static_cast<double>(d.d));
  kvc::UsageArgs a{q, k, pad, T, static_cast<float>(sc * 1.4426950408889634)};
  for (int pass = 1; pass <= 2; ++pass) {
    e = cfg->attn_kernel == 2 ? kvc::launch_attention_usage_pair(&h, a, pass, s, nullptr)
                              : kvc::launch_attention_usage(&h, a, pass, s, nullptr);
    if (e != cudaSuccess) {
      std::fprintf(stderr, "kvc_mass_noalloc: attention kernels: %s\n", cudaGetErrorString(e));
      cudaGetLastError();
      return KVC_ERR_CUDA;
    }
  }
  e = kvc::launch_mass_post(&h, T, pad, n_carry, credit_in, credit_post, mass, score, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KVC_ERR_CUDA;
  }
  return KVC_OK;
}
