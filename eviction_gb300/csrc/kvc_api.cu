// kvc_api.cu -- host side of the C ABI declared in include/kvc.h: argument
// validation, the handle and its workspace, and the stage / event entry points
// (each a fixed sequence of kernel launches on the caller's stream).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "kvc_internal.cuh"

namespace kvc {
size_t attention_usage_smem_bytes(int d, int R);
int attention_row_stride(int R);
size_t segment_smem_bytes(const kvc_config& c, int T);
size_t select_smem_bytes(const kvc_config& c, int T);
}  // namespace kvc

namespace {

constexpr int kMaxT = 65536;
constexpr int kMaxRows = 4096;  // G*W query rows per unit

int fail(kvc_handle* h, int code, const std::string& msg) {
  if (h) h->last_error = msg;
  return code;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

int check_T(kvc_handle* h, int T) {
  if (T < 1 || T > h->cfg.max_T)
    return fail(h, KVC_ERR_SHAPE, "T must lie in [1, max_T]");
  return KVC_OK;
}

int cuda_fail(kvc_handle* h, cudaError_t e, const char* where) {
  return fail(h, KVC_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

const char* const kKernelNames[kvc::kNumKernels] = {
    "usage_pass1_rowstats_tcgen05", "usage_pass2_colsum_tcgen05", "mass_pool_ema",
    "segment_quota", "select_topk", "gather_compact", "refresh_trigger", "compact_paged",
    "redundancy_score", "mass_segment_select"};

cudaEvent_t prof_event(kvc_handle* h) {
  auto& P = h->prof;
  if (!P.pool.empty()) {
    cudaEvent_t e = P.pool.back();
    P.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Record the start of one kernel launch (nullptr when tracing is off).
cudaEvent_t mark_begin(kvc_handle* h, cudaStream_t s) {
  if (!h->prof.enabled) return nullptr;
  cudaEvent_t e = prof_event(h);
  if (e) cudaEventRecord(e, s);
  return e;
}

void mark_end(kvc_handle* h, int kernel, cudaEvent_t begin, cudaStream_t s) {
  if (!begin) return;
  cudaEvent_t e = prof_event(h);
  if (!e) {
    h->prof.pool.push_back(begin);
    return;
  }
  cudaEventRecord(e, s);
  h->prof.pending.push_back({kernel, begin, e});
}

#define KVC_REQUIRE_PTR(p)                                                    \
  do {                                                                        \
    if (!(p)) return fail(h, KVC_ERR_ARG, "null pointer: " #p);               \
    if (!aligned16(p)) return fail(h, KVC_ERR_ALIGN, "not 16-byte aligned: " #p); \
  } while (0)

float scale_log2_of(const kvc_config& c) {
  const double s = c.softmax_scale > 0.f ? static_cast<double>(c.softmax_scale)
                                         : 1.0 / std::sqrt(static_cast<double>(c.head_dim));
  return static_cast<float>(s * 1.4426950408889634);
}

// Step 1: both passes of the window attention usage into the workspace.
int run_usage(kvc_handle* h, const uint16_t* q, const uint16_t* k, int T, const int32_t* pad,
              cudaStream_t s) {
  kvc::UsageArgs a{q, k, pad, T, scale_log2_of(h->cfg)};
  std::string err;
  for (int pass = 1; pass <= 2; ++pass) {
    cudaEvent_t b = mark_begin(h, s);
    cudaError_t e = h->cfg.attn_kernel == 2
                        ? kvc::launch_attention_usage_pair(h, a, pass, s, &err)
                        : kvc::launch_attention_usage(h, a, pass, s, &err);
    if (e != cudaSuccess)
      return err.empty() ? cuda_fail(h, e, "attention usage") : fail(h, KVC_ERR_CUDA, err);
    mark_end(h, pass == 1 ? kvc::kKernelUsagePass1 : kvc::kKernelUsagePass2, b, s);
  }
  return KVC_OK;
}

int run_mass(kvc_handle* h, const uint16_t* q, const uint16_t* k, int T, const int32_t* pad,
             const int32_t* n_carry, const float* credit_in, float* credit_post, float* mass,
             float* score, cudaStream_t s) {
  int rc = run_usage(h, q, k, T, pad, s);
  if (rc) return rc;
  cudaEvent_t b = mark_begin(h, s);
  cudaError_t e =
      kvc::launch_mass_post(h, T, pad, n_carry, credit_in, credit_post, mass, score, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "mass");
  mark_end(h, kvc::kKernelMass, b, s);
  return KVC_OK;
}

int run_segment_quota(kvc_handle* h, const float* mass, int T, const int32_t* pad,
                      int32_t* seg_start, int32_t* seg_len, int32_t* quota, int32_t* n_seg,
                      cudaStream_t s) {
  cudaEvent_t b = mark_begin(h, s);
  cudaError_t e =
      kvc::launch_segment_quota(h, mass, T, pad, seg_start, seg_len, quota, n_seg, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "segment_quota");
  mark_end(h, kvc::kKernelSegmentQuota, b, s);
  return KVC_OK;
}

int run_select(kvc_handle* h, const float* score, int T, const int32_t* pad,
               const int32_t* seg_start, const int32_t* seg_len, const int32_t* quota,
               const int32_t* n_seg, int32_t* kept_idx, int32_t* n_kept, cudaStream_t s) {
  cudaEvent_t b = mark_begin(h, s);
  cudaError_t e = kvc::launch_select(h, score, T, pad, seg_start, seg_len, quota, n_seg,
                                     kept_idx, n_kept, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "select");
  mark_end(h, kvc::kKernelSelect, b, s);
  return KVC_OK;
}

int run_redundancy(kvc_handle* h, const uint16_t* k, const float* score, int T,
                   const int32_t* pad, float* sel, float* red, cudaStream_t s) {
  cudaEvent_t b = mark_begin(h, s);
  cudaError_t e = kvc::launch_redundancy(h, k, score, T, pad, sel, red, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "redundancy score");
  mark_end(h, kvc::kKernelRedundancy, b, s);
  return KVC_OK;
}

int run_compact(kvc_handle* h, const uint16_t* k, const uint16_t* v, const float* credit_post,
                int T, const int32_t* kept_idx, const int32_t* n_kept, uint16_t* k_out,
                uint16_t* v_out, float* credit_out, cudaStream_t s) {
  cudaEvent_t b = mark_begin(h, s);
  cudaError_t e = kvc::launch_compact(h, k, v, credit_post, T, kept_idx, n_kept, k_out, v_out,
                                      credit_out, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "compact");
  mark_end(h, kvc::kKernelCompact, b, s);
  return KVC_OK;
}

// Steps 1-4 on validated pointers: usage, mass and credit, segments and
// quotas, kept indices.  Units of up to 4096 slots run mass, segmentation and
// selection as one fused launch (same bits as the three stand-alone kernels);
// the redundancy mix sits between segmentation and selection, so with it on,
// and for longer units, the stand-alone kernels run.
int run_mass_select(kvc_handle* h, const uint16_t* q, const uint16_t* k, int T,
                    const int32_t* pad, const int32_t* n_carry, const float* credit_in,
                    float* credit_post, float* mass, float* score, int32_t* seg_start,
                    int32_t* seg_len, int32_t* quota, int32_t* n_seg, int32_t* kept_idx,
                    int32_t* n_kept, cudaStream_t s) {
  const size_t fused_smem = kvc::unit_post_smem_bytes(h->cfg, T);
  if (!(h->cfg.redundancy_sigma > 0.f) && fused_smem > 0 && fused_smem <= h->smem_optin) {
    int rc = run_usage(h, q, k, T, pad, s);
    if (rc) return rc;
    cudaEvent_t b = mark_begin(h, s);
    cudaError_t e = kvc::launch_unit_post(h, T, pad, n_carry, credit_in, credit_post, mass,
                                          score, seg_start, seg_len, quota, n_seg, kept_idx,
                                          n_kept, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "mass/segment/select");
    mark_end(h, kvc::kKernelUnitPost, b, s);
    return KVC_OK;
  }
  int rc = run_mass(h, q, k, T, pad, n_carry, credit_in, credit_post, mass, score, s);
  if (rc) return rc;
  rc = run_segment_quota(h, mass, T, pad, seg_start, seg_len, quota, n_seg, s);
  if (rc) return rc;
  if (h->cfg.redundancy_sigma > 0.f) {  // the selection score, in place
    rc = run_redundancy(h, k, score, T, pad, score, nullptr, s);
    if (rc) return rc;
  }
  return run_select(h, score, T, pad, seg_start, seg_len, quota, n_seg, kept_idx, n_kept, s);
}

// Steps 1-6 on validated pointers, intermediates in the workspace.
int run_event(kvc_handle* h, const uint16_t* q, const uint16_t* k, const uint16_t* v, int T,
              const int32_t* pad, const int32_t* n_carry, const float* credit_in,
              uint16_t* k_out, uint16_t* v_out, float* credit_out, int32_t* kept_idx,
              int32_t* n_kept, cudaStream_t s) {
  const kvc::Workspace& w = h->ws;
  int rc = run_mass_select(h, q, k, T, pad, n_carry, credit_in, w.credit_post, w.mass, w.score,
                           w.seg_start, w.seg_len, w.quota, w.n_seg, kept_idx, n_kept, s);
  if (rc) return rc;
  return run_compact(h, k, v, w.credit_post, T, kept_idx, n_kept, k_out, v_out, credit_out, s);
}

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

void destroy_host_io(kvc::HostIO& io) {
  if (io.in) cudaStreamDestroy(io.in);
  if (io.start) cudaEventDestroy(io.start);
  for (int j = 0; j < 2; ++j) {
    if (io.out[j]) cudaStreamDestroy(io.out[j]);
    if (io.end[j]) cudaEventDestroy(io.end[j]);
  }
  for (int i = 0; i < kvc::kMaxHostStages; ++i) {
    if (io.landed[i]) cudaEventDestroy(io.landed[i]);
    if (io.done[i]) cudaEventDestroy(io.done[i]);
  }
  io = kvc::HostIO{};
}

bool create_host_io(kvc::HostIO& io) {
  bool ok = cudaStreamCreateWithFlags(&io.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&io.start, cudaEventDisableTiming) == cudaSuccess;
  for (int j = 0; ok && j < 2; ++j)
    ok = cudaStreamCreateWithFlags(&io.out[j], cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&io.end[j], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kvc::kMaxHostStages; ++i)
    ok = cudaEventCreateWithFlags(&io.landed[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&io.done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    destroy_host_io(io);
  }
  return ok;
}

}  // namespace

namespace kvc {

int validate_config(const kvc_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return KVC_ERR_ARG;
  };
  if (!c) return bad("config is null");
  if (c->n_layers < 1 || c->batch < 1 || c->n_kv_heads < 1 || c->group < 1)
    return bad("n_layers, batch, n_kv_heads and group must be >= 1");
  if (c->window < 1 || c->budget < 1 || c->max_T < 1)
    return bad("window, budget and max_T must be >= 1");
  if (c->max_T > kMaxT) return bad("max_T must be <= 65536");
  if (c->avg_pool < 1 || c->avg_pool % 2 == 0 || c->max_pool < 1 || c->max_pool % 2 == 0)
    return bad("avg_pool and max_pool must be odd and >= 1");
  if (!std::isfinite(c->delta) || static_cast<double>(c->delta) < 1.0 / 1024.0)
    return bad("delta must be finite and >= 1/1024");
  if (c->seg_min < 1 || c->seg_max < 2 * c->seg_min || c->seg_max < 16 || c->seg_max > 4096)
    return bad("need 1 <= seg_min, 2*seg_min <= seg_max, 16 <= seg_max <= 4096");
  if (c->q_min < 0 || c->n_sink < 0 || c->n_recent < 0)
    return bad("q_min, n_sink and n_recent must be >= 0");
  if (!(c->lambda >= 0.f && c->lambda <= 1.f) || !(c->beta >= 0.f && c->beta <= 1.f))
    return bad("lambda and beta must lie in [0, 1]");
  if (!(c->eps > 0.f) || !std::isfinite(c->eps)) return bad("eps must be finite and > 0");
  if (!(c->softmax_scale >= 0.f) || !std::isfinite(c->softmax_scale))
    return bad("softmax_scale must be finite and >= 0");
  if (c->seg_fixed < 0 || (c->seg_fixed > 0 && c->seg_fixed < c->seg_min))
    return bad("seg_fixed must be 0 or >= seg_min");
  if ((c->quota_by_len != 0 && c->quota_by_len != 1) ||
      (c->global_topk != 0 && c->global_topk != 1))
    return bad("quota_by_len and global_topk must be 0 or 1");
  if (!(c->redundancy_sigma >= 0.f && c->redundancy_sigma <= 1.f))
    return bad("redundancy_sigma must lie in [0, 1] (0 = off)");
  if (c->attn_kernel < 0 || c->attn_kernel > 2) return bad("attn_kernel must be 0, 1 or 2");
  if (c->head_dim != 64 && c->head_dim != 128) {
    *why = "head_dim must be 64 or 128";
    return KVC_ERR_UNSUPPORTED;
  }
  const long long rows = static_cast<long long>(c->group) * c->window;
  if (rows > kMaxRows) {
    *why = "group * window must be <= 4096";
    return KVC_ERR_UNSUPPORTED;
  }
  const long long units = static_cast<long long>(c->n_layers) * c->batch * c->n_kv_heads;
  if (units * c->max_T >= (1ll << 31) || units * rows >= (1ll << 31)) {
    *why = "units * max_T and units * group * window must be < 2^31";
    return KVC_ERR_UNSUPPORTED;
  }
  return KVC_OK;
}

}  // namespace kvc

extern "C" {

void kvc_default_config(kvc_config* c) {
  if (!c) return;
  std::memset(c, 0, sizeof(*c));
  c->window = 128;
  c->avg_pool = 5;
  c->max_pool = 7;
  c->delta = 0.1f;
  c->seg_min = 16;
  c->seg_max = 256;
  c->q_min = 1;
  c->n_sink = 4;
  c->n_recent = 64;
  c->lambda = 0.9f;
  c->beta = 0.9f;
  c->eps = 1e-6f;
  c->softmax_scale = 0.f;
}

const char* kvc_status_string(int code) {
  switch (code) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_ARG: return "KVC_ERR_ARG";
    case KVC_ERR_SHAPE: return "KVC_ERR_SHAPE";
    case KVC_ERR_ALIGN: return "KVC_ERR_ALIGN";
    case KVC_ERR_NOMEM: return "KVC_ERR_NOMEM";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA";
    case KVC_ERR_DEVICE: return "KVC_ERR_DEVICE";
    case KVC_ERR_TIMEOUT: return "KVC_ERR_TIMEOUT";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED";
    default: return "KVC_ERR_UNKNOWN";
  }
}

const char* kvc_last_error(const kvc_handle* h) {
  return h ? h->last_error.c_str() : "null handle";
}

int kvc_create(const kvc_config* cfg, kvc_handle** out) {
  if (!out) return KVC_ERR_ARG;
  *out = nullptr;
  std::string why;
  int rc = kvc::validate_config(cfg, &why);
  if (rc != KVC_OK) {
    std::fprintf(stderr, "kvc_create: %s\n", why.c_str());
    return rc;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KVC_ERR_DEVICE;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    cudaGetLastError();
    return KVC_ERR_DEVICE;
  }
  if (prop.major != 10 || prop.minor != 3) {
    std::fprintf(stderr, "kvc_create: device %d is sm_%d%d, this library is built for sm_103a\n",
                 dev, prop.major, prop.minor);
    return KVC_ERR_DEVICE;
  }
  kvc_handle* h = new (std::nothrow) kvc_handle();
  if (!h) return KVC_ERR_NOMEM;
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->smem_optin = prop.sharedMemPerBlockOptin;
  kvc::Dims& d = h->dims;
  d.L = cfg->n_layers;
  d.B = cfg->batch;
  d.H = cfg->n_kv_heads;
  d.G = cfg->group;
  d.W = cfg->window;
  d.d = cfg->head_dim;
  d.R = d.G * d.W;
  d.U = d.L * d.B * d.H;

  // shared-memory needs must fit the device
  const size_t smem_max = prop.sharedMemPerBlockOptin;
  if (kvc::attention_usage_smem_bytes(d.d, d.R) > smem_max ||
      kvc::segment_smem_bytes(*cfg, cfg->max_T) > smem_max - 16 * 1024 ||
      kvc::select_smem_bytes(*cfg, cfg->max_T) > smem_max - 1024 ||
      kvc::redundancy_smem_bytes(d.d, cfg->max_T) > smem_max) {
    delete h;
    std::fprintf(stderr, "kvc_create: configuration needs more shared memory than the device has\n");
    return KVC_ERR_UNSUPPORTED;
  }

  const size_t U = d.U, T = cfg->max_T;
  const size_t S = kvc::s_max_of(*cfg, cfg->max_T);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  const size_t Rp = kvc::attention_row_stride(d.R);
  const size_t o_negb = take(U * Rp * 4);
  const size_t o_pmax = take(U * Rp * 4);
  const size_t o_use = take(U * T * 4);
  const size_t o_mass = take(U * T * 4);
  const size_t o_score = take(U * T * 4);
  const size_t o_cp = take(U * T * 4);
  const size_t o_ss = take(U * S * 4);
  const size_t o_sl = take(U * S * 4);
  const size_t o_q = take(U * S * 4);
  const size_t o_ns = take(U * 4);
  const size_t o_st = take(256);
  void* base = nullptr;
  if (cudaMalloc(&base, off) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return KVC_ERR_NOMEM;
  }
  if (cudaMemset(base, 0, off) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(base);
    delete h;
    return KVC_ERR_CUDA;
  }
  char* p = static_cast<char*>(base);
  kvc::Workspace& w = h->ws;
  w.base = base;
  w.bytes = off;
  w.negb = reinterpret_cast<float*>(p + o_negb);
  w.pmax = reinterpret_cast<float*>(p + o_pmax);
  w.usage = reinterpret_cast<float*>(p + o_use);
  w.mass = reinterpret_cast<float*>(p + o_mass);
  w.score = reinterpret_cast<float*>(p + o_score);
  w.credit_post = reinterpret_cast<float*>(p + o_cp);
  w.seg_start = reinterpret_cast<int32_t*>(p + o_ss);
  w.seg_len = reinterpret_cast<int32_t*>(p + o_sl);
  w.quota = reinterpret_cast<int32_t*>(p + o_q);
  w.n_seg = reinterpret_cast<int32_t*>(p + o_ns);
  w.status = reinterpret_cast<uint32_t*>(p + o_st);
  if (!create_host_io(h->io)) {
    cudaFree(base);
    delete h;
    return KVC_ERR_CUDA;
  }
  *out = h;
  return KVC_OK;
}

void kvc_destroy(kvc_handle* h) {
  if (!h) return;
  if (h->ws.base) {
    cudaDeviceSynchronize();
    cudaFree(h->ws.base);
  }
  for (auto& m : h->prof.pending) {
    cudaEventDestroy(m.begin);
    cudaEventDestroy(m.end);
  }
  for (cudaEvent_t e : h->prof.pool) cudaEventDestroy(e);
  destroy_host_io(h->io);
  delete h;
}

int kvc_stage_sizes(const kvc_handle* h, int T, int* s_max) {
  if (!h || !s_max) return KVC_ERR_ARG;
  if (T < 1 || T > h->cfg.max_T) return KVC_ERR_SHAPE;
  *s_max = kvc::s_max_of(h->cfg, T);
  return KVC_OK;
}

int kvc_mass(kvc_handle* h, const uint16_t* q, const uint16_t* k, int T,
             const int32_t* pad, const int32_t* n_carry, const float* credit_in,
             float* credit_post, float* mass, float* score, void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  KVC_REQUIRE_PTR(q);
  KVC_REQUIRE_PTR(k);
  KVC_REQUIRE_PTR(pad);
  KVC_REQUIRE_PTR(n_carry);
  KVC_REQUIRE_PTR(credit_in);
  KVC_REQUIRE_PTR(credit_post);
  KVC_REQUIRE_PTR(mass);
  KVC_REQUIRE_PTR(score);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = run_mass(h, q, k, T, pad, n_carry, credit_in, credit_post, mass, score, s);
  return rc;
}

int kvc_segment_quota(kvc_handle* h, const float* mass, int T, const int32_t* pad,
                      int32_t* seg_start, int32_t* seg_len, int32_t* quota,
                      int32_t* n_seg, void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  KVC_REQUIRE_PTR(mass);
  KVC_REQUIRE_PTR(pad);
  KVC_REQUIRE_PTR(seg_start);
  KVC_REQUIRE_PTR(seg_len);
  KVC_REQUIRE_PTR(quota);
  KVC_REQUIRE_PTR(n_seg);
  return run_segment_quota(h, mass, T, pad, seg_start, seg_len, quota, n_seg,
                           static_cast<cudaStream_t>(stream));
}

int kvc_select(kvc_handle* h, const float* score, int T, const int32_t* pad,
               const int32_t* seg_start, const int32_t* seg_len, const int32_t* quota,
               const int32_t* n_seg, int32_t* kept_idx, int32_t* n_kept, void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  KVC_REQUIRE_PTR(score);
  KVC_REQUIRE_PTR(pad);
  KVC_REQUIRE_PTR(seg_start);
  KVC_REQUIRE_PTR(seg_len);
  KVC_REQUIRE_PTR(quota);
  KVC_REQUIRE_PTR(n_seg);
  KVC_REQUIRE_PTR(kept_idx);
  KVC_REQUIRE_PTR(n_kept);
  return run_select(h, score, T, pad, seg_start, seg_len, quota, n_seg, kept_idx, n_kept,
                    static_cast<cudaStream_t>(stream));
}

int kvc_compact(kvc_handle* h, const uint16_t* k, const uint16_t* v,
                const float* credit_post, int T, const int32_t* kept_idx,
                const int32_t* n_kept, uint16_t* k_out, uint16_t* v_out,
                float* credit_out, void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  KVC_REQUIRE_PTR(k);
  KVC_REQUIRE_PTR(v);
  KVC_REQUIRE_PTR(credit_post);
  KVC_REQUIRE_PTR(kept_idx);
  KVC_REQUIRE_PTR(n_kept);
  KVC_REQUIRE_PTR(k_out);
  KVC_REQUIRE_PTR(v_out);
  KVC_REQUIRE_PTR(credit_out);
  return run_compact(h, k, v, credit_post, T, kept_idx, n_kept, k_out, v_out, credit_out,
                     static_cast<cudaStream_t>(stream));
}

int kvc_redundancy_score(kvc_handle* h, const uint16_t* k, const float* score, int T,
                         const int32_t* pad, float* sel_score, float* redundancy,
                         void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  if (!(h->cfg.redundancy_sigma > 0.f))
    return fail(h, KVC_ERR_ARG, "redundancy_sigma is 0: the redundancy score is off");
  KVC_REQUIRE_PTR(k);
  KVC_REQUIRE_PTR(score);
  KVC_REQUIRE_PTR(pad);
  KVC_REQUIRE_PTR(sel_score);
  if (redundancy && !aligned16(redundancy))
    return fail(h, KVC_ERR_ALIGN, "not 16-byte aligned: redundancy");
  return run_redundancy(h, k, score, T, pad, sel_score, redundancy,
                        static_cast<cudaStream_t>(stream));
}

int kvc_compact_paged(kvc_handle* h, uint16_t* k_pool, uint16_t* v_pool, int n_blocks,
                      int block_size, int max_blocks, const int32_t* seq_len,
                      const int32_t* pad, const int32_t* kept_idx, const int32_t* n_kept,
                      const float* credit_post, int T, float* credit_out,
                      const int32_t* table_old, int32_t* table_new, int32_t* free_list,
                      int32_t* free_top, void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  if (n_blocks < 1 || block_size < 1 || max_blocks < 1)
    return fail(h, KVC_ERR_ARG, "n_blocks, block_size and max_blocks must be >= 1");
  if ((static_cast<int64_t>(block_size) * h->dims.d * 2) % 16 != 0)
    return fail(h, KVC_ERR_ALIGN, "block rows must be 16-byte multiples");
  KVC_REQUIRE_PTR(k_pool);
  KVC_REQUIRE_PTR(v_pool);
  KVC_REQUIRE_PTR(seq_len);
  KVC_REQUIRE_PTR(pad);
  KVC_REQUIRE_PTR(kept_idx);
  KVC_REQUIRE_PTR(n_kept);
  KVC_REQUIRE_PTR(credit_post);
  KVC_REQUIRE_PTR(credit_out);
  KVC_REQUIRE_PTR(table_old);
  KVC_REQUIRE_PTR(table_new);
  KVC_REQUIRE_PTR(free_list);
  if (!free_top || (reinterpret_cast<uintptr_t>(free_top) & 3u))
    return fail(h, KVC_ERR_ALIGN, "free_top must be a 4-byte aligned device int32");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kvc::PagedArgs a{k_pool,   v_pool,      n_blocks,   block_size, max_blocks, T,
                   seq_len,  pad,         kept_idx,   n_kept,     credit_post, credit_out,
                   table_old, table_new,  free_list,  free_top};
  cudaEvent_t b = mark_begin(h, s);
  cudaError_t e = kvc::launch_compact_paged(h, a, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "paged compaction");
  mark_end(h, kvc::kKernelCompactPaged, b, s);
  return KVC_OK;
}

int kvc_wait_self_test(kvc_handle* h, void* stream) {
  if (!h) return KVC_ERR_ARG;
  cudaError_t e = kvc::launch_wait_self_test(h, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "wait self-test");
  return KVC_OK;
}

int kvc_refresh_decision(kvc_handle* h, const uint16_t* q, float* q_ref, float threshold,
                         int32_t* flag, float* sim, void* stream) {
  if (!h) return KVC_ERR_ARG;
  if (!(threshold >= -1.f && threshold <= 1.f))
    return fail(h, KVC_ERR_ARG, "threshold must lie in [-1, 1]");
  KVC_REQUIRE_PTR(q);
  KVC_REQUIRE_PTR(q_ref);
  KVC_REQUIRE_PTR(flag);
  KVC_REQUIRE_PTR(sim);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t b = mark_begin(h, s);
  cudaError_t e = kvc::launch_refresh(h, q, q_ref, threshold, flag, sim, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "refresh trigger");
  mark_end(h, kvc::kKernelRefresh, b, s);
  return KVC_OK;
}

int kvc_mass_select(kvc_handle* h, const uint16_t* q, const uint16_t* k, int T,
                    const int32_t* pad, const int32_t* n_carry, const float* credit_in,
                    float* credit_post, float* mass, float* score, int32_t* seg_start,
                    int32_t* seg_len, int32_t* quota, int32_t* n_seg, int32_t* kept_idx,
                    int32_t* n_kept, void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  KVC_REQUIRE_PTR(q);
  KVC_REQUIRE_PTR(k);
  KVC_REQUIRE_PTR(pad);
  KVC_REQUIRE_PTR(n_carry);
  KVC_REQUIRE_PTR(credit_in);
  KVC_REQUIRE_PTR(credit_post);
  KVC_REQUIRE_PTR(mass);
  KVC_REQUIRE_PTR(score);
  KVC_REQUIRE_PTR(seg_start);
  KVC_REQUIRE_PTR(seg_len);
  KVC_REQUIRE_PTR(quota);
  KVC_REQUIRE_PTR(n_seg);
  KVC_REQUIRE_PTR(kept_idx);
  KVC_REQUIRE_PTR(n_kept);
  return run_mass_select(h, q, k, T, pad, n_carry, credit_in, credit_post, mass, score,
                         seg_start, seg_len, quota, n_seg, kept_idx, n_kept,
                         static_cast<cudaStream_t>(stream));
}

int kvc_event(kvc_handle* h, const uint16_t* q, const uint16_t* k, const uint16_t* v,
              int T, const int32_t* pad, const int32_t* n_carry, const float* credit_in,
              uint16_t* k_out, uint16_t* v_out, float* credit_out, int32_t* kept_idx,
              int32_t* n_kept, void* stream) {
  if (!h) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  KVC_REQUIRE_PTR(q);
  KVC_REQUIRE_PTR(k);
  KVC_REQUIRE_PTR(v);
  KVC_REQUIRE_PTR(pad);
  KVC_REQUIRE_PTR(n_carry);
  KVC_REQUIRE_PTR(credit_in);
  KVC_REQUIRE_PTR(k_out);
  KVC_REQUIRE_PTR(v_out);
  KVC_REQUIRE_PTR(credit_out);
  KVC_REQUIRE_PTR(kept_idx);
  KVC_REQUIRE_PTR(n_kept);
  return run_event(h, q, k, v, T, pad, n_carry, credit_in, k_out, v_out, credit_out, kept_idx,
                   n_kept, static_cast<cudaStream_t>(stream));
}

int kvc_event_host(kvc_handle* h, const kvc_host_buffers* io, int T, int layers_per_stage,
                   void* stream) {
  if (!h || !io) return KVC_ERR_ARG;
  int rc = check_T(h, T);
  if (rc) return rc;
  if (layers_per_stage < 1) return fail(h, KVC_ERR_ARG, "layers_per_stage must be >= 1");
  if (!io->q_host || !io->k_host || !io->v_host || !io->pad_host || !io->n_carry_host ||
      !io->credit_host || !io->k_out_host || !io->v_out_host || !io->credit_out_host ||
      !io->kept_idx_host || !io->n_kept_host)
    return fail(h, KVC_ERR_ARG, "null host pointer");
  KVC_REQUIRE_PTR(io->q_dev);
  KVC_REQUIRE_PTR(io->k_dev);
  KVC_REQUIRE_PTR(io->v_dev);
  KVC_REQUIRE_PTR(io->pad_dev);
  KVC_REQUIRE_PTR(io->n_carry_dev);
  KVC_REQUIRE_PTR(io->credit_dev);
  KVC_REQUIRE_PTR(io->k_out_dev);
  KVC_REQUIRE_PTR(io->v_out_dev);
  KVC_REQUIRE_PTR(io->credit_out_dev);
  KVC_REQUIRE_PTR(io->kept_idx_dev);
  KVC_REQUIRE_PTR(io->n_kept_dev);
  if (!h->io.in) return fail(h, KVC_ERR_CUDA, "the handle has no copy streams");
  const kvc::Dims full = h->dims;
  const int L = full.L, BH = full.B * full.H, K = h->cfg.budget, d = full.d;
  // Slab offsets are multiples of B*H*4 bytes at least (n_kept): a group of nl
  // layers keeps every slab 16-byte aligned when nl*B*H is a multiple of 4.
  const int m = 4 / gcd_int(BH, 4);
  int nl = ((std::min(layers_per_stage, L) + m - 1) / m) * m;
  while ((L + nl - 1) / nl + 1 > kvc::kMaxHostStages) nl += m;
  if (nl > L) nl = L;
  const size_t q_l = static_cast<size_t>(BH) * full.R * d;  // elements per layer
  const size_t kv_l = static_cast<size_t>(BH) * T * d;
  const size_t c_l = static_cast<size_t>(BH) * T;
  const size_t ko_l = static_cast<size_t>(BH) * K * d;
  const size_t co_l = static_cast<size_t>(BH) * K;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kvc::HostIO& x = h->io;
  auto h2d = [&](void* dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, x.in);
  };
  // device -> host: each slab in two halves, one per output stream
  auto d2h = [&](void* dst, const void* src, size_t bytes) {
    const size_t first = (bytes / 2) & ~size_t(15);
    cudaError_t r = cudaMemcpyAsync(dst, src, first, cudaMemcpyDeviceToHost, x.out[0]);
    if (r == cudaSuccess && bytes > first)
      r = cudaMemcpyAsync(static_cast<char*>(dst) + first, static_cast<const char*>(src) + first,
                          bytes - first, cudaMemcpyDeviceToHost, x.out[1]);
    return r;
  };
  // the copies start after the work already queued on `stream`
  cudaError_t e = cudaEventRecord(x.start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(x.in, x.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(x.out[0], x.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(x.out[1], x.start, 0);
  if (e == cudaSuccess) e = h2d(io->pad_dev, io->pad_host, static_cast<size_t>(full.B) * 4);
  if (e == cudaSuccess)
    e = h2d(io->n_carry_dev, io->n_carry_host, static_cast<size_t>(full.B) * 4);
  if (e != cudaSuccess) return cuda_fail(h, e, "host event: setup");
  // V is read only at the kept rows (by the gather): when the host buffer is
  // mapped into the device's address space, the gather reads it there and V
  // is not copied
  const uint16_t* v_mapped = nullptr;
  {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, io->v_host) == cudaSuccess) {
      if (pa.type == cudaMemoryTypeHost && pa.devicePointer)
        v_mapped = static_cast<const uint16_t*>(pa.devicePointer);
    } else {
      cudaGetLastError();
    }
  }
  int g = 0;
  // Stages of nl layers, except at the end: the host -> device copies are the
  // critical path, and what follows the last of them (that stage's event and
  // its device -> host copies) is shortest when the last stage is small.  So
  // the last stage keeps 1..m layers and the one before it the rest; every
  // stage but the last is a multiple of m layers, so every stage starts aligned.
  auto stage_layers = [&](int l0) {
    const int left = L - l0;
    if (left <= m) return left;
    const int last = (left - 1) % m + 1;
    return left - last <= nl ? left - last : nl;
  };
  for (int l0 = 0, n = 0; l0 < L; l0 += n, ++g) {
    n = stage_layers(l0);
    const size_t lq = l0 * q_l, lkv = l0 * kv_l, lc = l0 * c_l, lko = l0 * ko_l, lco = l0 * co_l;
    e = h2d(io->q_dev + lq, io->q_host + lq, n * q_l * 2);
    if (e == cudaSuccess) e = h2d(io->k_dev + lkv, io->k_host + lkv, n * kv_l * 2);
    if (e == cudaSuccess && !v_mapped)
      e = h2d(io->v_dev + lkv, io->v_host + lkv, n * kv_l * 2);
    if (e == cudaSuccess) e = h2d(io->credit_dev + lc, io->credit_host + lc, n * c_l * 4);
    if (e == cudaSuccess) e = cudaEventRecord(x.landed[g], x.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, x.landed[g], 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "host event: inputs");
    // the event on layers [l0, l0 + n): the same kernels on a handle view of n layers
    h->dims.L = n;
    h->dims.U = n * BH;
    rc = run_event(h, io->q_dev + lq, io->k_dev + lkv,
                   v_mapped ? v_mapped + lkv : io->v_dev + lkv, T, io->pad_dev, io->n_carry_dev, io->credit_dev + lc, io->k_out_dev + lko,
                   io->v_out_dev + lko, io->credit_out_dev + lco, io->kept_idx_dev + lco,
                   io->n_kept_dev + static_cast<size_t>(l0) * BH, s);
    h->dims = full;
    if (rc) return rc;
    e = cudaEventRecord(x.done[g], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(x.out[0], x.done[g], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(x.out[1], x.done[g], 0);
    if (e == cudaSuccess) e = d2h(io->k_out_host + lko, io->k_out_dev + lko, n * ko_l * 2);
    if (e == cudaSuccess) e = d2h(io->v_out_host + lko, io->v_out_dev + lko, n * ko_l * 2);
    if (e == cudaSuccess)
      e = d2h(io->credit_out_host + lco, io->credit_out_dev + lco, n * co_l * 4);
    if (e == cudaSuccess)
      e = d2h(io->kept_idx_host + lco, io->kept_idx_dev + lco, n * co_l * 4);
    if (e == cudaSuccess)
      e = d2h(io->n_kept_host + static_cast<size_t>(l0) * BH,
              io->n_kept_dev + static_cast<size_t>(l0) * BH, static_cast<size_t>(n) * BH * 4);
    if (e != cudaSuccess) return cuda_fail(h, e, "host event: outputs");
  }
  // `stream` completes only after the last host copy
  for (int j = 0; j < 2 && e == cudaSuccess; ++j) {
    e = cudaEventRecord(x.end[j], x.out[j]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, x.end[j], 0);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "host event: end");
  return KVC_OK;
}

int kvc_profile(kvc_handle* h, int enable) {
  if (!h) return KVC_ERR_ARG;
  auto& P = h->prof;
  if (enable) {
    for (auto& m : P.pending) {
      cudaEventSynchronize(m.end);
      P.pool.push_back(m.begin);
      P.pool.push_back(m.end);
    }
    P.pending.clear();
    for (int i = 0; i < kvc::kNumKernels; ++i) {
      P.launches[i] = 0;
      P.total_ms[i] = 0.0;
    }
  }
  P.enabled = enable != 0;
  return KVC_OK;
}

int kvc_profile_read(kvc_handle* h, kvc_kernel_time* out, int capacity, int* n_out,
                     int reset) {
  if (!h || (!out && capacity > 0) || !n_out) return KVC_ERR_ARG;
  auto& P = h->prof;
  for (auto& m : P.pending) {
    cudaError_t e = cudaEventSynchronize(m.end);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, m.begin, m.end);
    if (e != cudaSuccess) return cuda_fail(h, e, "profile read");
    P.launches[m.kernel] += 1;
    P.total_ms[m.kernel] += ms;
    P.pool.push_back(m.begin);
    P.pool.push_back(m.end);
  }
  P.pending.clear();
  int n = 0;
  for (int i = 0; i < kvc::kNumKernels; ++i) {
    if (n < capacity) {
      out[n].name = kKernelNames[i];
      out[n].launches = P.launches[i];
      out[n].total_ms = P.total_ms[i];
    }
    ++n;
  }
  *n_out = n < capacity ? n : capacity;
  if (reset) {
    for (int i = 0; i < kvc::kNumKernels; ++i) {
      P.launches[i] = 0;
      P.total_ms[i] = 0.0;
    }
  }
  return KVC_OK;
}

int kvc_get_device_status(kvc_handle* h, uint32_t* bits, void* stream) {
  if (!h || !bits) return KVC_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "status sync");
  uint32_t v = 0;
  e = cudaMemcpy(&v, h->ws.status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "status read");
  e = cudaMemset(h->ws.status, 0, sizeof v);
  if (e != cudaSuccess) return cuda_fail(h, e, "status clear");
  *bits = v;
  return v ? KVC_ERR_TIMEOUT : KVC_OK;
}

}  // extern "C"
