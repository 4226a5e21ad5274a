"""ctypes binding of libkvc.so (argument marshalling only).

Every method maps one-to-one onto an entry point of ``include/kvc.h`` and takes
torch tensors that must already live on the CUDA device with the documented
dtype and layout; the binding checks dtype/device/contiguity, then passes
``data_ptr()`` values and ``torch.cuda.current_stream()``. All arithmetic runs in
the library's kernels.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, fields

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libkvc.so")

# every function declared in include/kvc.h
ENTRY_POINTS = ("kvc_default_config", "kvc_create", "kvc_destroy", "kvc_stage_sizes",
                "kvc_mass", "kvc_segment_quota", "kvc_select", "kvc_compact", "kvc_event",
                "kvc_get_device_status", "kvc_last_error", "kvc_status_string", "kvc_profile",
                "kvc_profile_read", "kvc_mass_noalloc", "kvc_refresh_decision",
                "kvc_compact_paged", "kvc_redundancy_score", "kvc_wait_self_test",
                "kvc_event_host", "kvc_mass_select")

STATUS = {0: "KVC_OK", -1: "KVC_ERR_ARG", -2: "KVC_ERR_SHAPE", -3: "KVC_ERR_ALIGN",
          -4: "KVC_ERR_NOMEM", -5: "KVC_ERR_CUDA", -6: "KVC_ERR_DEVICE", -7: "KVC_ERR_TIMEOUT",
          -8: "KVC_ERR_UNSUPPORTED"}


class KvcError(RuntimeError):
    def __init__(self, code, msg=""):
        self.code = code
        super().__init__(f"{STATUS.get(code, code)}: {msg}")


class _KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


class _CConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("batch", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("group", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_T", ctypes.c_int), ("window", ctypes.c_int),
                ("budget", ctypes.c_int), ("avg_pool", ctypes.c_int), ("max_pool", ctypes.c_int),
                ("delta", ctypes.c_float), ("seg_min", ctypes.c_int), ("seg_max", ctypes.c_int),
                ("q_min", ctypes.c_int), ("n_sink", ctypes.c_int), ("n_recent", ctypes.c_int),
                ("lambda_", ctypes.c_float), ("beta", ctypes.c_float), ("eps", ctypes.c_float),
                ("softmax_scale", ctypes.c_float), ("seg_fixed", ctypes.c_int),
                ("quota_by_len", ctypes.c_int), ("global_topk", ctypes.c_int),
                ("redundancy_sigma", ctypes.c_float), ("attn_kernel", ctypes.c_int)]


# The ablations of the method's ablation table as Config keyword switches
# ("none" = the method; "no_credit" sets beta = 1, which turns the credit mix off).
ABLATIONS = {
    "none": {},
    "fixed_segments": {"seg_fixed": 64},
    "no_mass_quota": {"quota_by_len": 1},
    "no_credit": {"beta": 1.0},
    "global_topk": {"global_topk": 1},
}


@dataclass
class Config:
    """Mirror of kvc_config (defaults: the method's schedule values)."""
    n_layers: int
    batch: int
    n_kv_heads: int
    group: int
    head_dim: int
    max_T: int
    budget: int
    window: int = 128
    avg_pool: int = 5
    max_pool: int = 7
    delta: float = 0.1
    seg_min: int = 16
    seg_max: int = 256
    q_min: int = 1
    n_sink: int = 4
    n_recent: int = 64
    lam: float = 0.9
    beta: float = 0.9
    eps: float = 1e-6
    softmax_scale: float = 0.0
    seg_fixed: int = 0       # ablation: fixed-length segments (0 = mass cut points)
    quota_by_len: int = 0    # ablation: quotas by segment length instead of mass
    global_topk: int = 0     # ablation: one segment, per-head global top-k
    redundancy_sigma: float = 0.0  # > 0: select on sigma*I - (1-sigma)*R (key redundancy)
    attn_kernel: int = 0     # step-1 tensor-core kernel: 1 one SM per MMA, 2 CTA pairs, 0 auto (1)

    def c(self) -> _CConfig:
        return _CConfig(self.n_layers, self.batch, self.n_kv_heads, self.group, self.head_dim,
                        self.max_T, self.window, self.budget, self.avg_pool, self.max_pool,
                        self.delta, self.seg_min, self.seg_max, self.q_min, self.n_sink,
                        self.n_recent, self.lam, self.beta, self.eps, self.softmax_scale,
                        self.seg_fixed, self.quota_by_len, self.global_topk,
                        self.redundancy_sigma, self.attn_kernel)

    @property
    def units(self):
        return self.n_layers * self.batch * self.n_kv_heads


_HOST_BUFFER_FIELDS = ("q", "k", "v", "pad", "n_carry", "credit")
_HOST_OUT_FIELDS = ("k_out", "v_out", "credit_out", "kept_idx", "n_kept")


class _HostBuffers(ctypes.Structure):
    """kvc_host_buffers: (host, device) pointer pairs, inputs then outputs
    (outputs are listed device first, as in the C struct)."""
    _fields_ = ([(f"{k}_{side}", ctypes.c_void_p) for k in _HOST_BUFFER_FIELDS
                 for side in ("host", "dev")] +
                [(f"{k}_{side}", ctypes.c_void_p) for k in _HOST_OUT_FIELDS
                 for side in ("dev", "host")])


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libkvc.so; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with eviction_gb300.build.build()")
    L = ctypes.CDLL(_LIB_PATH)
    L.kvc_default_config.argtypes = [ctypes.POINTER(_CConfig)]
    L.kvc_default_config.restype = None
    L.kvc_create.argtypes = [ctypes.POINTER(_CConfig), ctypes.POINTER(_P)]
    L.kvc_destroy.argtypes = [_P]
    L.kvc_destroy.restype = None
    L.kvc_stage_sizes.argtypes = [_P, _I, ctypes.POINTER(_I)]
    L.kvc_mass.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P]
    L.kvc_segment_quota.argtypes = [_P, _P, _I, _P, _P, _P, _P, _P, _P]
    L.kvc_select.argtypes = [_P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P]
    L.kvc_compact.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P]
    L.kvc_event.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    L.kvc_mass_select.argtypes = [_P, _P, _P, _I] + [_P] * 13
    L.kvc_get_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32), _P]
    L.kvc_last_error.argtypes = [_P]
    L.kvc_last_error.restype = ctypes.c_char_p
    L.kvc_profile.argtypes = [_P, _I]
    L.kvc_profile_read.argtypes = [_P, ctypes.POINTER(_KernelTime), _I, ctypes.POINTER(_I), _I]
    L.kvc_mass_noalloc.argtypes = [ctypes.POINTER(_CConfig), _P, _P, _I, _P, _P, _P, _P, _P, _P,
                                   _P, _P]
    L.kvc_refresh_decision.argtypes = [_P, _P, _P, ctypes.c_float, _P, _P, _P]
    L.kvc_compact_paged.argtypes = [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P,
                                    _P, _P, _P]
    L.kvc_redundancy_score.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P]
    L.kvc_wait_self_test.argtypes = [_P, _P]
    L.kvc_event_host.argtypes = [_P, ctypes.POINTER(_HostBuffers), _I, _I, _P]
    L.kvc_status_string.argtypes = [_I]
    L.kvc_status_string.restype = ctypes.c_char_p
    for name in ENTRY_POINTS:
        if name not in ("kvc_default_config", "kvc_destroy", "kvc_last_error",
                        "kvc_status_string"):
            getattr(L, name).restype = _I
    _lib = L
    return L


def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def mass_noalloc(cfg: Config, q, k, T, pad, n_carry, credit_in, credit_post, mass, score,
                 status=None, stream=None) -> int:
    """kvc_mass_noalloc: steps 1-2 without a handle and without any device
    allocation (for callers that cannot allocate; see include/kvc.h).
    Returns the library's status code (0 = KVC_OK)."""
    import torch
    c = cfg.c()
    st = _dev(status, torch.int32, "status") if status is not None else ctypes.c_void_p(0)
    return load_library().kvc_mass_noalloc(
        ctypes.byref(c), _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), T,
        _dev(pad, torch.int32, "pad"), _dev(n_carry, torch.int32, "n_carry"),
        _dev(credit_in, torch.float32, "credit_in"), _dev(credit_post, torch.float32, "credit_post"),
        _dev(mass, torch.float32, "mass"), _dev(score, torch.float32, "score"), st,
        _stream_ptr(stream))


class Handle:
    """A kvc_handle: validated config plus the device workspace."""

    def __init__(self, cfg: Config):
        L = load_library()
        self.cfg = cfg
        self._c = cfg.c()
        h = _P()
        rc = L.kvc_create(ctypes.byref(self._c), ctypes.byref(h))
        if rc != 0:
            raise KvcError(rc, "kvc_create failed")
        self._h = h

    # -- helpers -------------------------------------------------------------
    def _check(self, rc, what):
        if rc != 0:
            msg = load_library().kvc_last_error(self._h)
            raise KvcError(rc, f"{what}: {msg.decode() if msg else ''}")

    def close(self):
        if getattr(self, "_h", None):
            load_library().kvc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def s_max(self, T: int) -> int:
        out = _I()
        self._check(load_library().kvc_stage_sizes(self._h, T, ctypes.byref(out)), "stage_sizes")
        return out.value

    # -- entry points --------------------------------------------------------
    def mass(self, q, k, T, pad, n_carry, credit_in, credit_post, mass, score, stream=None):
        import torch
        rc = load_library().kvc_mass(
            self._h, _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), T,
            _dev(pad, torch.int32, "pad"), _dev(n_carry, torch.int32, "n_carry"),
            _dev(credit_in, torch.float32, "credit_in"),
            _dev(credit_post, torch.float32, "credit_post"), _dev(mass, torch.float32, "mass"),
            _dev(score, torch.float32, "score"), _stream_ptr(stream))
        self._check(rc, "kvc_mass")

    def segment_quota(self, mass, T, pad, seg_start, seg_len, quota, n_seg, stream=None):
        import torch
        rc = load_library().kvc_segment_quota(
            self._h, _dev(mass, torch.float32, "mass"), T, _dev(pad, torch.int32, "pad"),
            _dev(seg_start, torch.int32, "seg_start"), _dev(seg_len, torch.int32, "seg_len"),
            _dev(quota, torch.int32, "quota"), _dev(n_seg, torch.int32, "n_seg"),
            _stream_ptr(stream))
        self._check(rc, "kvc_segment_quota")

    def select(self, score, T, pad, seg_start, seg_len, quota, n_seg, kept_idx, n_kept,
               stream=None):
        import torch
        rc = load_library().kvc_select(
            self._h, _dev(score, torch.float32, "score"), T, _dev(pad, torch.int32, "pad"),
            _dev(seg_start, torch.int32, "seg_start"), _dev(seg_len, torch.int32, "seg_len"),
            _dev(quota, torch.int32, "quota"), _dev(n_seg, torch.int32, "n_seg"),
            _dev(kept_idx, torch.int32, "kept_idx"), _dev(n_kept, torch.int32, "n_kept"),
            _stream_ptr(stream))
        self._check(rc, "kvc_select")

    def compact(self, k, v, credit_post, T, kept_idx, n_kept, k_out, v_out, credit_out,
                stream=None):
        import torch
        rc = load_library().kvc_compact(
            self._h, _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
            _dev(credit_post, torch.float32, "credit_post"), T,
            _dev(kept_idx, torch.int32, "kept_idx"), _dev(n_kept, torch.int32, "n_kept"),
            _dev(k_out, torch.bfloat16, "k_out"), _dev(v_out, torch.bfloat16, "v_out"),
            _dev(credit_out, torch.float32, "credit_out"), _stream_ptr(stream))
        self._check(rc, "kvc_compact")

    def mass_select(self, q, k, T, pad, n_carry, credit_in, credit_post, mass, score,
                    seg_start, seg_len, quota, n_seg, kept_idx, n_kept, stream=None):
        """kvc_mass_select: steps 1-5 (kvc_mass, kvc_segment_quota, kvc_select
        chained) with every intermediate in the given buffers."""
        import torch
        rc = load_library().kvc_mass_select(
            self._h, _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"), T,
            _dev(pad, torch.int32, "pad"), _dev(n_carry, torch.int32, "n_carry"),
            _dev(credit_in, torch.float32, "credit_in"),
            _dev(credit_post, torch.float32, "credit_post"), _dev(mass, torch.float32, "mass"),
            _dev(score, torch.float32, "score"), _dev(seg_start, torch.int32, "seg_start"),
            _dev(seg_len, torch.int32, "seg_len"), _dev(quota, torch.int32, "quota"),
            _dev(n_seg, torch.int32, "n_seg"), _dev(kept_idx, torch.int32, "kept_idx"),
            _dev(n_kept, torch.int32, "n_kept"), _stream_ptr(stream))
        self._check(rc, "kvc_mass_select")

    def event(self, q, k, v, T, pad, n_carry, credit_in, k_out, v_out, credit_out, kept_idx,
              n_kept, stream=None):
        import torch
        rc = load_library().kvc_event(
            self._h, _dev(q, torch.bfloat16, "q"), _dev(k, torch.bfloat16, "k"),
            _dev(v, torch.bfloat16, "v"), T, _dev(pad, torch.int32, "pad"),
            _dev(n_carry, torch.int32, "n_carry"), _dev(credit_in, torch.float32, "credit_in"),
            _dev(k_out, torch.bfloat16, "k_out"), _dev(v_out, torch.bfloat16, "v_out"),
            _dev(credit_out, torch.float32, "credit_out"),
            _dev(kept_idx, torch.int32, "kept_idx"), _dev(n_kept, torch.int32, "n_kept"),
            _stream_ptr(stream))
        self._check(rc, "kvc_event")

    def redundancy_score(self, k, score, T, pad, sel_score, redundancy=None, stream=None):
        """kvc_redundancy_score: k [L,B,H,T,d] bf16, score [L,B,H,T] fp32 ->
        sel_score [L,B,H,T] fp32 (may be score itself), redundancy (optional)
        [L,B,H,T] fp32.  Needs cfg.redundancy_sigma > 0."""
        import torch
        red = _dev(redundancy, torch.float32, "redundancy") if redundancy is not None \
            else ctypes.c_void_p(0)
        rc = load_library().kvc_redundancy_score(
            self._h, _dev(k, torch.bfloat16, "k"), _dev(score, torch.float32, "score"), T,
            _dev(pad, torch.int32, "pad"), _dev(sel_score, torch.float32, "sel_score"), red,
            _stream_ptr(stream))
        self._check(rc, "kvc_redundancy_score")

    def refresh_decision(self, q, q_ref, threshold, flag, sim, stream=None):
        """kvc_refresh_decision: q [L,B,H*G,d] bf16 (the current token), q_ref
        [L,B,d] fp32 in/out, flag [L,B] int32 out, sim [L,B] fp32 out."""
        import torch
        rc = load_library().kvc_refresh_decision(
            self._h, _dev(q, torch.bfloat16, "q"), _dev(q_ref, torch.float32, "q_ref"),
            ctypes.c_float(threshold), _dev(flag, torch.int32, "flag"),
            _dev(sim, torch.float32, "sim"), _stream_ptr(stream))
        self._check(rc, "kvc_refresh_decision")

    def compact_paged(self, k_pool, v_pool, block_size, seq_len, pad, kept_idx, n_kept,
                      credit_post, T, credit_out, table_old, table_new, free_list, free_top,
                      stream=None):
        """kvc_compact_paged: pools [L, n_blocks, H, bs, d] bf16 (in/out), tables
        [B, max_blocks] int32, free_list [n_blocks] int32 and free_top [1] int32
        (in/out), credit_post [L,B,H,T] -> credit_out [L,B,H,budget]."""
        import torch
        n_blocks = k_pool.shape[1]
        max_blocks = table_old.shape[1]
        rc = load_library().kvc_compact_paged(
            self._h, _dev(k_pool, torch.bfloat16, "k_pool"), _dev(v_pool, torch.bfloat16, "v_pool"),
            n_blocks, block_size, max_blocks, _dev(seq_len, torch.int32, "seq_len"),
            _dev(pad, torch.int32, "pad"), _dev(kept_idx, torch.int32, "kept_idx"),
            _dev(n_kept, torch.int32, "n_kept"), _dev(credit_post, torch.float32, "credit_post"), T,
            _dev(credit_out, torch.float32, "credit_out"),
            _dev(table_old, torch.int32, "table_old"), _dev(table_new, torch.int32, "table_new"),
            _dev(free_list, torch.int32, "free_list"), _dev(free_top, torch.int32, "free_top"),
            _stream_ptr(stream))
        self._check(rc, "kvc_compact_paged")

    def wait_self_test(self, stream=None):
        """kvc_wait_self_test: a bounded wait that runs out on purpose (about
        2 s); afterwards device_status() reports KVC_STATUS_WAIT_TIMEOUT."""
        self._check(load_library().kvc_wait_self_test(self._h, _stream_ptr(stream)),
                    "kvc_wait_self_test")

    def device_status(self, stream=None) -> int:
        bits = ctypes.c_uint32(0)
        rc = load_library().kvc_get_device_status(self._h, ctypes.byref(bits), _stream_ptr(stream))
        if rc not in (0, -7):
            self._check(rc, "kvc_get_device_status")
        return bits.value

    # -- tracing ---------------------------------------------------------------
    def profile(self, enable: bool = True):
        """Start (clearing totals) or stop per-kernel CUDA-event tracing."""
        self._check(load_library().kvc_profile(self._h, 1 if enable else 0), "kvc_profile")

    def profile_read(self, reset: bool = False):
        """[{name, launches, total_ms}] per kernel (waits for the recorded events)."""
        arr = (_KernelTime * 16)()
        n = _I()
        self._check(load_library().kvc_profile_read(self._h, arr, 16, ctypes.byref(n),
                                                    1 if reset else 0), "kvc_profile_read")
        return [dict(name=arr[i].name.decode(), launches=arr[i].launches,
                     total_ms=arr[i].total_ms) for i in range(n.value)]

    # -- end to end from host buffers ------------------------------------------
    def event_host(self, host_in: dict, dev_in: dict, host_out: dict, dev_out: dict, T: int,
                   stream=None):
        """One event from pinned host inputs to pinned host outputs.

        Copies q, k, v, credit, pad, n_carry host -> device into `dev_in`, runs
        kvc_event into `dev_out`, copies every output back into `host_out`, all
        on one stream (asynchronous; the caller synchronises). Returns the bytes
        moved each way.
        """
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        h2d = d2h = 0
        with torch.cuda.stream(s):
            for key in ("q", "k", "v", "credit", "pad", "n_carry"):
                dev_in[key].copy_(host_in[key], non_blocking=True)
                h2d += host_in[key].numel() * host_in[key].element_size()
            self.event(dev_in["q"], dev_in["k"], dev_in["v"], T, dev_in["pad"],
                       dev_in["n_carry"], dev_in["credit"], dev_out["k_out"], dev_out["v_out"],
                       dev_out["credit_out"], dev_out["kept_idx"], dev_out["n_kept"], stream=s)
            for key in ("k_out", "v_out", "credit_out", "kept_idx", "n_kept"):
                host_out[key].copy_(dev_out[key], non_blocking=True)
                d2h += dev_out[key].numel() * dev_out[key].element_size()
        return h2d, d2h

    def event_from_host(self, host_in: dict, dev_in: dict, host_out: dict, dev_out: dict,
                        T: int, layers_per_stage: int = 2, stream=None):
        """kvc_event_host: the event from pinned host buffers, pipelined over
        groups of layers (host -> device copies of the next group and device ->
        host copies of the previous one overlap the current group's event).
        host_in / dev_in: q, k, v, pad, n_carry, credit; host_out / dev_out:
        k_out, v_out, credit_out, kept_idx, n_kept.  Returns the bytes copied
        each way; a page-locked V is read in place at the kept rows only (not
        counted here: n_kept * d * 2 bytes per unit).  The work is complete
        once `stream` is."""
        import torch
        hb = _HostBuffers()
        dtypes = dict(q=torch.bfloat16, k=torch.bfloat16, v=torch.bfloat16, pad=torch.int32,
                      n_carry=torch.int32, credit=torch.float32, k_out=torch.bfloat16,
                      v_out=torch.bfloat16, credit_out=torch.float32, kept_idx=torch.int32,
                      n_kept=torch.int32)
        h2d = d2h = 0
        for key in _HOST_BUFFER_FIELDS + _HOST_OUT_FIELDS:
            hs = host_in[key] if key in host_in else host_out[key]
            ds = dev_in[key] if key in dev_in else dev_out[key]
            if hs.is_cuda or hs.dtype != dtypes[key] or not hs.is_contiguous():
                raise ValueError(f"{key}: host tensor must be a contiguous CPU {dtypes[key]}")
            if hs.numel() != ds.numel():
                raise ValueError(f"{key}: host and device sizes differ")
            setattr(hb, f"{key}_host", hs.data_ptr())
            setattr(hb, f"{key}_dev", _dev(ds, dtypes[key], key).value)
            nbytes = hs.numel() * hs.element_size()
            if key == "v" and hs.is_pinned():
                continue  # read in place at the kept rows by the gather
            if key in _HOST_BUFFER_FIELDS:
                h2d += nbytes
            else:
                d2h += nbytes
        rc = load_library().kvc_event_host(self._h, ctypes.byref(hb), T, int(layers_per_stage),
                                           _stream_ptr(stream))
        self._check(rc, "kvc_event_host")
        return h2d, d2h

    # -- allocation conveniences (torch allocates; the library never does) ---
    def outputs(self, T, device="cuda"):
        """Output tensors of one event: k_out, v_out, credit_out, kept_idx, n_kept."""
        import torch
        c = self.cfg
        L, B, H, d, Kb = c.n_layers, c.batch, c.n_kv_heads, c.head_dim, c.budget
        return dict(
            k_out=torch.empty((L, B, H, Kb, d), dtype=torch.bfloat16, device=device),
            v_out=torch.empty((L, B, H, Kb, d), dtype=torch.bfloat16, device=device),
            credit_out=torch.empty((L, B, H, Kb), dtype=torch.float32, device=device),
            kept_idx=torch.empty((L, B, H, Kb), dtype=torch.int32, device=device),
            n_kept=torch.empty((L, B, H), dtype=torch.int32, device=device))

    def stage_buffers(self, T, device="cuda"):
        """Intermediate tensors for the stage-by-stage entry points."""
        import torch
        c = self.cfg
        L, B, H = c.n_layers, c.batch, c.n_kv_heads
        S = self.s_max(T)
        f = dict(dtype=torch.float32, device=device)
        i = dict(dtype=torch.int32, device=device)
        return dict(mass=torch.empty((L, B, H, T), **f), score=torch.empty((L, B, H, T), **f),
                    credit_post=torch.empty((L, B, H, T), **f),
                    seg_start=torch.empty((L, B, H, S), **i),
                    seg_len=torch.empty((L, B, H, S), **i),
                    quota=torch.empty((L, B, H, S), **i), n_seg=torch.empty((L, B, H), **i))
