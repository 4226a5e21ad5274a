"""The C ABI without a GPU: the library loads, exports every entry point that
include/kvc.h declares, validates configurations on the host, and reports a
missing device instead of crashing. No kernel is launched here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    from eviction_gb300 import build
    build.build()
    import eviction_gb300
    return eviction_gb300.load_library()


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", text)))


def test_header_lists_all_entry_points():
    import eviction_gb300
    assert set(_declared("kvc.h")) == set(eviction_gb300.ENTRY_POINTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared("kvc.h"):
        assert hasattr(lib, name), name


def test_status_strings(lib):
    import eviction_gb300.kvc as k
    for code, name in k.STATUS.items():
        assert lib.kvc_status_string(code).decode() == name


def test_default_config(lib):
    import eviction_gb300.kvc as k
    c = k._CConfig()
    lib.kvc_default_config(ctypes.byref(c))
    assert (c.window, c.avg_pool, c.max_pool, c.seg_min, c.seg_max, c.q_min, c.n_sink) == \
        (128, 5, 7, 16, 256, 1, 4)
    assert abs(c.delta - 0.1) < 1e-7 and abs(c.lambda_ - 0.9) < 1e-7 and abs(c.beta - 0.9) < 1e-7


def _create(lib, **over):
    import eviction_gb300.kvc as k
    cfg = k.Config(n_layers=1, batch=1, n_kv_heads=1, group=1, head_dim=64, max_T=768,
                   budget=256)
    for key, val in over.items():
        setattr(cfg, key, val)
    c = cfg.c()
    h = ctypes.c_void_p()
    return lib.kvc_create(ctypes.byref(c), ctypes.byref(h))


@pytest.mark.parametrize("over,code", [
    (dict(avg_pool=4), -1), (dict(max_pool=0), -1), (dict(delta=0.0), -1),
    (dict(delta=1e-4), -1), (dict(seg_min=16, seg_max=20), -1), (dict(lam=1.5), -1),
    (dict(eps=0.0), -1), (dict(budget=0), -1), (dict(max_T=70000), -1),
    (dict(head_dim=96), -8), (dict(group=64, window=128), -8)])
def test_create_rejects_bad_config(lib, over, code):
    assert _create(lib, **over) == code


def test_create_without_gpu_reports_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _create(lib) == -6


def test_null_arguments(lib):
    assert lib.kvc_create(None, None) == -1
    out = ctypes.c_int()
    assert lib.kvc_stage_sizes(None, 10, ctypes.byref(out)) == -1
    assert lib.kvc_mass(None, *([None] * 2), 10, *([None] * 6), None) == -1
