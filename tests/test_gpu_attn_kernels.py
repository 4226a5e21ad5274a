"""Step 1 on both tensor-core kernels (kvc_config.attn_kernel): one SM per MMA
(1) and CTA pairs sharing an M256 MMA (2), each against the oracle, on shapes
that reach every edge of the pair kernel's item walk: a single 32-row window
(one pair whose second tile is absent), query-row counts that are not a
multiple of 256 (an odd number of 128-row tiles), caches that are not a
multiple of 128 slots, left padding that leaves whole tiles empty, an
all-padding sequence, both head sizes, and more units than CTA pairs.
Mass, score and credit within 1e-4 relative (+1e-9); the two kernels differ
only in fp32 summation order, so they agree to 1e-5 relative."""
import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


SHAPES = {
    "tiny": (wl.CONFIGS["tiny"], None),
    "odd_tiles": (wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=2, group=3, window=96,
                            T=1000, budget=300), None),
    "ragged_d64": (wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=1, batch=5, n_kv_heads=2,
                             group=4, head_dim=64, prefill=(10, 400), generated=300,
                             budget=300), [0, 37, 250, 620, 700]),
    "many_units": (wl.scaled(wl.CONFIGS["qwen_1l"], n_layers=2, batch=40, n_kv_heads=4, T=600,
                             budget=200), None),
}


def _inputs(name):
    w, pads = SHAPES[name]
    inp = wl.generate(w)
    if pads is not None:
        T = inp.T
        pad = torch.tensor([min(p, T) for p in pads], dtype=torch.int32)
        slot = torch.arange(T).view(1, 1, 1, T, 1)
        valid = slot >= pad.view(1, -1, 1, 1, 1)
        inp.k = torch.where(valid, inp.k, torch.zeros((), dtype=inp.k.dtype))
        inp.v = torch.where(valid, inp.v, torch.zeros((), dtype=inp.v.dtype))
        inp.pad = pad
        inp.n_carry = (T - pad).to(torch.int32)
    return w, inp


@pytest.fixture(scope="module")
def oracle_mass(ref):
    out = {}
    for name in SHAPES:
        w, inp = _inputs(name)
        p = gu.ref_params(ref, w)
        q, k, _, c, pad, nc = gu.oracle_inputs(inp)
        out[name] = (w, inp, ref.mass(p, q, k, c, pad, nc, threads=8))
    return out


@pytest.mark.parametrize("name", list(SHAPES))
def test_both_kernels_against_oracle(oracle_mass, name):
    import eviction_gb300 as kvc
    w, inp, (m_r, s_r, c_r) = oracle_mass[name]
    got = {}
    for kern in (1, 2):
        h = kvc.Handle(gu.config_for(w, inp.T, attn_kernel=kern))
        m, s, c = gu.gpu_mass(h, gu.to_device(inp), inp.T)
        assert h.device_status() == 0, f"attn_kernel {kern}: device status"
        for label, g, r in (("mass", m, m_r), ("score", s, s_r), ("credit", c, c_r)):
            ok, rel = gu.mass_close(g, r)
            assert ok, f"attn_kernel {kern} {label}: rel {rel:.3g}"
        got[kern] = (m, s, c)
        h.close()
    for a, b in zip(got[1], got[2]):
        ok, rel = gu.mass_close(a, b, rtol=1e-5, atol=1e-12)
        assert ok, f"kernels differ: rel {rel:.3g}"


def test_pair_kernel_repeatable():
    """Same inputs, same bits, twice in a row on the pair kernel."""
    import eviction_gb300 as kvc
    w, inp = _inputs("odd_tiles")
    h = kvc.Handle(gu.config_for(w, inp.T, attn_kernel=2))
    g = gu.to_device(inp)
    first = gu.gpu_mass(h, g, inp.T)
    second = gu.gpu_mass(h, g, inp.T)
    for a, b in zip(first, second):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
