"""The event at the library's maximum sizes, against the oracle unit by unit:
T = max_T = 65536 slots (one unit left-padded), and the largest query window
G*W = 4096 rows.  Same per-unit checks as the full-size tests (mass and score
within 1e-4, kept sets equal up to near-ties or a cut moved at a threshold,
exact compaction)."""
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402
from tests.test_gpu_fullsize import _check, _run, _unit_inputs  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _with_pads(inp, pads):
    """Left-pad sequence b by pads[b] slots (zero keys and values there; every
    valid slot carries credit, as on a first event)."""
    T = inp.T
    pad = torch.tensor([min(p, T) for p in pads], dtype=torch.int32, device=inp.k.device)
    slot = torch.arange(T, device=inp.k.device).view(1, 1, 1, T, 1)
    valid = slot >= pad.view(1, -1, 1, 1, 1)
    inp.k = torch.where(valid, inp.k, torch.zeros((), dtype=inp.k.dtype, device=inp.k.device))
    inp.v = torch.where(valid, inp.v, torch.zeros((), dtype=inp.v.dtype, device=inp.v.device))
    inp.pad = pad
    inp.n_carry = (T - pad).to(torch.int32)
    return inp


def test_max_T(ref):
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["long"], n_layers=1, batch=2, n_kv_heads=1, group=1, T=65536,
                  budget=4096, n_recent=256, regions=(300, 300))
    inp = _with_pads(wl.generate(w, device="cuda"), [0, 12345])
    p = gu.ref_params(ref, w)
    h = kvc.Handle(gu.config_for(w, inp.T))
    out, st = _run(h, inp)
    units = [0, 1]
    r = ref.event(p, *_unit_inputs(inp, units))
    _check(ref, p, w, inp, out, st, units, r)


def test_max_query_rows(ref):
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["qwen_1l"], batch=1, n_kv_heads=1, group=32, window=128, T=4096,
                  budget=1024)
    assert w.group * w.window == 4096
    inp = wl.generate(w, device="cuda")
    p = gu.ref_params(ref, w)
    h = kvc.Handle(gu.config_for(w, inp.T))
    out, st = _run(h, inp)
    r = ref.event(p, *_unit_inputs(inp, [0]))
    _check(ref, p, w, inp, out, st, [0], r)


def test_more_units_than_grid_y(ref):
    """More than 65535 units (the CUDA limit on a grid's y extent, which the
    gather's unit axis uses): the gather launches in chunks of units, so units
    past 65535 are compacted too.  Every unit's compaction is checked against a
    torch gather of its own kept slots; units on both sides of the limit go
    through the end-to-end checker against the oracle."""
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["qwen_1l"], n_layers=1, batch=16500, n_kv_heads=4, group=1,
                  head_dim=64, T=48, window=4, budget=24, n_recent=8, regions=(1, 1),
                  region_len=("uniform", 4, 8))
    assert w.units > 65535
    inp = wl.generate(w, device="cuda")
    p = gu.ref_params(ref, w)
    h = kvc.Handle(gu.config_for(w, inp.T))
    out, st = _run(h, inp)
    U, T, d = w.units, inp.T, w.head_dim
    kept = out["kept_idx"].reshape(U, -1).long()
    assert bool((out["n_kept"] == w.budget).all())
    for name in ("k", "v"):
        src = getattr(inp, name).reshape(U, T, d)
        ref_rows = torch.gather(src, 1, kept[:, :, None].expand(-1, -1, d))
        assert torch.equal(out[f"{name}_out"].reshape(U, -1, d).view(torch.int16),
                           ref_rows.view(torch.int16)), name
    units = [0, 65534, 65535, 65536, U - 1]
    r = ref.event(p, *_unit_inputs(inp, units))
    _check(ref, p, w, inp, out, st, units, r)
