"""The whole event on seeded random small shapes, unit by unit against the
oracle: head_dim 64 / 128, T not a multiple of 32, windows from 1 to 128,
odd GQA groups, budgets above T, sequences that are all padding or nearly so,
no sinks or no recent suffix.  Same per-unit bar as the full-size tests (mass
and score within 1e-4 relative, kept sets equal up to near-ties or a cut that
moved at a threshold, exact compaction)."""
import numpy as np
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


def _shape(seed):
    rng = np.random.default_rng(1000 + seed)
    d = int(rng.choice([64, 128]))
    T = int(rng.integers(17, 3000))
    W = int(min(T, rng.choice([1, 7, 32, 64, 100, 128])))
    G = int(rng.choice([1, 3, 4, 7]))
    B = int(rng.integers(1, 4))
    H = int(rng.integers(1, 3))
    budget = int(rng.integers(1, T + 50))
    n_recent = int(rng.integers(0, 65))
    n_sink = int(rng.integers(0, 5))
    pads = [int(x) for x in rng.integers(0, T + 1, B)]
    if B > 1:
        pads[0] = 0
    if seed % 4 == 1:
        pads[-1] = T        # a sequence that is all padding
    if seed % 4 == 2:
        pads[-1] = T - 1    # one valid slot
    return dict(d=d, T=T, W=W, G=G, B=B, H=H, budget=budget, n_recent=n_recent, n_sink=n_sink,
                pads=pads)


def _with_pads(inp, pads):
    T = inp.T
    pad = torch.tensor([min(p, T) for p in pads], dtype=torch.int32, device=inp.k.device)
    slot = torch.arange(T, device=inp.k.device).view(1, 1, 1, T, 1)
    valid = slot >= pad.view(1, -1, 1, 1, 1)
    zero = torch.zeros((), dtype=inp.k.dtype, device=inp.k.device)
    inp.k = torch.where(valid, inp.k, zero)
    inp.v = torch.where(valid, inp.v, zero)
    inp.pad = pad
    inp.n_carry = (T - pad).to(torch.int32)
    return inp


@pytest.mark.parametrize("seed", range(24))
def test_random_shape(ref, seed):
    import eviction_gb300 as kvc
    s = _shape(seed)
    w = wl.scaled(wl.CONFIGS["qwen_1l"], n_layers=1, batch=s["B"], n_kv_heads=s["H"],
                  group=s["G"], head_dim=s["d"], T=s["T"], window=s["W"], budget=s["budget"],
                  n_recent=s["n_recent"], n_sink=s["n_sink"], regions=(2, 6), seed=seed)
    inp = _with_pads(wl.generate(w, device="cuda"), s["pads"])
    p = gu.ref_params(ref, w)
    h = kvc.Handle(gu.config_for(w, inp.T))
    out, st = _run(h, inp)
    units = list(range(w.units))
    r = ref.event(p, *_unit_inputs(inp, units))
    _check(ref, p, w, inp, out, st, units, r)
