"""kvc_event_host: the event from pinned host buffers, pipelined over groups of
layers, gives exactly the device-side kvc_event's results (the same kernels on
slabs of layers), for group sizes that need rounding to 16-byte slab starts
and a ragged last group."""
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


@pytest.mark.parametrize("n_layers,batch,heads,per_stage", [
    (6, 2, 2, 2),   # B*H = 4: stages of 2 layers
    (5, 1, 2, 1),   # B*H = 2: 1 rounds up to 2 layers; last stage holds 1 layer
    (3, 3, 1, 4),   # B*H = 3: a single stage of all layers
    (7, 2, 2, 1),   # one layer per stage
])
def test_host_pipelined_equals_device_event(n_layers, batch, heads, per_stage):
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=n_layers, batch=batch, n_kv_heads=heads,
                  group=4, head_dim=128, prefill=(50, 400), generated=300, budget=256)
    inp = wl.generate(w)
    T = inp.T
    g = gu.to_device(inp)
    h = kvc.Handle(gu.config_for(w, T))
    ref = gu.gpu_event(h, g, T)
    assert h.device_status() == 0
    keys_in = ("q", "k", "v", "pad", "n_carry", "credit")
    host_in = {k: g[k].cpu().pin_memory() for k in keys_in}
    dev_in = {k: torch.empty_like(g[k]) for k in keys_in}
    dev_out = h.outputs(T)
    host_out = {k: torch.full(v.shape, 7, dtype=v.dtype).pin_memory() for k, v in dev_out.items()}
    stream = torch.cuda.Stream()
    h2d, d2h = h.event_from_host(host_in, dev_in, host_out, dev_out, T,
                                 layers_per_stage=per_stage, stream=stream)
    stream.synchronize()
    assert h.device_status() == 0
    # every input is copied except V, which the gather reads in place (pinned)
    assert h2d == sum(t.numel() * t.element_size() for k, t in host_in.items() if k != "v")
    for k in ("k_out", "v_out", "credit_out", "kept_idx", "n_kept"):
        assert torch.equal(host_out[k], ref[k].cpu()), k
    for k in keys_in:
        if k != "v":
            assert torch.equal(dev_in[k], g[k]), k


def test_host_pipelined_argument_errors():
    import eviction_gb300 as kvc
    h = kvc.Handle(kvc.Config(2, 1, 1, 1, 64, 64, 16, window=8))
    with pytest.raises(KeyError):
        h.event_from_host({}, {}, {}, {}, 64)  # missing buffers are caught before the call
    T = 64
    dev_out = h.outputs(T)
    keys = dict(q=(2, 1, 1, 8, 64), k=(2, 1, 1, T, 64), v=(2, 1, 1, T, 64))
    dev_in = {k: torch.zeros(s, dtype=torch.bfloat16, device="cuda") for k, s in keys.items()}
    dev_in.update(pad=torch.zeros(1, dtype=torch.int32, device="cuda"),
                  n_carry=torch.zeros(1, dtype=torch.int32, device="cuda"),
                  credit=torch.zeros((2, 1, 1, T), device="cuda"))
    host_in = {k: v.cpu().pin_memory() for k, v in dev_in.items()}
    host_out = {k: v.cpu().pin_memory() for k, v in dev_out.items()}
    with pytest.raises(kvc.KvcError):  # layers_per_stage must be >= 1
        h.event_from_host(host_in, dev_in, host_out, dev_out, T, layers_per_stage=0)
    h.event_from_host(host_in, dev_in, host_out, dev_out, T, layers_per_stage=1)
    torch.cuda.synchronize()
    assert h.device_status() == 0


def test_host_pipelined_pageable_v_falls_back_to_copies():
    """V in pageable host memory is copied like the other inputs (the gather
    reads V in place only from page-locked, device-mapped memory)."""
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=4, batch=2, n_kv_heads=2, group=4,
                  head_dim=128, prefill=(50, 400), generated=300, budget=256)
    inp = wl.generate(w)
    T = inp.T
    g = gu.to_device(inp)
    h = kvc.Handle(gu.config_for(w, T))
    ref = gu.gpu_event(h, g, T)
    keys_in = ("q", "k", "v", "pad", "n_carry", "credit")
    host_in = {k: (g[k].cpu() if k == "v" else g[k].cpu().pin_memory()) for k in keys_in}
    assert not host_in["v"].is_pinned()
    dev_in = {k: torch.empty_like(g[k]) for k in keys_in}
    dev_out = h.outputs(T)
    host_out = {k: torch.full(v.shape, 7, dtype=v.dtype).pin_memory() for k, v in dev_out.items()}
    h2d, _ = h.event_from_host(host_in, dev_in, host_out, dev_out, T, layers_per_stage=2)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    assert h2d == sum(t.numel() * t.element_size() for t in host_in.values())
    assert torch.equal(dev_in["v"], g["v"])
    for k in ("k_out", "v_out", "credit_out", "kept_idx", "n_kept"):
        assert torch.equal(host_out[k], ref[k].cpu()), k
