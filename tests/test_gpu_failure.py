"""The failure path on the GPU without a fault: a bounded wait that runs out on
purpose (a barrier nothing completes) reports KVC_STATUS_WAIT_TIMEOUT through
the status word, and the context keeps working afterwards."""
import time

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


def test_wait_timeout_is_reported_and_context_survives():
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=2)
    inp = wl.generate(w)
    T = inp.T
    g = gu.to_device(inp)
    h = kvc.Handle(gu.config_for(w, T))
    before = gu.gpu_event(h, g, T)
    kept0 = before["kept_idx"].clone()
    assert h.device_status() == 0

    t0 = time.monotonic()
    h.wait_self_test()
    bits = h.device_status()  # synchronises the stream
    dt = time.monotonic() - t0
    assert bits & 0x1, f"status {bits:#x}: the timeout bit is missing"
    assert 1.0 <= dt < 60.0, f"the wait gave up after {dt:.2f} s"
    assert h.device_status() == 0  # reading clears the word

    # the context still runs the whole event, with the same result
    after = gu.gpu_event(h, g, T)
    assert h.device_status() == 0
    assert torch.equal(after["kept_idx"], kept0)
    assert torch.equal(after["k_out"], before["k_out"])
    torch.cuda.synchronize()
    assert np.isfinite(after["credit_out"].cpu().numpy()).all()
