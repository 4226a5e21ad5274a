"""GPU parity of the query-similarity refresh trigger ("RefreshKV: Updating Small
KV Cache During Long-form Generation", dynamic scheduling) against the oracle.

The decision is an integer decided by a floating comparison: flags must agree
wherever the oracle's fp64 cosine is more than 1e-5 away from the threshold;
cosines agree within 1e-5, updated references within 1e-6 relative."""
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


@pytest.mark.parametrize("L,B,H,G,d,thr", [(4, 8, 4, 7, 128, 0.3), (2, 5, 8, 4, 64, 0.0),
                                           (1, 3, 1, 1, 64, 0.9)])
def test_refresh_matches_oracle_twice(ref, L, B, H, G, d, thr):
    import eviction_gb300 as kvc
    g = torch.Generator().manual_seed(L * 100 + B)
    Hq = H * G
    base = torch.randn((L, B, 1, d), generator=g)
    q = (base + 0.8 * torch.randn((L, B, Hq, d), generator=g)).to(torch.bfloat16)
    q_ref = torch.randn((L, B, d), generator=g)
    q_ref[0, 0] = 0.0                                   # no full step yet
    q_ref[-1, -1] = q[-1, -1].float().mean(dim=0)       # same direction: cosine ~1
    h = kvc.Handle(kvc.Config(L, B, H, G, d, 256, 64))
    r_ref = q_ref.reshape(L * B, d).double().numpy()
    q_bits = wl.bf16_bits(q.reshape(L * B, Hq, d))
    dq = q.cuda().contiguous()
    dref = q_ref.cuda().contiguous()
    flag = torch.empty((L, B), dtype=torch.int32, device="cuda")
    sim = torch.empty((L, B), dtype=torch.float32, device="cuda")
    for call in range(2):
        f_r, s_r, r_ref = ref.refresh_decision(q_bits, r_ref, thr)
        h.refresh_decision(dq, dref, thr, flag, sim)
        torch.cuda.synchronize()
        f_g = flag.reshape(-1).cpu().numpy()
        s_g = sim.reshape(-1).cpu().numpy()
        assert np.all(np.abs(s_g - s_r) <= 1e-5), np.max(np.abs(s_g - s_r))
        far = np.abs(s_r - thr) > 1e-5
        assert np.array_equal(f_g[far], f_r[far])
        assert f_r[0] == 1 and s_r[0] == -2.0 if call == 0 else True
        got = dref.reshape(L * B, d).cpu().double().numpy()
        assert np.allclose(got, r_ref, rtol=1e-6, atol=1e-7)
        if call == 1:
            # every row refreshed by the first call now matches its reference
            assert np.all(s_r[f_r == 0] >= thr - 1e-12)
