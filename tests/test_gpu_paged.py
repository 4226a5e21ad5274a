"""GPU parity of the paged compaction ("Adaptive Mass-Segmented KV Compression for
Long-Form Reasoning", Appendix E) against the oracle: pools, new block tables,
free stack and compacted credit bit-exact; failures change nothing; and after a
real event, the paged result read through the new tables equals the dense
compaction."""
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


def _pool_state(rng, L, H, d, bs, lens, extra_free):
    B = len(lens)
    max_blocks = max((n + bs - 1) // bs for n in lens)
    n_old = sum((n + bs - 1) // bs for n in lens)
    n_blocks = n_old + extra_free
    perm = rng.permutation(n_blocks).astype(np.int32)
    table = np.full((B, max_blocks), -1, np.int32)
    k = 0
    for b, n in enumerate(lens):
        nb = (n + bs - 1) // bs
        table[b, :nb] = perm[k:k + nb]
        k += nb
    free = np.zeros(n_blocks, np.int32)
    free[:n_blocks - n_old] = perm[n_old:]
    kp = rng.integers(0, 65535, (L, n_blocks, H, bs, d)).astype(np.uint16)
    vp = rng.integers(0, 65535, (L, n_blocks, H, bs, d)).astype(np.uint16)
    return table, free, n_blocks - n_old, kp, vp


def _dev_bf16(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _run_gpu(h, kp, vp, bs, lens, pad, kept, nk, credit, T, table, free, top):
    L, B, H, budget = kept.shape
    k_pool, v_pool = _dev_bf16(kp.copy()), _dev_bf16(vp.copy())
    t_new = torch.full(table.shape, -7, dtype=torch.int32, device="cuda")
    fl = torch.from_numpy(free.copy()).cuda()
    ft = torch.tensor([top], dtype=torch.int32, device="cuda")
    c_out = torch.full((L, B, H, budget), 9.0, device="cuda")
    h.compact_paged(k_pool, v_pool, bs, torch.from_numpy(np.asarray(lens, np.int32)).cuda(),
                    torch.from_numpy(pad).cuda(), torch.from_numpy(kept).cuda(),
                    torch.from_numpy(nk).cuda(), torch.from_numpy(credit).cuda(), T, c_out,
                    torch.from_numpy(table).cuda(), t_new, fl, ft)
    torch.cuda.synchronize()
    return (wl.bf16_bits(k_pool), wl.bf16_bits(v_pool), t_new.cpu().numpy(), fl.cpu().numpy(),
            int(ft.item()), c_out.cpu().numpy(), h.device_status())


@pytest.mark.parametrize("seed,bs,d", [(0, 16, 64), (1, 8, 128), (2, 64, 64)])
def test_paged_matches_oracle(ref, seed, bs, d):
    import eviction_gb300 as kvc
    rng = np.random.default_rng(seed)
    L, H, G, budget = 2, 2, 2, 48
    lens = [100, 37, 160, 5]
    B, T = len(lens), max(lens)
    pad = np.array([T - n for n in lens], np.int32)
    table, free, top, kp, vp = _pool_state(rng, L, H, d, bs, lens, extra_free=20)
    kept = np.full((L, B, H, budget), -1, np.int32)
    nk = np.zeros((L, B, H), np.int32)
    for l in range(L):
        for b, n in enumerate(lens):
            for hh in range(H):
                m = min(budget, n)
                kept[l, b, hh, :m] = np.sort(rng.choice(n, m, replace=False)) + pad[b]
                nk[l, b, hh] = m
    credit = rng.random((L, B, H, T)).astype(np.float32)
    h = kvc.Handle(kvc.Config(L, B, H, G, d, T, budget, window=8))
    gk, gv, gt, gf, gtop, gc, st = _run_gpu(h, kp, vp, bs, lens, pad, kept, nk, credit, T, table,
                                            free, top)
    rc, rk, rv, rt, rf, rtop = ref.compact_paged(kp, vp, lens, pad, kept, nk, table, free, top, bs)
    assert rc == 0 and st == 0
    assert np.array_equal(gt, rt)
    assert gtop == rtop and np.array_equal(gf[:gtop], rf[:rtop])
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
    # credit: dense gather at the kept slots, zero past n_kept
    for l in range(L):
        for b in range(B):
            for hh in range(H):
                n = nk[l, b, hh]
                assert np.array_equal(gc[l, b, hh, :n], credit[l, b, hh, kept[l, b, hh, :n]])
                assert not gc[l, b, hh, n:].any()


def test_paged_failures_change_nothing(ref):
    import eviction_gb300 as kvc
    rng = np.random.default_rng(4)
    L, H, G, d, bs, budget = 1, 2, 1, 64, 16, 40
    lens = [90, 70]
    B, T = len(lens), max(lens)
    pad = np.array([T - n for n in lens], np.int32)
    table, free, top, kp, vp = _pool_state(rng, L, H, d, bs, lens, extra_free=2)  # needs 6
    kept = np.zeros((L, B, H, budget), np.int32)
    nk = np.full((L, B, H), budget, np.int32)
    for b, n in enumerate(lens):
        kept[0, b, :, :] = np.arange(budget) + pad[b]
    credit = np.zeros((L, B, H, T), np.float32)
    h = kvc.Handle(kvc.Config(L, B, H, G, d, T, budget, window=8))
    gk, gv, gt, gf, gtop, gc, st = _run_gpu(h, kp, vp, bs, lens, pad, kept, nk, credit, T, table,
                                            free, top)
    assert st & 0x4 and gtop == top and np.array_equal(gk, kp) and np.array_equal(gf, free)
    # bad index: a slot in the left padding of sequence 1
    table, free, top, kp, vp = _pool_state(rng, L, H, d, bs, lens, extra_free=20)
    kept[0, 1, 0, 0] = 0
    h2 = kvc.Handle(kvc.Config(L, B, H, G, d, T, budget, window=8))
    gk, gv, gt, gf, gtop, gc, st = _run_gpu(h2, kp, vp, bs, lens, pad, kept, nk, credit, T, table,
                                            free, top)
    assert st & 0x2 and gtop == top and np.array_equal(gv, vp) and np.array_equal(gf, free)


def test_event_then_paged_equals_dense():
    """A real event's kept indices, applied to a paged copy of its cache, give the
    same rows (read through the new tables) as the dense compaction."""
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=2, batch=4, n_kv_heads=2, group=4,
                  head_dim=64, prefill=(50, 300), generated=200, budget=128)
    inp = wl.generate(w)
    T = inp.T
    g = gu.to_device(inp)
    h = kvc.Handle(gu.config_for(w, T))
    out = gu.gpu_event(h, g, T)
    L, B, H, d = w.n_layers, w.batch, w.n_kv_heads, w.head_dim
    bs = 16
    lens = (T - inp.pad).tolist()
    rng = np.random.default_rng(0)
    table, free, top, _, _ = _pool_state(rng, L, H, d, bs, lens, extra_free=64)
    n_blocks = len(free)
    # scatter the dense cache into the pool through the old table
    kd = wl.bf16_bits(inp.k)   # [L, B, H, T, d]
    vd = wl.bf16_bits(inp.v)
    kp = np.zeros((L, n_blocks, H, bs, d), np.uint16)
    vp = np.zeros_like(kp)
    pad = inp.pad.numpy()
    for b, n in enumerate(lens):
        for t in range(n):
            kp[:, table[b, t // bs], :, t % bs] = kd[:, b, :, pad[b] + t]
            vp[:, table[b, t // bs], :, t % bs] = vd[:, b, :, pad[b] + t]
    kept = out["kept_idx"].cpu().numpy()
    nk = out["n_kept"].cpu().numpy()
    credit = np.zeros((L, B, H, T), np.float32)
    gk, gv, gt, gf, gtop, gc, st = _run_gpu(h, kp, vp, bs, lens, pad.astype(np.int32), kept, nk,
                                            credit, T, table, free, top)
    assert st == 0
    k_dense = wl.bf16_bits(out["k_out"])
    for b in range(B):
        n = int(nk[0, b, 0])
        for j in range(n):
            assert np.array_equal(gk[:, gt[b, j // bs], :, j % bs], k_dense[:, b, :, j])
