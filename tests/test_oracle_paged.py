"""Pins of the oracle's paged compaction ("Adaptive Mass-Segmented KV Compression
for Long-Form Reasoning", Appendix E): per-head content through the new block
table equals a plain gather of the kept positions, blocks are conserved, the
allocation order is the stated one, and failures change nothing."""
import numpy as np
import pytest


def _setup(seed, L=2, H=3, d=8, bs=4, lens=(10, 7, 13), budget=6, extra_free=6):
    rng = np.random.default_rng(seed)
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
    top = n_blocks - n_old
    kp = rng.integers(0, 65535, (L, n_blocks, H, bs, d)).astype(np.uint16)
    vp = rng.integers(0, 65535, (L, n_blocks, H, bs, d)).astype(np.uint16)
    T = max(lens)
    pad = np.array([T - n for n in lens], np.int32)
    kept = np.full((L, B, H, budget), -1, np.int32)
    nk = np.zeros((L, B, H), np.int32)
    for l in range(L):
        for b, n in enumerate(lens):
            for h in range(H):
                m = min(budget, n)
                sel = np.sort(rng.choice(n, m, replace=False)) + pad[b]
                kept[l, b, h, :m] = sel
                nk[l, b, h] = m
    return dict(kp=kp, vp=vp, table=table, free=free, top=top, kept=kept, nk=nk,
                lens=np.array(lens, np.int32), pad=pad, bs=bs, budget=budget)


def _logical(pool, table, b, t, bs):
    """Rows [L, H, d] of logical token t of sequence b."""
    return pool[:, table[b, t // bs], :, t % bs, :]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_content_through_new_table(ref, seed):
    s = _setup(seed)
    rc, kp, vp, tnew, fl, top = ref.compact_paged(s["kp"], s["vp"], s["lens"], s["pad"], s["kept"],
                                                  s["nk"], s["table"], s["free"], s["top"], s["bs"])
    assert rc == 0
    L, B, H, _ = s["kept"].shape
    for l in range(L):
        for b in range(B):
            for h in range(H):
                for j in range(s["nk"][l, b, h]):
                    t = s["kept"][l, b, h, j] - s["pad"][b]
                    src_k = _logical(s["kp"], s["table"], b, t, s["bs"])[l, h]
                    src_v = _logical(s["vp"], s["table"], b, t, s["bs"])[l, h]
                    assert np.array_equal(_logical(kp, tnew, b, j, s["bs"])[l, h], src_k)
                    assert np.array_equal(_logical(vp, tnew, b, j, s["bs"])[l, h], src_v)


def test_blocks_conserved_and_allocation_order(ref):
    s = _setup(5)
    rc, kp, vp, tnew, fl, top = ref.compact_paged(s["kp"], s["vp"], s["lens"], s["pad"], s["kept"],
                                                  s["nk"], s["table"], s["free"], s["top"], s["bs"])
    assert rc == 0
    n_blocks = s["kp"].shape[1]
    used = tnew[tnew >= 0]
    free = fl[:top]
    assert len(set(used.tolist())) == len(used)                 # no block used twice
    assert sorted(used.tolist() + free.tolist()) == list(range(n_blocks))  # none lost
    # the old blocks are free again
    old = s["table"][s["table"] >= 0]
    assert set(old.tolist()) <= set(free.tolist())
    # sequence b takes the next ceil(n_kept/bs) entries from the top of the stack
    need = [(int(s["nk"][0, b, 0]) + s["bs"] - 1) // s["bs"] for b in range(len(s["lens"]))]
    start = s["top"] - sum(need)
    k = start
    for b, nb in enumerate(need):
        assert tnew[b, :nb].tolist() == s["free"][k:k + nb].tolist()
        assert np.all(tnew[b, nb:] == -1)
        k += nb


def test_exhausted_pool_and_bad_index_change_nothing(ref):
    s = _setup(7, extra_free=1)  # 1 free block: not enough for the new blocks
    rc, kp, vp, tnew, fl, top = ref.compact_paged(s["kp"], s["vp"], s["lens"], s["pad"], s["kept"],
                                                  s["nk"], s["table"], s["free"], s["top"], s["bs"])
    assert rc == -1 and top == s["top"] and np.array_equal(kp, s["kp"])
    s = _setup(8)
    s["kept"][1, 1, 0, 0] = 0  # before the left padding of sequence 1 (pad 6): out of range
    rc, kp, vp, tnew, fl, top = ref.compact_paged(s["kp"], s["vp"], s["lens"], s["pad"], s["kept"],
                                                  s["nk"], s["table"], s["free"], s["top"], s["bs"])
    assert rc == -1 and top == s["top"] and np.array_equal(vp, s["vp"])
