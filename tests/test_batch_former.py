"""Host-only tests of the live-batch former (slots for sessions, per-step
metadata).  No GPU: the former is plain host code behind the C ABI."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def dsb():
    import os
    from session_decode_step_dsb_gb300 import build, dsb
    if not os.path.exists(dsb.LIB_PATH):
        build.build()
    return dsb


def test_join_form_commit_leave(dsb):
    bf = dsb.BatchFormer(4, 100, 1)
    a = bf.join(10)
    b = bf.join(20)
    assert (a, b) == (0, 1)
    bf.submit(b, [7])
    bf.submit(a, [5])
    bi, sl, tk = bf.form()
    assert list(bi) == [0, 1] and list(sl) == [11, 21] and list(tk) == [5, 7]
    bf.commit(bi)
    assert bf.length(a) == 11 and bf.length(b) == 21
    bi, sl, tk = bf.form()
    assert len(bi) == 0  # nothing queued
    bf.leave(a)
    c = bf.join(0)
    assert c == 0 and bf.length(c) == 0  # the freed slot is reused, lowest first
    bf.submit(c, [1])
    bf.submit(b, [2])
    bi, sl, tk = bf.form()
    assert list(bi) == [0, 1] and list(sl) == [1, 22]


def test_slot_exhaustion_and_bad_calls(dsb):
    bf = dsb.BatchFormer(2, 10, 2)
    bf.join(0)
    bf.join(8)
    with pytest.raises(dsb.DsbError):
        bf.join(0)                 # every slot is live
    with pytest.raises(dsb.DsbError):
        bf.submit(1, [1, 2])       # 8 + 2 = 10 ok ... then
        bf.commit([1])
        bf.submit(1, [3, 4])       # 10 + 2 > ctx
    with pytest.raises(dsb.DsbError):
        bf.leave(5)
    with pytest.raises(dsb.DsbError):
        bf.commit([0])             # slot 0 has nothing queued


def test_form_matches_step_contract(dsb):
    """Formed metadata satisfies the step's contract: distinct slots in range,
    seq_lens in [T, ctx], T tokens per sequence, slot order."""
    rng = np.random.default_rng(0)
    F, C, T = 16, 64, 3
    bf = dsb.BatchFormer(F, C, T)
    live = {}
    for step in range(200):
        op = rng.integers(0, 3)
        if op == 0 and len(live) < F:
            s = bf.join(int(rng.integers(0, C - T)))
            live[s] = True
        elif op == 1 and live:
            s = int(rng.choice(list(live)))
            bf.leave(s)
            del live[s]
        for s in list(live):
            if bf.length(s) + T <= C:
                bf.submit(s, rng.integers(0, 1000, T))
        bi, sl, tk = bf.form()
        assert len(set(bi)) == len(bi) and np.all(np.diff(bi) > 0)
        assert np.all((bi >= 0) & (bi < F))
        assert np.all((sl >= T) & (sl <= C)) and tk.size == T * len(bi)
        before = {int(s): bf.length(int(s)) for s in bi}
        bf.commit(bi)
        for s in bi:
            assert bf.length(int(s)) == before[int(s)] + T


def test_random_ops_match_a_dictionary_model(dsb):
    """Random join / leave / submit / form / commit sequences against a plain
    model: lowest free slot on join, lengths advanced by T on commit, and
    form() listing exactly the queued sessions in slot order with their
    tokens; rejected calls change nothing."""
    rng = np.random.default_rng(5)
    F, C, T = 6, 40, 2
    bf = dsb.BatchFormer(F, C, T)
    length, queued = {}, {}
    for _ in range(400):
        op = int(rng.integers(0, 4))
        if op == 0:
            pre = int(rng.integers(0, C))
            if len(length) == F:
                with pytest.raises(dsb.DsbError):
                    bf.join(pre)
            else:
                s = bf.join(pre)
                assert s == min(set(range(F)) - set(length))
                length[s] = pre
        elif op == 1:
            s = int(rng.integers(0, F))
            if s in length:
                bf.leave(s)
                del length[s]
                queued.pop(s, None)
            else:
                with pytest.raises(dsb.DsbError):
                    bf.leave(s)
        elif op == 2 and length:
            s = int(rng.choice(sorted(length)))
            toks = rng.integers(0, 50000, T).astype(np.int32)
            if length[s] + T > C:
                with pytest.raises(dsb.DsbError):
                    bf.submit(s, toks)
            else:
                bf.submit(s, toks)
                queued[s] = toks
        else:
            bi, sl, tk = bf.form()
            want = sorted(queued)
            assert list(bi) == want
            assert list(sl) == [length[s] + T for s in want]
            assert np.array_equal(tk, np.concatenate([queued[s] for s in want]) if want else np.zeros(0, np.int32))
            if want and rng.random() < 0.8:
                bf.commit(bi)
                for s in want:
                    length[s] += T
                queued.clear()
        for s in range(F):
            assert bf.length(s) == length.get(s, -1)
