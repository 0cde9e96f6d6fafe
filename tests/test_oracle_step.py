"""Pins of the oracle's selection and residency logic against independent models.

Inputs are small integers so every score is an exact integer; the expected
top-k is a plain full sort, the expected residency comes from an explicit
recency-list model (tests.helpers.ListLRU), which shares no code with the
oracle's stamp-and-sort formulation.
"""
import numpy as np
import pytest

import oracle
import workload as W
from tests.helpers import ListLRU, check_residency_invariants, exact_topk, int_bf16, rand_int_bf16


def _drive(seed, n_init, n_steps, n_new, k, C, P, distinct_queries=True, lo=-2, hi=2,
           dup_rows=False):
    """Run the oracle and the independent models side by side on integer data."""
    rng = np.random.default_rng(seed)
    tmax = n_init + n_steps * n_new
    kint, kb = rand_int_bf16(rng, (tmax, 128), lo, hi)
    if dup_rows:  # force many exact score ties
        src = rng.integers(0, max(1, tmax // 4), size=tmax)
        kint, kb = kint[src], kb[src]
    rows = rng.integers(0, 65535, size=(tmax, 8), dtype=np.uint16)
    u = oracle.OracleUnit(tmax, k, C, P, row_elems=8, keep_rows=True)
    assert u.append(kb[:n_init], rows[:n_init]) == oracle.OK
    model = ListLRU(C)
    length = n_init
    for s in range(n_steps):
        if s > 0 and n_new:
            assert u.append(kb[length:length + n_new], rows[length:length + n_new]) == oracle.OK
            length += n_new
        if distinct_queries:
            qint, qb = rand_int_bf16(rng, (P, 128), lo, hi)
        else:
            qi1, qb1 = rand_int_bf16(rng, (1, 128), lo, hi)
            qint, qb = np.repeat(qi1, P, 0), np.repeat(qb1, P, 0)
        cs_before = u.cache_slots()
        r = u.step(qb)
        # --- top-k per position against a plain full sort (R2, R3) ---
        wanted = set()
        for p in range(P):
            vis = max(0, length - (P - 1 - p))
            sc = kint[:vis] @ qint[p]
            toks, scs = exact_topk(sc, vis, k)
            assert r.tok[p].tolist() == toks
            assert r.score[p].tolist() == scs
            for i, t in enumerate(toks):
                if t < 0:
                    assert r.pay[p, i] == oracle.PAD_PAYLOAD
                else:
                    wanted.add(t)
                    cs = cs_before[t]
                    assert r.pay[p, i] == (cs if cs >= 0 else -(t + 1))  # R4
        # --- residency against the explicit-list model (R5, R6, R7) ---
        fills = model.step(wanted)
        if fills is None:
            assert r.status == oracle.ECAPACITY
            assert np.all(r.slot == -1)
            assert r.n_miss == 0
            assert np.array_equal(u.cache_slots(), cs_before)
            continue
        assert r.status == oracle.OK
        assert r.misses() == fills
        for p in range(P):
            for i in range(k):
                t = r.tok[p, i]
                assert r.slot[p, i] == (model.tok_slot[t] if t >= 0 else -1)
        assert u.slot_token().tolist() == model.slot_tok
        # recency order of the oracle's stamps equals the model's list order
        lu = u.last_use()
        assert sorted(range(C), key=lambda s_: (int(lu[s_]), s_)) == model.order
        check_residency_invariants(u.cache_slots(), u.slot_token(), lu, u.stamp, length)
        hot = u.hot()
        st = u.slot_token()
        for s_ in np.nonzero(st >= 0)[0]:
            assert np.array_equal(hot[s_], rows[st[s_]])
    return u


@pytest.mark.parametrize("seed", range(40))
def test_tiny_single_position(seed):
    _drive(seed, n_init=24, n_steps=6, n_new=1, k=5, C=9, P=1)


@pytest.mark.parametrize("seed", range(40))
def test_tiny_mtp_positions(seed):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([2, 3, 4]))
    _drive(seed, n_init=40, n_steps=6, n_new=P, k=6, C=16, P=P)


@pytest.mark.parametrize("seed", range(20))
def test_forced_ties(seed):
    _drive(seed, n_init=48, n_steps=5, n_new=2, k=8, C=12, P=2, lo=-1, hi=1, dup_rows=True)


@pytest.mark.parametrize("seed", range(10))
def test_capacity_overflow_is_transactional(seed):
    # distinct queries per position with C < P*k overflow often
    _drive(seed, n_init=40, n_steps=6, n_new=4, k=6, C=7, P=4)


def test_fewer_visible_tokens_than_k_pads():
    _drive(1, n_init=3, n_steps=4, n_new=1, k=8, C=8, P=1)
    _drive(2, n_init=1, n_steps=3, n_new=2, k=5, C=12, P=3)


def test_empty_unit_selects_nothing():
    u = oracle.OracleUnit(8, 4, 4, 2, row_elems=8)
    r = u.step(np.zeros((2, 128), np.uint16))
    assert r.status == oracle.OK and r.n_miss == 0
    assert np.all(r.tok == -1) and np.all(r.slot == -1)
    assert np.all(r.pay == oracle.PAD_PAYLOAD) and np.all(np.isneginf(r.score))


def test_mtp_visibility_excludes_later_tokens():
    # the last tokens score highest; position p must not see the last P-1-p
    P, L0 = 4, 20
    keys = np.zeros((L0, 128), np.float32)
    keys[:, 0] = np.arange(L0)
    u = oracle.OracleUnit(L0, 3, 16, P, row_elems=8)
    u.append(int_bf16(keys))
    q = np.zeros((P, 128), np.float32)
    q[:, 0] = 1.0
    r = u.step(int_bf16(q))
    for p in range(P):
        top = L0 - 1 - (P - 1 - p)
        assert r.tok[p].tolist() == [top, top - 1, top - 2]


def test_full_capacity_never_evicts():
    # capacity >= every token ever cached: no slot is ever overwritten
    rng = np.random.default_rng(5)
    n0, steps, k = 30, 8, 6
    tmax = n0 + steps
    _, kb = rand_int_bf16(rng, (tmax, 128))
    u = oracle.OracleUnit(tmax, k, tmax, 1, row_elems=8)
    u.append(kb[:n0])
    filled = {}
    for s in range(steps):
        if s:
            u.append(kb[n0 + s - 1:n0 + s])
        _, qb = rand_int_bf16(rng, (1, 128))
        r = u.step(qb)
        for t, sl in r.misses():
            assert sl not in filled.values()
            filled[t] = sl
        st = u.slot_token()
        for t, sl in filled.items():
            assert st[sl] == t


def test_disjoint_selections_evict_every_resident():
    # keys in G groups, group g has a dedicated dimension; step s queries group s % G,
    # so consecutive selections are disjoint and C = |W| forces a full turnover.
    G, per, k = 4, 6, 6
    L0 = G * per
    keys = np.zeros((L0, 128), np.float32)
    for t in range(L0):
        keys[t, t // per] = 1.0 + (t % per)
    u = oracle.OracleUnit(L0, k, k, 1, row_elems=8, keep_rows=True)
    u.append(int_bf16(keys), np.arange(L0 * 8, dtype=np.uint16).reshape(L0, 8))
    for s in range(2 * G):
        g = s % G
        q = np.zeros((1, 128), np.float32)
        q[0, g] = 1.0
        r = u.step(int_bf16(q))
        assert r.status == oracle.OK
        assert sorted(r.tok[0].tolist()) == list(range(g * per, (g + 1) * per))
        assert r.n_miss == k  # every selected token was absent
        assert sorted(u.slot_token().tolist()) == list(range(g * per, (g + 1) * per))


def test_repeated_step_moves_no_rows():
    # the same queries again with no append: a 100%-hit step fills nothing
    rng = np.random.default_rng(9)
    _, kb = rand_int_bf16(rng, (64, 128))
    u = oracle.OracleUnit(64, 8, 32, 3, row_elems=8)
    u.append(kb)
    _, qb = rand_int_bf16(rng, (3, 128))
    r1 = u.step(qb)
    assert r1.n_miss > 0
    hot_before = u.hot().copy()
    r2 = u.step(qb)
    assert r2.n_miss == 0 and r2.status == oracle.OK
    assert np.array_equal(r2.tok, r1.tok) and np.array_equal(r2.slot, r1.slot)
    assert np.all(r2.pay >= 0)  # every winner already says "hit"
    assert np.array_equal(u.hot(), hot_before)


def test_append_past_capacity_is_rejected():
    u = oracle.OracleUnit(4, 2, 4, 1, row_elems=8)
    assert u.append(np.zeros((3, 128), np.uint16)) == oracle.OK
    assert u.append(np.zeros((2, 128), np.uint16)) == oracle.ERANGE
    assert u.length == 3


def test_generated_workload_invariants():
    # a slice of the 16x8 MTP3 workload shape at reduced size, random N(0,1) data
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=1, n_layers=2, context=2048,
                   topk=128, hot_capacity=256, steps=8)
    units = wl.units_rl()
    tmax = wl.max_tokens()
    keys = W.token_rows(wl.seed, W.KIND_KEYS, units, 0, tmax, 128)
    rows = W.token_rows(wl.seed, W.KIND_ROWS, units, 0, tmax, wl.row_elems)
    qs = W.unit_queries(wl.seed, units, wl.drift, wl.steps, wl.n_pos)
    for i in range(len(units)):
        u = oracle.OracleUnit(tmax, wl.topk, wl.hot_capacity, wl.n_pos, wl.row_elems)
        u.append(keys[i, :wl.context], rows[i, :wl.context])
        length = wl.context
        total_miss = 0
        for s in range(wl.steps):
            if s:
                u.append(keys[i, length:length + wl.n_new], rows[i, length:length + wl.n_new])
                length += wl.n_new
            r = u.step(qs[s, i])
            assert r.status == oracle.OK
            total_miss += r.n_miss
            check_residency_invariants(u.cache_slots(), u.slot_token(), u.last_use(), u.stamp,
                                       length)
            st = u.slot_token()
            hot = u.hot()
            occ = np.nonzero(st >= 0)[0]
            assert np.array_equal(hot[occ], rows[i, st[occ]])
            # every winner resident, slot output points at it
            cs = u.cache_slots()
            ok = r.tok >= 0
            assert np.all(cs[r.tok[ok]] == r.slot[ok])
            # scores are non-increasing along each list
            assert np.all(np.diff(r.score, axis=1) <= 0)
        assert total_miss < wl.steps * wl.topk  # the walk gives a nontrivial hit rate


def test_thousand_random_tiny_shapes():
    # brute force over many shapes at once: L <= 64, k <= 8, C <= 16, P in 1..4, small
    # integer values (so ties are frequent), distinct or shared queries across positions
    for seed in range(1000):
        rng = np.random.default_rng(50_000 + seed)
        P = int(rng.integers(1, 5))
        k = int(rng.integers(1, 9))
        C = int(rng.integers(k, 17))
        n_new = int(rng.integers(0, 3))
        n_steps = int(rng.integers(1, 5))
        n_init = int(rng.integers(0, 64 - n_steps * n_new + 1))
        _drive(seed, n_init=n_init, n_steps=n_steps, n_new=n_new, k=k, C=C, P=P,
               distinct_queries=bool(rng.integers(0, 2)), lo=-1, hi=int(rng.integers(1, 3)),
               dup_rows=bool(rng.integers(0, 2)))
