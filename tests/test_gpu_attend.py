"""Sparse attention over the hot buffer (kvo_attend) vs the CPU oracle (reading R13).

The CUDA path attends over the hot rows its own kvo_step made resident, by slot; the
oracle attends over its own copy of the main-KV history, by the tokens its own step
selected (identical to the CUDA path's, which the step parity checks bit for bit).

Tolerance, from the arithmetic of the kernel: scores are exact bf16 products summed in
fp32 (relative error far below 2^-8); each softmax weight is rounded to bf16 (relative
error <= 2^-8) and the output is the exact mean under the rounded weights, so it moves by
at most 2^-8 * max_i |v_i - out| / (1 - 2^-8); the output is then rounded to bf16 (another
2^-8 * |out|).  lse moves by at most log(1 + 2^-8) < 2^-8 from the rounded weights.  The
test allows 1.1 times these bounds plus 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import workload as W
from tests.gpu_harness import Runner
from top_cache_gb300 import kvo as K

pytestmark = pytest.mark.gpu

SCALE = 1.0 / np.sqrt(192.0)
EPS = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    from top_cache_gb300 import build
    build.build()
    yield


def _bf16(a):
    return W.bf16_to_f32(a).astype(np.float64)


def _attend_gpu(r, step, H, scale, units=None):
    """kvo_attend on the slots of the last kvo_step; returns (queries, out, lse) on the host."""
    ids = list(range(r.U)) if units is None else list(units)
    P = r.wl.n_pos
    q = W.attention_queries(r.wl.seed, [r.units_rl[u] for u in ids], step, P, H)
    qd = torch.from_numpy(q.view(np.int16)).cuda()
    out = torch.full((len(ids), P, H, 512), -1, dtype=torch.int16, device="cuda")
    lse = torch.full((len(ids), P, H), float("nan"), dtype=torch.float32, device="cuda")
    r.kv.attend(qd, scale, out, lse, units=None if units is None else ids)
    torch.cuda.synchronize()
    assert r.kv.stats()["timeouts"] == 0
    return q, out.cpu().numpy().view(np.uint16), lse.cpu().numpy()


def _compare(r, res, q, out, lse, scale, ids=None):
    """Every checked unit and position against the oracle."""
    ids = list(range(r.U)) if ids is None else list(ids)
    checked = 0
    for j, u in enumerate(ids):
        if u not in res:
            continue
        o = r.oracles[u]
        toks = res[u][0].tok
        rows = o.rows()
        for p in range(r.wl.n_pos):
            ref, ref_lse = o.attend(toks[p], q[j, p], scale)
            got = _bf16(out[j, p])
            valid = toks[p][(toks[p] >= 0) & (toks[p] < o.length)]
            if valid.size == 0:
                assert np.all(got == 0)
                assert np.all(np.isneginf(lse[j, p]))
                continue
            v = _bf16(rows[valid, :512])                     # [n][512]
            spread = np.abs(v[None, :, :] - ref[:, None, :]).max(axis=1)  # [H][512]
            tol = 1.1 * EPS * (spread / (1 - EPS) + np.abs(ref)) + 1e-5
            err = np.abs(got - ref)
            bad = err > tol
            assert not bad.any(), "unit %d pos %d: %d elements off, worst %.3g (tol %.3g)" % (
                u, p, bad.sum(), err[bad].max(), tol[bad][np.argmax(err[bad])])
            assert np.all(np.abs(lse[j, p] - ref_lse) <= 1.1 * EPS + 1e-5 * (1 + np.abs(ref_lse)))
            checked += 1
    return checked


def _run(wl, H=128, scales=(SCALE,), steps=None, check_units=None, units_each_step=None):
    r = Runner(wl, steps=steps, check_units=check_units)
    try:
        n = 0
        for s in range(r.steps):
            r.append(wl.n_new)
            res = r.step(s)
            r.compare(res, state=False)
            for sc in scales:
                q, out, lse = _attend_gpu(r, s, H, sc)
                n += _compare(r, res, q, out, lse, sc)
        return n
    finally:
        r.close()


def test_attend_reduced_mtp3():
    # two 128-row blocks per list (one for each CTA of a pair's rope turn), four
    # positions, three steps of a drifting query
    wl = W.Workload("att", 2, 2, 3000, 4, 4, 256, 1100, 3, 0.9, 90)
    assert _run(wl, scales=(SCALE, 0.5, 0.01)) == 2 * 2 * 4 * 3 * 3


def test_attend_ragged_list_and_pads():
    # k = 200 is not a multiple of 128 (last block partial) and the context is shorter
    # than k, so every list carries pads (slot -1)
    wl = W.Workload("attpad", 1, 2, 120, 2, 2, 200, 512, 2, 0.5, 91)
    assert _run(wl) > 0


def test_attend_two_head_groups():
    # k = 96: a single, partial block (the rope slab goes to the first CTA of each pair)
    wl = W.Workload("atth", 1, 2, 2000, 2, 2, 96, 400, 2, 0.8, 92)
    assert _run(wl, H=256, scales=(SCALE, 0.3)) > 0


def test_attend_growing_maximum_rescales():
    # a large scale makes the running maximum jump by far more than 2^8 from block to
    # block, so the output accumulator is rescaled in TMEM many times
    wl = W.Workload("attgrow", 1, 1, 4000, 1, 1, 512, 1024, 1, 0.9, 93)
    assert _run(wl, scales=(2.0, 8.0)) > 0


def test_attend_unit_subset():
    # k = 64: a single, partial block
    wl = W.Workload("attsub", 2, 2, 1500, 2, 2, 64, 256, 2, 0.7, 94)
    r = Runner(wl)
    try:
        r.append(wl.n_new)
        res = r.step(0)
        r.compare(res, state=False)
        # attention of units 3 and 1 only, in that order, on their rows of the step output
        ids = [3, 1]
        slots = torch.stack([r.kv.slots[3], r.kv.slots[1]]).contiguous()
        q = W.attention_queries(wl.seed, [r.units_rl[u] for u in ids], 0, wl.n_pos, 128)
        qd = torch.from_numpy(q.view(np.int16)).cuda()
        out = torch.zeros((2, wl.n_pos, 128, 512), dtype=torch.int16, device="cuda")
        r.kv.attend(qd, SCALE, out, None, slots=slots, units=ids)
        torch.cuda.synchronize()
        lse = np.zeros((2, wl.n_pos, 128), np.float32)
        got = out.cpu().numpy().view(np.uint16)
        sub = {u: res[u] for u in ids}
        # lse not requested: compare the outputs only
        for j, u in enumerate(ids):
            o = r.oracles[u]
            for p in range(wl.n_pos):
                ref, ref_lse = o.attend(sub[u][0].tok[p], q[j, p], SCALE)
                lse[j, p] = ref_lse
        assert _compare(r, sub, q, got, lse, SCALE, ids=ids) == 2 * wl.n_pos
    finally:
        r.close()


def test_attend_bad_arguments():
    wl = W.Workload("attbad", 1, 1, 256, 1, 1, 32, 64, 1, 0.5, 95)
    r = Runner(wl)
    try:
        r.append(1)
        r.step(0)
        q = torch.zeros((1, 1, 128, 576), dtype=torch.int16, device="cuda")
        out = torch.zeros((1, 1, 128, 512), dtype=torch.int16, device="cuda")
        with pytest.raises(K.KvoError):
            r.kv.attend(q[..., :64, :].contiguous(), SCALE, out)  # 64 heads: not a multiple of 128
        with pytest.raises(K.KvoError):
            r.kv.attend(q[..., ::2], SCALE, out)  # a strided view is refused by the binding
        with pytest.raises(K.KvoError):
            r.kv.attend(q, float("nan"), out)
        qm = torch.zeros(1 * 128 * 576 + 8, dtype=torch.int16, device="cuda")[1:1 + 128 * 576]
        with pytest.raises(K.KvoError):
            r.kv.attend(qm.view(1, 1, 128, 576), SCALE, out)  # misaligned queries
        with pytest.raises(K.KvoError):
            r.kv.attend(q, SCALE, out, units=[5])  # unit out of range
    finally:
        r.close()


def test_full_batch16x8_mtp3_attend_sampled():
    # the benchmark workload at full size: 128 units x 4 positions x 128 heads, k = 2048;
    # the oracle replays three units
    wl = W.WORKLOADS["batch16x8_32k_mtp3"]
    assert _run(wl, steps=2, check_units=[0, 77, 127]) == 3 * 4 * 2


# ---------------------------------------------------------------------------
# Deferred fill (KVO_OPT_DEFER_FILL): the step assigns the miss rows' slots and the
# attention kernel reads those rows from the pinned pool itself, uses them and writes
# them to their hot slots (the pages' Copy-SFA operator: misses fetched inside sparse
# attention).  After the attention call the state must be exactly the oracle's, hot
# rows included, and every miss row must have crossed the host link once.
# ---------------------------------------------------------------------------
def _run_fetch(wl, H=128, scale=SCALE, steps=None, check_units=None, distinct=False, paged=0, fused=None):
    opts = {K.KVO_OPT_DEFER_FILL: 1}
    if fused is not None:
        opts[K.KVO_OPT_FUSED] = fused
    r = Runner(wl, steps=steps, check_units=check_units, distinct=distinct, paged=paged, options=opts)
    try:
        n = 0
        for s in range(r.steps):
            r.append(wl.n_new)
            st0 = r.kv.stats()
            res = r.step(s)
            r.compare(res, state=False)  # outputs only: exporting the state would complete the fill
            q, out, lse = _attend_gpu(r, s, H, scale)
            n += _compare(r, res, q, out, lse, scale)
            st1 = r.kv.stats()
            misses = st1["misses"] - st0["misses"]
            # each part of each miss row is claimed and written by exactly one CTA
            assert st1["bytes_h2d"] - st0["bytes_h2d"] == misses * wl.row_elems * 2
            assert st1["rows_h2d"] - st0["rows_h2d"] == misses
            for u in res:
                r.compare_state(u)  # slot maps, stamps and every occupied hot row
        return n
    finally:
        r.close()


def test_fetch_reduced_mtp3():
    # four positions of one query walk share most rows: the first position's pairs
    # fetch them, the others find them written (or read the host pool again)
    wl = W.Workload("attf", 2, 2, 3000, 4, 4, 256, 1100, 3, 0.9, 96)
    assert _run_fetch(wl) == 2 * 2 * 4 * 3


def test_fetch_distinct_queries_staged_and_fused():
    # positions with their own queries list different rows; both step paths
    wl = W.Workload("attfd", 2, 3, 2500, 4, 4, 128, 700, 3, 0.6, 97)
    assert _run_fetch(wl, distinct=True, fused=0) == 2 * 3 * 4 * 3
    assert _run_fetch(wl, distinct=True, fused=1) == 2 * 3 * 4 * 3


def test_fetch_all_misses_and_ragged():
    # drift 0: nearly every selected row is a miss; k = 200 leaves a partial last block
    wl = W.Workload("attf0", 3, 2, 2000, 4, 4, 200, 900, 3, 0.0, 98)
    assert _run_fetch(wl) > 0


def test_fetch_paged_pool():
    # rows reached through scattered 128-row blocks of a paged pool
    wl = W.Workload("attfp", 2, 2, 1800, 2, 2, 256, 600, 3, 0.8, 99)
    assert _run_fetch(wl, paged=128) > 0


def test_fetch_flushed_when_no_attention_follows():
    # a deferred step followed by another step, by an export or by attention on another
    # unit list completes the fill with a copy kernel; the state stays the oracle's
    wl = W.Workload("attff", 2, 2, 2000, 2, 2, 128, 512, 4, 0.7, 100)
    r = Runner(wl, options={K.KVO_OPT_DEFER_FILL: 1})
    try:
        r.append(wl.n_new)
        r.compare(r.step(0), state=True)  # export: flushed
        r.append(wl.n_new)
        res = r.step(1)
        r.compare(res, state=False)
        r.append(wl.n_new)
        res = r.step(2)  # flushes step 1's rows first
        r.compare(res, state=False)
        ids = [1, 3]  # another unit list: flushed, then plain attention
        slots = torch.stack([r.kv.slots[1], r.kv.slots[3]]).contiguous()
        q = W.attention_queries(wl.seed, [r.units_rl[u] for u in ids], 2, wl.n_pos, 128)
        out = torch.zeros((2, wl.n_pos, 128, 512), dtype=torch.int16, device="cuda")
        lse = torch.zeros((2, wl.n_pos, 128), dtype=torch.float32, device="cuda")
        r.kv.attend(torch.from_numpy(q.view(np.int16)).cuda(), SCALE, out, lse, slots=slots, units=ids)
        torch.cuda.synchronize()
        sub = {u: res[u] for u in ids}
        assert _compare(r, sub, q, out.cpu().numpy().view(np.uint16), lse.cpu().numpy(), SCALE, ids=ids) == 2 * wl.n_pos
        for u in range(r.U):
            r.compare_state(u)
        r.append(wl.n_new)
        r.compare(r.step(3), state=True)
        assert r.kv.stats()["timeouts"] == 0
    finally:
        r.close()


def test_full_batch16x8_mtp3_fetch_sampled():
    # the benchmark workload at full size with the fill inside the attention kernel
    wl = W.WORKLOADS["batch16x8_32k_mtp3"]
    assert _run_fetch(wl, steps=2, check_units=[0, 77, 127]) == 3 * 4 * 2


def test_fetch_sweep_drift0_reduced():
    # the hit-rate sweep's all-miss point (drift 0), reduced: 32 units
    wl = W.reduced(W.WORKLOADS["sweep64x4_16k_mtp3"], n_requests=8, drift=0.0, steps=3)
    assert _run_fetch(wl, check_units=[0, 13, 31]) == 3 * 4 * 3
