"""CUDA path vs CPU oracle, element by element, through the C ABI.

Reduced sizes check every unit at every step (tokens, payloads, slots, status
bit-exact; scores within 1e-5 relative and, by construction, bit-identical;
exported residency state and hot rows bit-exact).  The full-size workloads
run in the launch configuration the benchmark times and check sampled units,
which the oracle replays one by one.  Every workload test runs twice: through
the fused step (one cooperative launch) and through the staged step (one
launch per stage, the default).
"""
import numpy as np
import pytest
import torch

import oracle
import workload as W
from tests import gpu_harness
from tests.gpu_harness import Runner
from tests.helpers import int_bf16
from top_cache_gb300 import kvo as K

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from top_cache_gb300 import build
    build.build()
    yield


@pytest.fixture(params=["fused", "staged"], autouse=True)
def path(request):
    gpu_harness.PATH_OPTIONS = {K.KVO_OPT_FUSED: 1 if request.param == "fused" else 0}
    yield request.param
    gpu_harness.PATH_OPTIONS = {}


def _staged_only(path):
    if path != "staged":
        pytest.skip("option of the staged step")


def _once(path):
    if path != "fused":
        pytest.skip("does not depend on the step path")


def _run(wl, steps=None, check_state=True, count_rows=True, **kw):
    r = Runner(wl, steps=steps, **kw)
    try:
        before = r.kv.stats()
        n_miss = 0
        for s in range(r.steps):
            r.append(wl.n_new)
            res = r.step(s)
            r.compare(res, state=check_state)
            n_miss += sum(v[0].n_miss for v in res.values())
        st = r.kv.stats()
        if count_rows and len(r.check) == r.U:
            # transferred rows == deduplicated miss count, counted by the copy kernel
            assert st["rows_h2d"] - before["rows_h2d"] == n_miss
            assert st["misses"] - before["misses"] == n_miss
        return st, n_miss
    finally:
        r.close()


# ---------------------------------------------------------------- reduced sizes
def test_single_4k_full_size():
    st, n_miss = _run(W.WORKLOADS["single_4k"])
    assert st["unit_steps"] == 20 and 0 < n_miss < 20 * 256


def test_batch16x8_mtp3_reduced():
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=2, n_layers=2, context=4001,
                   topk=256, hot_capacity=512, steps=8)
    _run(wl)


def test_batch32x16_reduced_ragged():
    wl = W.reduced(W.WORKLOADS["batch32x16_64k"], n_requests=2, n_layers=3, context=6003,
                   topk=300, hot_capacity=1200, steps=6)
    _run(wl)


def test_long_context_reduced_multi_piece():
    # two units of ~150k tokens: each unit spans dozens of score CTAs and the
    # candidate union exceeds the select kernel's shared-memory buffer
    wl = W.reduced(W.WORKLOADS["long_1m_mtp3"], n_requests=1, n_layers=2, context=150001,
                   topk=512, hot_capacity=4096, steps=3)
    _run(wl)


@pytest.mark.parametrize("drift", W.SWEEP_DRIFTS)
def test_sweep_reduced(drift):
    wl = W.reduced(W.WORKLOADS["sweep64x4_16k_mtp3"], n_requests=4, n_layers=2, context=3000,
                   topk=128, hot_capacity=256, steps=6, drift=drift)
    _run(wl)


def test_bulk_gather_mode(path):
    _staged_only(path)
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=2, n_layers=2, context=3000,
                   topk=256, hot_capacity=600, steps=5)
    _run(wl, gather_mode=K.KVO_GATHER_BULK)


@pytest.mark.parametrize("spec", [0, 500, 900])
def test_speculation_settings_agree(spec):
    # 0: every scan starts from an empty threshold; otherwise from the last
    # step's k-th score scaled by spec/1000
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=2, n_layers=2, context=5000,
                   topk=256, hot_capacity=600, steps=6)
    _run(wl, options={K.KVO_OPT_SPECULATE: spec})


@pytest.mark.parametrize("drift", [0.0, 0.9])
def test_speculation_without_margin_falls_back_exactly(drift):
    # no margin and fresh queries: the previous k-th score is often too high;
    # those units must be rescored and the results must stay exact
    wl = W.Workload("nomargin", 3, 2, 4000, 4, 4, 200, 900, 8, drift, 84)
    st, _ = _run(wl, distinct=True, options={K.KVO_OPT_SPECULATE: 1000})
    if drift == 0.0:
        assert st["rescored"] > 0


@pytest.mark.parametrize("groups", [2, 3, 5])
def test_unit_groups_two_streams(groups, path):
    _staged_only(path)
    # the miss-row copy of each group overlaps the next group's scoring
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=3, n_layers=2, context=3001,
                   topk=256, hot_capacity=600, steps=5)
    _run(wl, options={K.KVO_OPT_GROUPS: groups})


@pytest.mark.parametrize("groups,sms,int8", [(2, 8, False), (3, 32, False), (5, 2, False), (2, 8, True)])
def test_unit_groups_split_sms(groups, sms, int8, path):
    _staged_only(path)
    # the first `sms` CTAs of each group's score launch copy the previous group's rows
    # while the others score, then help with what is left (KVO_OPT_GROUP_GATHER_SMS):
    # results as without groups, each row copied once
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=3, n_layers=2, context=3001,
                   topk=256, hot_capacity=600, steps=5)
    _run(wl, idx_int8=int8, options={K.KVO_OPT_GROUPS: groups, K.KVO_OPT_GROUP_GATHER_SMS: sms})


def test_few_score_ctas_long_pieces(path):
    _staged_only(path)
    # a cap on scoring CTAs makes each CTA stream long pieces (many compactions)
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=1, n_layers=3, context=40000,
                   topk=512, hot_capacity=1024, steps=3)
    _run(wl, options={K.KVO_OPT_SCORE_CTAS: 2})


def test_positions_1_to_8():
    for P in (2, 3, 5, 8):
        wl = W.Workload("p%d" % P, 1, 2, 2500, P, P, 64, 64 * P, 4, 0.5, 77)
        _run(wl, distinct=True)


def test_capacity_overflow_transactional():
    # distinct per-position queries with P*k > C overflow on some steps
    wl = W.Workload("cap", 2, 2, 2000, 4, 4, 64, 160, 6, 0.3, 78)
    r = Runner(wl, distinct=True)
    try:
        seen = 0
        for s in range(r.steps):
            r.append(wl.n_new)
            res = r.step(s)
            r.compare(res)
            seen += sum(1 for v in res.values() if v[0].status == oracle.ECAPACITY)
        assert seen > 0
    finally:
        r.close()


def test_forced_ties_and_zero_query():
    # integer keys in {-1, 0, 1}, each row repeated three times: many equal scores
    def keys_fn(units_rl, t0, n):
        out = np.empty((len(units_rl), n, 128), np.uint16)
        for i, rl in enumerate(units_rl):
            base = W.token_rows(5, W.KIND_KEYS, [rl], t0 // 3, (t0 + n + 2) // 3 - t0 // 3 + 1, 128)[0]
            f = np.clip(np.rint(W.bf16_to_f32(base)), -1, 1)
            idx = np.arange(t0, t0 + n) // 3 - t0 // 3
            out[i] = int_bf16(f[idx])
        return out

    wl = W.Workload("ties", 1, 3, 1500, 2, 2, 100, 300, 5, 0.9, 79)
    q = W.unit_queries(wl.seed, wl.units_rl(), wl.drift, wl.steps, wl.n_pos, distinct=True)
    qf = np.clip(np.rint(W.bf16_to_f32(q)), -1, 1)
    q = int_bf16(qf)
    q[1, :, 0, :] = 0  # step 1, position 0: all scores are +0, order by token alone
    _run(wl, keys_fn=keys_fn, queries=q)


def test_units_subset_ragged_lengths_and_repeat():
    wl = W.Workload("subset", 2, 3, 2048, 2, 2, 128, 400, 6, 0.8, 80)
    r = Runner(wl)
    try:
        # append to every unit, then step a changing subset; lengths diverge
        for s in range(r.steps):
            sub = [u for u in range(r.U) if (u + s) % 3 != 0]
            r.append(wl.n_new, units=sub)
            res = r.step(s, units=sub)
            r.compare(res)
        # a repeated step with the same queries and no append is all hits
        last = [u for u in range(r.U) if (u + r.steps - 1) % 3 != 0]
        before = r.kv.stats()
        res = r.step(r.steps - 1, units=last[:2])
        r.compare(res)
        assert all(v[0].n_miss == 0 for v in res.values())
        after = r.kv.stats()
        assert after["rows_h2d"] == before["rows_h2d"]
        assert after["bytes_h2d"] == before["bytes_h2d"]
    finally:
        r.close()


def test_empty_and_short_units():
    # context 0: the first steps see fewer tokens than k (and than P)
    wl = W.Workload("short", 1, 2, 0, 3, 3, 16, 64, 8, 0.9, 81)
    _run(wl)


def test_append_past_max_tokens_rejected(path):
    _once(path)
    wl = W.Workload("range", 1, 1, 64, 1, 1, 8, 16, 2, 0.9, 82)
    r = Runner(wl)
    try:
        r.append(1)
        r.append(1)
        with pytest.raises(K.KvoError) as e:
            r.append(1)
        assert e.value.code == K.KVO_ERANGE
        assert r.kv.export_state(0)["length"] == 66
    finally:
        r.close()


def test_bad_arguments(path):
    _once(path)
    with pytest.raises(K.KvoError) as e:
        K.kvo_create(1, 1, 100, 64, 32, 1)  # capacity < k
    assert e.value.code == K.KVO_EINVAL
    kv = K.Kvo(1, 2, 100, 8, 16, 1)
    try:
        q = torch.zeros((2, 1, 128), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(K.KvoError) as e:
            kv.step(q, units=[1, 1])
        assert e.value.code == K.KVO_EINVAL
        with pytest.raises(K.KvoError) as e:
            kv.step(q, units=[0, 5])
        assert e.value.code == K.KVO_ERANGE
        with pytest.raises(K.KvoError):
            kv.set_option(99, 0)
    finally:
        kv.close()


def test_select_stateless(path):
    _once(path)
    n, P, k = 5, 3, 200
    lengths = [0, 150, 3000, 12345, 777]
    stride = 12352
    keys = np.zeros((n, stride, 128), np.uint16)
    for i in range(n):
        keys[i, : lengths[i]] = W.token_rows(83, W.KIND_KEYS, [(i, 0)], 0, lengths[i], 128)[0]
    q = W.unit_queries(83, [(i, 0) for i in range(n)], 0.9, 1, P, distinct=True)[0]
    rng = np.random.default_rng(83)
    cs = np.full((n, stride), -1, np.int32)
    for i in range(n):
        res = rng.choice(max(1, lengths[i]), size=min(lengths[i], 400), replace=False)
        cs[i, res] = rng.permutation(len(res)).astype(np.int32)
    dev = lambda a: torch.from_numpy(a).cuda()
    kd, qd, csd = dev(keys), dev(np.ascontiguousarray(q)), dev(cs)
    tok = torch.empty((n, P, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((n, P, k), dtype=torch.float32, device="cuda")
    pay = torch.empty((n, P, k), dtype=torch.int32, device="cuda")
    wsb = K.kvo_select_workspace_size(n, P, k, 0)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    K.kvo_select(kd, stride, csd, lengths, n, P, k, qd, tok, sc, pay, ws, wsb)
    torch.cuda.synchronize()
    tok, sc, pay = tok.cpu().numpy(), sc.cpu().numpy(), pay.cpu().numpy()
    for i in range(n):
        o = oracle.OracleUnit(max(1, lengths[i]), k, k * P, P, row_elems=8, keep_rows=False)
        o.append(keys[i, : lengths[i]])
        r = o.step(q[i])
        assert np.array_equal(tok[i], r.tok)
        fin = np.isfinite(r.score)
        assert np.array_equal(sc[i][fin].view(np.uint32), r.score[fin].view(np.uint32))
        # payload rule applied to the caller's cache_slots
        exp = np.where(r.tok >= 0, np.where(cs[i][np.maximum(r.tok, 0)] >= 0,
                                            cs[i][np.maximum(r.tok, 0)], -(r.tok + 1)),
                       K.KVO_PAD_PAYLOAD)
        assert np.array_equal(pay[i], exp)


# ---------------------------------------------------------------- fused step only
@pytest.mark.parametrize("piece", [128, 384])
def test_fused_small_pieces(piece, path):
    # many pieces per unit: several CTAs share each unit, the piece ring of a
    # CTA wraps many times, and finishers run while other units still score
    _once(path)
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=2, n_layers=3, context=6001,
                   topk=256, hot_capacity=600, steps=5)
    _run(wl, options={K.KVO_OPT_PIECE_TOKENS: piece})


@pytest.mark.parametrize("gather_ctas", [0, 1, -2])
def test_fused_gather_cta_split(gather_ctas, path):
    # 0: only scorer CTAs fill rows, after their last piece; -2 (all SMs but
    # two): two scorer CTAs do every piece while the rest wait for rows
    _once(path)
    if gather_ctas < 0:
        gather_ctas += torch.cuda.get_device_properties(0).multi_processor_count
    wl = W.reduced(W.WORKLOADS["sweep64x4_16k_mtp3"], n_requests=3, n_layers=2, context=5000,
                   topk=128, hot_capacity=256, steps=4, drift=0.5)
    _run(wl, options={K.KVO_OPT_GATHER_CTAS: gather_ctas, K.KVO_OPT_PIECE_TOKENS: 1024})


def test_fused_options_validated(path):
    _once(path)
    kv = K.Kvo(1, 2, 1000, 16, 64, 2)
    try:
        for key, value in ((K.KVO_OPT_PIECE_TOKENS, 100), (K.KVO_OPT_PIECE_TOKENS, 0),
                           (K.KVO_OPT_FUSED, 3), (K.KVO_OPT_GATHER_CTAS, -1),
                           (K.KVO_OPT_GATHER_CTAS, 1 << 20)):
            with pytest.raises(K.KvoError) as e:
                kv.set_option(key, value)
            assert e.value.code == K.KVO_EINVAL
        assert kv.get_option(K.KVO_OPT_FUSED) == 2  # the default: chosen per call
        kv.set_option(K.KVO_OPT_GATHER_CTAS, 3)
        assert kv.get_option(K.KVO_OPT_GATHER_CTAS) == 3
        kv.set_option(K.KVO_OPT_PROFILE, 1)
        q = torch.zeros((2, 2, 128), dtype=torch.bfloat16, device="cuda")
        kv.step(q)
        prof = kv.profile_read()
        assert prof["fused"][1] == 1 and prof["score"][1] == 0  # no measurement yet: fused
        assert kv.stats()["fused_steps"] == 1
    finally:
        kv.close()


def test_paths_alternate_per_step(path):
    # the two step paths share all persistent state (residency, LRU lists,
    # speculative thresholds): switching between them every call stays exact
    _once(path)
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=2, n_layers=3, context=5001,
                   topk=256, hot_capacity=600, steps=8)
    r = Runner(wl)
    try:
        for s in range(r.steps):
            r.kv.set_option(K.KVO_OPT_FUSED, s % 2)
            r.append(wl.n_new)
            r.compare(r.step(s))
        assert r.kv.stats()["fused_steps"] == r.steps // 2
    finally:
        r.close()


# ---------------------------------------------------------------- int8 indexer
def test_int8_indexer_reduced(path):
    wl = W.reduced(W.WORKLOADS["batch16x8_32k_mtp3"], n_requests=2, n_layers=2, context=4001,
                   topk=256, hot_capacity=512, steps=6)
    _run(wl, idx_int8=True)


def test_int8_indexer_positions_and_host_prefill(path):
    for P in (1, 3, 8):
        wl = W.Workload("i8p%d" % P, 1, 2, 2300, P, P, 64, 64 * P, 4, 0.5, 85)
        _run(wl, distinct=True, idx_int8=True, prefill_from_host=(P == 3))


def test_int8_indexer_ties_short_units_and_rescans(path):
    # integer keys make many equal int8 scores; context 0 starts below k and P
    wl = W.Workload("i8short", 1, 2, 0, 3, 3, 16, 64, 8, 0.9, 86)
    _run(wl, idx_int8=True)
    wl = W.Workload("i8nomargin", 3, 2, 4000, 4, 4, 200, 900, 6, 0.0, 87)
    st, _ = _run(wl, distinct=True, idx_int8=True, options={K.KVO_OPT_SPECULATE: 1000})
    assert st["rescored"] > 0


# ---------------------------------------------------------------- full sizes
def _meminfo_gb():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 1e6
    except OSError:
        pass
    return 0.0


def test_full_batch16x8_mtp3_sampled():
    wl = W.WORKLOADS["batch16x8_32k_mtp3"]
    _run(wl, check_units=[0, 61, 127], count_rows=False)


def test_full_batch16x8_mtp3_grouped_sampled(path):
    _staged_only(path)
    wl = W.WORKLOADS["batch16x8_32k_mtp3"]
    _run(wl, steps=20, check_units=[0, 40, 127], count_rows=False, options={K.KVO_OPT_GROUPS: 4})


def test_full_batch16x8_mtp3_split_sms_sampled(path):
    _staged_only(path)
    wl = W.WORKLOADS["batch16x8_32k_mtp3"]
    _run(wl, steps=12, check_units=[1, 63, 126], count_rows=False,
         options={K.KVO_OPT_GROUPS: 2, K.KVO_OPT_GROUP_GATHER_SMS: 32})


def test_full_batch16x8_mtp3_int8_sampled():
    wl = W.WORKLOADS["batch16x8_32k_mtp3"]
    _run(wl, steps=20, check_units=[0, 77, 127], count_rows=False, idx_int8=True)


def test_full_long_1m_mtp3_sampled():
    wl = W.WORKLOADS["long_1m_mtp3"]
    _run(wl, steps=5, check_units=[3], count_rows=False)


def test_full_sweep_sampled():
    base = W.WORKLOADS["sweep64x4_16k_mtp3"]
    for drift in W.SWEEP_DRIFTS:
        wl = W.reduced(base, drift=drift)
        _run(wl, steps=10, check_units=[0, 255], count_rows=False)


def test_full_batch32x16_sampled():
    wl = W.WORKLOADS["batch32x16_64k"]
    need = wl.n_units * wl.max_tokens() * wl.row_elems * 2 / 1e9
    if _meminfo_gb() < need * 1.3 + 16:
        pytest.skip("host memory below %.0f GB for the pinned pool" % (need * 1.3 + 16))
    _run(wl, steps=12, check_units=[5, 400], count_rows=False)


# ---------------------------------------------------------------- paged host pool
def test_paged_host_pool():
    # the host pool in 64-row blocks scattered through it by per-unit block tables: every
    # appended row and every miss row goes through the table
    wl = W.Workload("paged", 2, 2, 3000, 4, 4, 256, 1100, 6, 0.5, 96)
    _run(wl, paged=64)


def test_paged_host_pool_bulk_gather(path):
    _staged_only(path)
    wl = W.Workload("pagedb", 2, 2, 1500, 2, 2, 128, 400, 4, 0.3, 97)
    _run(wl, paged=32, gather_mode=K.KVO_GATHER_BULK)


def test_paged_unmapped_block_is_counted_not_touched():
    # unit 1's block for the appended tokens is unmapped: its rows are neither written nor
    # read (a gather leaves the hot row as it was); unit 0 still matches the oracle
    wl = W.Workload("pagedx", 1, 2, 256, 2, 2, 64, 256, 3, 0.5, 98)
    B = 64
    r = Runner(wl, paged=B, unmapped=[(1, wl.context // B)], check_units=[0])
    try:
        before = r.kv.stats()
        for s in range(r.steps):
            r.append(wl.n_new)
            r.compare(r.step(s))
        st = r.kv.stats()
        assert st["block_errors"] - before["block_errors"] >= r.steps * wl.n_new
        assert st["timeouts"] == 0
    finally:
        r.close()


def test_paged_pool_arguments():
    kv = K.Kvo(1, 2, 100, 8, 16, 1, 576, host_block_tokens=16)
    try:
        with pytest.raises(K.KvoError):
            kv.set_blocks(0, [0] * 8)  # 7 entries per unit (ceil(100 / 16))
        with pytest.raises(K.KvoError):
            kv.set_blocks(0, [14])  # 2 units x 7 blocks = 14 blocks: ids 0..13
        with pytest.raises(K.KvoError):
            kv.set_blocks(2, [0])  # unit out of range
        with pytest.raises(K.KvoError):
            kv.host_block(14)
        with pytest.raises(K.KvoError):
            K.kvo_host_rows(kv.h, 0)  # paged: rows are reached by block
        kv.set_blocks(1, [13, -1], first_block=5)
        assert kv.host_block(13) > 0
    finally:
        kv.close()
    with pytest.raises(K.KvoError):
        K.Kvo(1, 1, 100, 8, 16, 1, 576, host_block_tokens=12)  # not a multiple of 8
