"""Drive the CUDA path (through the C ABI binding) and the CPU oracle side by side.

Both sides get the same seeded inputs from `workload`; nothing the oracle sees
or expects comes from the CUDA path.
"""
import numpy as np
import torch

import oracle
import workload as W
from tests.helpers import check_residency_invariants
from top_cache_gb300 import kvo as K


def _fill_host_rows(kv, wl, units_rl, unit_ids, t0, n_tok, tables=None):
    """Write generator rows for the given units straight into the pinned pool (through the
    units' block tables when the pool is paged)."""
    if not unit_ids:
        return
    if tables is not None:
        B = kv.block_tokens
        for u in unit_ids:
            t = t0
            while t < t0 + n_tok:
                j = t // B
                n = min((j + 1) * B, t0 + n_tok) - t
                pb = int(tables[u][j])
                if pb >= 0:
                    W.token_rows_into(kv.host_block(pb) + (t - j * B) * wl.row_elems * 2, 0, wl.seed,
                                      W.KIND_ROWS, [units_rl[u]], t, n, wl.row_elems)
                t += n
        return
    if kv.U > 1:
        unit_stride = (kv.host_rows(1) - kv.host_rows(0)) // 2
    else:
        unit_stride = 0
    for u in unit_ids:
        base = kv.host_rows(u) + t0 * wl.row_elems * 2
        W.token_rows_into(base, unit_stride, wl.seed, W.KIND_ROWS, [units_rl[u]], t0, n_tok,
                          wl.row_elems)


# Options every Runner applies first (the parity tests select the step path here).
PATH_OPTIONS = {}


class Runner:
    """One workload run: GPU handle + oracle replicas of the checked units."""

    def __init__(self, wl, check_units=None, distinct=False, rows_for=None, steps=None,
                 gather_mode=K.KVO_GATHER_LDG, keys_fn=None, queries=None, max_tokens=None,
                 options=None, idx_int8=False, prefill_from_host=False, paged=0, unmapped=None):
        self.wl = wl
        self.steps = wl.steps if steps is None else steps
        self.units_rl = wl.units_rl()
        self.U = len(self.units_rl)
        self.check = list(range(self.U)) if check_units is None else list(check_units)
        rows_for = self.check if rows_for is None else rows_for
        self.tmax = wl.max_tokens(self.steps) if max_tokens is None else max_tokens
        self.kv = K.Kvo(wl.n_requests, wl.n_layers, self.tmax, wl.topk, wl.hot_capacity,
                        wl.n_pos, wl.row_elems,
                        idx_dtype=K.KVO_IDX_INT8 if idx_int8 else K.KVO_IDX_BF16,
                        host_block_tokens=paged)
        self.tables = None
        if paged:
            # every unit's blocks scattered through the pool (seeded permutation); the
            # (unit, logical block) pairs in `unmapped` are left unmapped (-1)
            mb = -(-self.tmax // paged)
            perm = np.random.default_rng(wl.seed).permutation(self.U * mb).astype(np.int32)
            self.tables = perm.reshape(self.U, mb).copy()
            for (u, j) in (unmapped or ()):
                self.tables[u][j] = -1
            for u in range(self.U):
                self.kv.set_blocks(u, self.tables[u])
        self.kv.set_option(K.KVO_OPT_GATHER_MODE, gather_mode)
        for key, value in {**PATH_OPTIONS, **(options or {})}.items():
            self.kv.set_option(key, value)
        self.keys_fn = keys_fn
        # prefill: rows into the pinned pool, keys into the indexer cache
        _fill_host_rows(self.kv, wl, self.units_rl, rows_for, 0, wl.context, self.tables)
        self.length = wl.context
        self.oracles = {u: oracle.OracleUnit(self.tmax, wl.topk, wl.hot_capacity, wl.n_pos,
                                             wl.row_elems, keep_rows=True, idx_int8=idx_int8)
                        for u in self.check}
        chunk = 16
        for b in range(0, self.U, chunk):
            ids = list(range(b, min(self.U, b + chunk)))
            keys = self._keys([self.units_rl[u] for u in ids], 0, wl.context)
            kd = torch.from_numpy(keys).cuda()
            for j, u in enumerate(ids):
                # host (pageable) or device keys: the library handles both
                self.kv.prefill(u, wl.context, np.ascontiguousarray(keys[j]) if prefill_from_host else kd[j])
                if u in self.oracles:
                    rows = W.token_rows(wl.seed, W.KIND_ROWS, [self.units_rl[u]], 0, wl.context,
                                        wl.row_elems)[0]
                    assert self.oracles[u].append(keys[j], rows) == oracle.OK
            torch.cuda.synchronize()
        if queries is None:
            queries = W.unit_queries(wl.seed, self.units_rl, wl.drift, self.steps, wl.n_pos,
                                     distinct=distinct)
        self.queries = queries

    def _keys(self, units_rl, t0, n):
        if self.keys_fn is not None:
            return self.keys_fn(units_rl, t0, n)
        return W.token_rows(self.wl.seed, W.KIND_KEYS, units_rl, t0, n, 128)

    def append(self, n_new, units=None):
        wl = self.wl
        ids = list(range(self.U)) if units is None else list(units)
        rl = [self.units_rl[u] for u in ids]
        keys = self._keys(rl, self.length, n_new)
        rows = W.token_rows(wl.seed, W.KIND_ROWS, rl, self.length, n_new, wl.row_elems)
        self.kv.append(torch.from_numpy(rows).cuda(), torch.from_numpy(keys).cuda(),
                       units=None if units is None else ids)
        for j, u in enumerate(ids):
            if u in self.oracles:
                assert self.oracles[u].append(keys[j], rows[j]) == oracle.OK
        if units is None:
            self.length += n_new

    def step(self, s, units=None):
        ids = list(range(self.U)) if units is None else list(units)
        q = torch.from_numpy(np.ascontiguousarray(self.queries[s][ids])).cuda()
        out = self.kv.step(q, units=None if units is None else ids)
        torch.cuda.synchronize()
        tok, sl, sc, pay, st = [t.cpu().numpy() for t in out]
        res = {}
        for j, u in enumerate(ids):
            if u in self.oracles:
                r = self.oracles[u].step(self.queries[s][u])
                res[u] = (r, tok[j], sl[j], sc[j], pay[j], st[j])
        return res

    def compare(self, res, state=True):
        for u, (r, tok, sl, sc, pay, st) in res.items():
            assert st == r.status, (u, st, r.status)
            assert np.array_equal(tok, r.tok), "tokens differ, unit %d" % u
            assert np.array_equal(pay, r.pay), "payload differs, unit %d" % u
            assert np.array_equal(sl, r.slot), "slots differ, unit %d" % u
            fin = np.isfinite(r.score)
            assert np.array_equal(np.isfinite(sc), fin)
            # contract: 1e-5 relative; by construction the scores are bit-identical
            assert np.allclose(sc[fin], r.score[fin], rtol=1e-5, atol=0.0)
            assert np.array_equal(sc[fin].view(np.uint32), r.score[fin].view(np.uint32))
            if state:
                self.compare_state(u)

    def compare_state(self, u):
        o = self.oracles[u]
        g = self.kv.export_state(u, with_rows=True)
        assert g["length"] == o.length
        assert g["stamp"] == o.stamp
        assert np.array_equal(g["cache_slots"][: o.length], o.cache_slots()[: o.length])
        assert np.array_equal(g["slot_token"], o.slot_token())
        assert np.array_equal(g["last_use"], o.last_use())
        check_residency_invariants(g["cache_slots"], g["slot_token"], g["last_use"], g["stamp"],
                                   g["length"])
        st = g["slot_token"]
        occ = np.nonzero(st >= 0)[0]
        assert np.array_equal(g["hot"][occ], o.hot()[occ]), "hot rows differ, unit %d" % u
        assert np.array_equal(g["hot"][occ], o.rows()[st[occ]])

    def close(self):
        self.kv.close()
