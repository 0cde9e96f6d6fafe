"""Layerwise prefill offload (kvo_lw_*) vs the CPU oracle (readings R14-R16 of
oracle/layerwise.py; "Layerwise and Sparse KV Cache Offloading Design", section 3).

Each pass runs a stand-in compute per layer on the caller's stream: it reads the layer's
cached rows from the buffer the library hands out (their digest must equal the oracle's, so
a load of the wrong rows, or a buffer reused before its compute read it, is caught) and
writes the chunk's new rows after them; the library saves those rows to the host pool,
which must equal the oracle's after every pass.  Bytes moved are checked against the plan.
"""
import numpy as np
import pytest
import torch

import workload as W
from oracle import layerwise as LW
from top_cache_gb300 import kvo as K

pytestmark = pytest.mark.gpu

SEED = 3001


@pytest.fixture(scope="module", autouse=True)
def _built():
    from top_cache_gb300 import build
    build.build()
    yield


def _run(N, L0, chunks, I=1, B=3, lookahead=1, row=576, spin=0):
    T = L0 + sum(chunks)
    lw = K.Layerwise(N, T, I, B, lookahead, row)
    try:
        n_phys, phys = LW.plan(N, tuple(range(I)), B)
        assert lw.n_phys == n_phys and lw.phys.tolist() == phys
        units = [(0, l) for l in range(N)]
        o = LW.LayerwiseOracle(N, T, row)
        prefix = W.token_rows(SEED, W.KIND_ROWS, units, 0, L0, row)
        for l in range(N):
            lw.host_rows(l)[:L0] = prefix[l]
        o.fill_prefix(prefix)
        lw.set_length(L0)
        t = L0
        h2d = 0
        for p, c in enumerate(chunks):
            chunk = W.token_rows(SEED, W.KIND_ROWS, units, t, c, row)
            cd = torch.from_numpy(chunk.view(np.int16)).cuda()
            expect = o.forward(chunk)
            digests = torch.zeros(N, dtype=torch.int64, device="cuda")
            lw.begin(c)
            for l in range(N):
                buf = lw.layer(l)
                if spin:  # a longer compute, so that loads run ahead of it
                    torch.cuda._sleep(spin)
                digests[l] = (buf[:t].to(torch.int64) & 0xFFFF).sum()
                buf[t:t + c].copy_(cd[l])
                lw.layer_done(l)
            lw.end()
            torch.cuda.synchronize()
            assert digests.cpu().tolist() == expect, "pass %d: a layer read the wrong cached rows" % p
            # every reusable layer reloads unless it has a buffer to itself; independent
            # layers load only on the first pass
            reload = (N - I) if min(B, N - I) < (N - I) else 0
            loads = N if p == 0 else reload
            h2d += loads * t * row * 2
            t += c
        for l in range(N):
            assert np.array_equal(lw.host_rows(l)[:t], o.host[l, :t]), "host rows of layer %d" % l
        st = lw.stats()
        assert st["bytes_d2h"] == N * sum(chunks) * row * 2
        assert st["bytes_h2d"] == h2d
    finally:
        lw.close()


def test_four_trays_several_passes():
    _run(8, 300, [100, 57, 128], I=1, B=3, lookahead=1)


def test_one_shared_buffer_with_deep_lookahead():
    # every reusable layer shares one buffer: each load must wait for the previous layer's save
    _run(6, 200, [64, 64], I=1, B=1, lookahead=3, spin=20000)


def test_a_buffer_per_layer_stays_resident():
    _run(5, 150, [32, 32, 32], I=1, B=8, lookahead=2)


def test_no_independent_layer_and_empty_prefix():
    _run(7, 0, [40, 24], I=0, B=2, lookahead=2)


def test_zero_token_chunk_and_ragged_rows():
    _run(4, 99, [0, 33, 1], I=2, B=1, lookahead=1, row=64)


def test_pages_plan_78_layers_four_trays():
    _run(78, 2048, [512, 512], I=1, B=3, lookahead=1)


def test_usage_errors():
    lw = K.Layerwise(3, 100, 1, 1, 1, 576)
    try:
        with pytest.raises(K.KvoError):
            lw.layer(0)  # no open pass
        lw.set_length(10)
        lw.begin(5)
        with pytest.raises(K.KvoError):
            lw.begin(5)  # pass already open
        with pytest.raises(K.KvoError):
            lw.layer(1)  # out of order
        lw.layer(0)
        with pytest.raises(K.KvoError):
            lw.layer_done(1)
        with pytest.raises(K.KvoError):
            lw.end()  # layers missing
        lw.layer_done(0)
        for l in (1, 2):
            lw.layer(l)
            lw.layer_done(l)
        with pytest.raises(K.KvoError):
            lw.set_length(3)  # inside a pass
        lw.end()
        with pytest.raises(K.KvoError):
            lw.begin(90)  # past max_tokens
        torch.cuda.synchronize()
    finally:
        lw.close()
    with pytest.raises(K.KvoError):
        K.Layerwise(4, 100, 1, 0, 1, 576)  # reusable layers without a shared buffer
    with pytest.raises(K.KvoError):
        K.Layerwise(4, 100, 1, 2, 0, 576)  # lookahead 0
