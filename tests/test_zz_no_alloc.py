"""kvo_select_noalloc against kvo_select, through the C ABI.

kvo_select_noalloc serves callers that may not allocate memory where they
select, such as an operator hosted by a framework that owns all device memory
and forbids its extensions to call cudaMalloc, or a latency-critical decode
loop that cannot afford an allocation.  It runs the same scoring and fused
top-k as kvo_select with its scratch in a fixed array inside the library.

This file is collected last so that, when it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workload as W
from top_cache_gb300 import kvo as K

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from top_cache_gb300 import build
    build.build()
    yield


def _case(seed, n, P, k, lengths, stride):
    keys = np.zeros((n, stride, 128), np.uint16)
    for i in range(n):
        keys[i, : lengths[i]] = W.token_rows(seed, W.KIND_KEYS, [(i, 0)], 0, lengths[i], 128)[0]
    q = np.ascontiguousarray(W.unit_queries(seed, [(i, 0) for i in range(n)], 0.5, 1, P,
                                            distinct=True)[0])
    rng = np.random.default_rng(seed)
    cs = np.full((n, stride), -1, np.int32)
    for i in range(n):
        m = min(lengths[i], 200)
        if m:
            res = rng.choice(lengths[i], size=m, replace=False)
            cs[i, res] = rng.permutation(m).astype(np.int32)
    return (torch.from_numpy(keys).cuda(), torch.from_numpy(q).cuda(), torch.from_numpy(cs).cuda())


def _outputs(n, P, k):
    return (torch.full((n, P, k), 7, dtype=torch.int32, device="cuda"),
            torch.full((n, P, k), 7.0, dtype=torch.float32, device="cuda"),
            torch.full((n, P, k), 7, dtype=torch.int32, device="cuda"))


def _free_bytes_after(call, tries=3):
    """Free device memory before and after call(); repeated when other users of the
    device move the figure (the comparison only detects memory the call keeps)."""
    for _ in range(tries):
        torch.cuda.synchronize()
        before = torch.cuda.mem_get_info()[0]
        call()
        torch.cuda.synchronize()
        after = torch.cuda.mem_get_info()[0]
        if after >= before:
            return True
    return False


def test_noalloc_matches_select_on_two_calls():
    stride = 12352
    cases = [(5, 3, 160, [0, 77, 3001, 12345, 640], 91), (7, 2, 256, [4096, 1, 9000, 129, 0, 5000, 12000], 92)]
    for call, (n, P, k, lengths, seed) in enumerate(cases):
        keys, q, cs = _case(seed, n, P, k, lengths, stride)
        ref = _outputs(n, P, k)
        wsb = K.kvo_select_workspace_size(n, P, k, 0)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        st_ref = torch.full((1,), 0xAB, dtype=torch.int32, device="cuda")
        K.kvo_select(keys, stride, cs, lengths, n, P, k, q, ref[0], ref[1], ref[2], ws, wsb, status=st_ref)
        out = _outputs(n, P, k)
        st = torch.full((1,), 0xAB, dtype=torch.int32, device="cuda")
        kept = _free_bytes_after(lambda: K.kvo_select_noalloc(keys, stride, cs, lengths, n, P, k, q,
                                                              out[0], out[1], out[2], status=st))
        tok, sc, pay = [t.cpu().numpy() for t in out]
        rtok, rsc, rpay = [t.cpu().numpy() for t in ref]
        # both calls completed normally: the status word was cleared and nothing set it
        assert int(st_ref.item()) == 0 and int(st.item()) == 0
        assert np.array_equal(tok, rtok)
        assert np.array_equal(pay, rpay)
        fin = np.isfinite(rsc)
        assert np.array_equal(np.isfinite(sc), fin)
        assert np.allclose(sc[fin], rsc[fin], rtol=1e-5, atol=0.0)
        if call > 0:
            # after the first call on the device (which materialises the fixed
            # array under lazy module loading), calls keep no device memory
            assert kept


def test_noalloc_rejects_sizes_beyond_its_scratch():
    keys = torch.zeros((65, 64, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((65, 1, 128), dtype=torch.bfloat16, device="cuda")
    tok, sc, pay = _outputs(65, 1, 8)
    with pytest.raises(K.KvoError) as e:
        K.kvo_select_noalloc(keys, 64, None, [64] * 65, 65, 1, 8, q, tok, sc, pay)
    assert e.value.code == K.KVO_ERANGE
    # 64 units, 4 positions, k = 2048: accepted exactly when kvo_select's workspace
    # for that shape fits the 16 MiB fixed scratch (the need grows with the SM count)
    keys = torch.zeros((64, 64, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((64, 4, 128), dtype=torch.bfloat16, device="cuda")
    tok, sc, pay = _outputs(64, 4, 2048)
    need = K.kvo_select_workspace_size(64, 4, 2048, torch.cuda.current_device())
    if need > 16 << 20:
        with pytest.raises(K.KvoError) as e:
            K.kvo_select_noalloc(keys, 64, None, [64] * 64, 64, 4, 2048, q, tok, sc, pay)
        assert e.value.code == K.KVO_ERANGE
        return
    K.kvo_select_noalloc(keys, 64, None, [64] * 64, 64, 4, 2048, q, tok, sc, pay)
    torch.cuda.synchronize()
    t = tok.cpu().numpy()
    for p in range(4):  # position p sees 64 - (3 - p) tokens, then padding
        vis = 64 - (3 - p)
        assert np.all(t[:, p, :vis] >= 0) and np.all(t[:, p, vis:] == -1)
