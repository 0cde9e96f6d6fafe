"""Failure detection without a GPU fault: the bounded waits give up and report it.

kvo_wait_selftest runs one thread through the library's two wait primitives (a spin on a
global flag, an mbarrier phase wait) on conditions nothing satisfies; both must expire after
their limit and be reported as KVO_ETIMEOUT, and the device must stay usable (a decode step
afterwards still matches the oracle bit for bit)."""
import pytest

import workload as W
from tests.gpu_harness import Runner
from top_cache_gb300 import kvo as K

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from top_cache_gb300 import build
    build.build()
    yield


def test_bounded_waits_expire_and_the_device_survives():
    limit = 2_000_000  # 2 ms per wait
    rc, waited = K.kvo_wait_selftest(0, limit)
    assert rc == K.KVO_ETIMEOUT
    assert 2 * limit <= waited < 2_000_000_000
    wl = W.Workload("afterwait", 1, 2, 800, 2, 2, 32, 96, 3, 0.9, 99)
    r = Runner(wl)
    try:
        for s in range(r.steps):
            r.append(wl.n_new)
            r.compare(r.step(s))
        assert r.kv.stats()["timeouts"] == 0
    finally:
        r.close()


def test_wait_selftest_arguments():
    assert K.kvo_wait_selftest(0, 10)[0] == K.KVO_EINVAL
    assert K.kvo_wait_selftest(0, 20_000_000_000)[0] == K.KVO_EINVAL
