"""An allocation failure is reported and leaves the device and the thread clean.

The out-of-memory condition is a real request, not a hook: hot buffers that cannot fit
in HBM (128 units x 2^20 slots x 4096 bf16 elements, 1.1 TB).  cudaMalloc refuses such a
request at once without touching memory, so nothing faults.  kvo_create must return
KVO_ENOMEM with a message and free what it had allocated.  A failed cudaMalloc is also
recorded as the thread's last CUDA error; the library must not leave it there, or the
caller's next launch check (PyTorch's, or this library's) would report it as its own.
So a PyTorch kernel and a decode sequence run right after, the decode still matching the
oracle bit for bit.
"""
import pytest
import torch

import workload as W
from tests.gpu_harness import Runner
from top_cache_gb300 import kvo as K

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from top_cache_gb300 import build
    build.build()
    yield


def test_device_allocation_failure_is_reported_and_cleared():
    torch.cuda.synchronize()
    with pytest.raises(K.KvoError) as err:
        K.kvo_create(128, 1, 8, 1, 1 << 20, 1, 4096, 128, 0, K.KVO_IDX_BF16, 0, 0)
    assert err.value.code == K.KVO_ENOMEM
    assert "device allocation" in str(err.value)
    # the thread's CUDA error state is clean: PyTorch launches and checks a kernel
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2
    torch.cuda.synchronize()
    # and the library still creates handles and runs decode steps that match the oracle
    wl = W.Workload("after_enomem", 1, 2, 700, 2, 2, 32, 96, 3, 0.9, 77)
    r = Runner(wl)
    try:
        for s in range(r.steps):
            r.append(wl.n_new)
            r.compare(r.step(s))
    finally:
        r.close()
