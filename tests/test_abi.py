"""The C-ABI library builds, loads and exports every entry point include/kvo.h declares.

No compute call is made here (no GPU needed): only argument validation that
happens before any device is touched.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvo.h")


@pytest.fixture(scope="module")
def L():
    from top_cache_gb300 import build, kvo
    build.build()
    return kvo.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kvo_\w+)\s*\(", src, flags=re.M))


def test_header_declares_the_boundary():
    d = _declared()
    for name in ("kvo_create", "kvo_destroy", "kvo_append", "kvo_step"):
        assert name in d


def test_every_declared_symbol_is_exported(L):
    from top_cache_gb300 import kvo
    d = _declared()
    for name in d:
        assert hasattr(L, name), name  # dlsym succeeds
    assert set(kvo.EXPORTED) == d


def test_invalid_config_rejected_before_device(L):
    from top_cache_gb300 import kvo
    bad = [
        dict(idx_dim=64),
        dict(row_elems=570),
        dict(topk=0),
        dict(hot_capacity=10),          # < topk
        dict(n_positions=9),
        dict(max_tokens=0),
        dict(n_requests=0),
        dict(topk=4000, hot_capacity=8192, n_positions=8),  # candidate buffer too small
        dict(idx_dtype=2),
    ]
    for over in bad:
        cfg = dict(n_requests=1, n_layers=1, max_tokens=100, idx_dim=128, row_elems=576,
                   topk=16, hot_capacity=32, n_positions=1, device=0, idx_dtype=0)
        cfg.update(over)
        c = kvo.KvoConfig(cfg["n_requests"], cfg["n_layers"], cfg["max_tokens"], cfg["idx_dim"],
                          cfg["row_elems"], cfg["topk"], cfg["hot_capacity"], cfg["n_positions"],
                          cfg["device"], cfg["idx_dtype"])
        h = ctypes.c_void_p()
        rc = L.kvo_create(ctypes.byref(c), ctypes.byref(h))
        assert rc == kvo.KVO_EINVAL, over
        assert h.value is None
        assert len(L.kvo_last_error()) > 0


def test_null_handles(L):
    from top_cache_gb300 import kvo
    assert L.kvo_destroy(None) == kvo.KVO_OK
    assert L.kvo_host_rows(None, 0) is None
    assert L.kvo_step(None, None, 1, None, None, None, None, None, None, None) == kvo.KVO_EINVAL
    assert L.kvo_append(None, None, 1, 1, None, None, None) == kvo.KVO_EINVAL
    assert L.kvo_set_option(None, 1, 0) == kvo.KVO_EINVAL
    assert L.kvo_get_option(None, 1, None) == kvo.KVO_EINVAL


def test_header_constants_match_binding():
    from top_cache_gb300 import kvo
    src = open(HEADER).read()
    defs = dict((m.group(1), int(m.group(2)))
                for m in re.finditer(r"^#define\s+(KVO_\w+)\s+(-?\d+)", src, flags=re.M))
    for name, value in defs.items():
        if name.startswith("KVO_PROF_") and name != "KVO_PROF_KINDS":
            assert kvo.PROF_KINDS[value] == name[len("KVO_PROF_"):].lower(), name
        elif name == "KVO_PROF_KINDS":
            assert len(kvo.PROF_KINDS) == value
        else:
            assert getattr(kvo, name) == value, name


def test_binding_refuses_strided_buffers():
    # argument marshalling only, but it must not hand a strided view to the C ABI as dense
    import numpy as np
    import torch
    from top_cache_gb300 import kvo
    a = np.zeros((4, 8), np.int32)
    assert kvo._ptr(a) == a.ctypes.data
    assert kvo._ptr(a[1:3]) == a[1:3].ctypes.data  # leading-dimension slices stay dense
    with pytest.raises(kvo.KvoError) as e:
        kvo._ptr(a[:, :4])
    assert e.value.code == kvo.KVO_EINVAL
    t = torch.zeros((4, 8), dtype=torch.int32)
    assert kvo._ptr(t[2:]) == t[2:].data_ptr()
    for bad in (t[:, 1:], t.t()):
        with pytest.raises(kvo.KvoError):
            kvo._ptr(bad)
    assert kvo._ptr(None) is None and kvo._ptr(1234) == 1234
