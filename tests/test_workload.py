"""The seeded generator matches its documented definition and distribution."""
import math
import struct

import numpy as np

import workload as W

M64 = (1 << 64) - 1


def _mix(z):
    z &= M64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & M64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & M64
    z ^= z >> 31
    return z


def _key(seed, kind, r, l, sub):
    h = _mix(seed ^ (kind << 56))
    h = _mix(h + r)
    h = _mix(h + l)
    return _mix(h + sub)


def _uniform(key, j):
    x = _mix(key + (j + 1) * 0x9E3779B97F4A7C15)
    return ((x >> 11) + 0.5) * 2.0 ** -53


def _normal(key, j):
    i = j >> 1
    rad = math.sqrt(-2.0 * math.log(_uniform(key, 2 * i)))
    th = 2.0 * math.pi * _uniform(key, 2 * i + 1)
    return rad * (math.sin(th) if j & 1 else math.cos(th))


def _bf16(v):
    b = struct.unpack("<I", struct.pack("<f", v))[0]
    b += 0x7FFF + ((b >> 16) & 1)
    return (b >> 16) & 0xFFFF


def test_stream_matches_definition():
    for (seed, kind, r, l, sub, j0) in [(1001, 1, 0, 0, 0, 0), (1002, 2, 15, 7, 0, 12345),
                                        (7, 3, 3, 1, 2, 1)]:
        key = _key(seed, kind, r, l, sub)
        assert W.lib().gen_stream_key(seed, kind, r, l, sub) == key
        got = W.normal_f64(seed, kind, r, l, sub, j0, 64)
        ref = np.array([_normal(key, j0 + j) for j in range(64)])
        assert np.allclose(got, ref, rtol=0, atol=1e-12)
        gb = W.normal_bf16(seed, kind, r, l, sub, j0, 64)
        refb = [_bf16(float(np.float32(v))) for v in ref]
        assert gb.tolist() == refb


def test_token_rows_index_layout():
    units = [(0, 0), (2, 3)]
    rows = W.token_rows(1002, W.KIND_ROWS, units, 10, 3, 576)
    for i, (r, l) in enumerate(units):
        flat = W.normal_bf16(1002, W.KIND_ROWS, r, l, 0, 10 * 576, 3 * 576)
        assert np.array_equal(rows[i].reshape(-1), flat)


def test_query_walk_recursion():
    a, n = 0.9, 6
    w = W.query_walk(1002, 1, 2, 0, a, n)
    ki = _key(1002, W.KIND_QINIT, 1, 2, 0)
    kn = _key(1002, W.KIND_QNOISE, 1, 2, 0)
    q = [_normal(ki, d) for d in range(128)]
    c = math.sqrt(1 - a * a)
    for s in range(n):
        assert w[s].tolist() == [_bf16(float(np.float32(x))) for x in q]
        q = [a * q[d] + c * _normal(kn, s * 128 + d) for d in range(128)]


def test_normal_moments():
    x = W.normal_f64(99, 1, 0, 0, 0, 0, 1 << 18)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1) < 0.01
    assert abs(np.mean(x ** 3)) < 0.03 and abs(np.mean(x ** 4) - 3) < 0.06


def test_frozen_walk_and_fresh_walk():
    w1 = W.query_walk(5, 0, 0, 0, 1.0, 4)
    assert all(np.array_equal(w1[0], w1[s]) for s in range(4))
    w0 = W.query_walk(5, 0, 0, 0, 0.0, 64)
    f = W.bf16_to_f32(w0).astype(np.float64)
    c = np.corrcoef(f[:-1].ravel(), f[1:].ravel())[0, 1]
    assert abs(c) < 0.05
