"""ctypes wrapper around gen.c (the seeded generator).  No method arithmetic here."""
import ctypes
import os
import subprocess
import threading

import numpy as np

KIND_KEYS = 1
KIND_ROWS = 2
KIND_QINIT = 3
KIND_QNOISE = 4
KIND_ATTN_Q = 5  # attention queries (one 576-element row per position and head)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_SO = os.path.join(_HERE, "libkvogen.so")
_lock = threading.Lock()
_lib = None


def build(force=False):
    """Compile gen.c into libkvogen.so next to it (plain gcc, OpenMP)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            u64, i32, i64, dbl = ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            L.gen_stream_key.restype = u64
            L.gen_stream_key.argtypes = [u64, i32, i64, i64, i64]
            L.gen_normal_bf16.restype = None
            L.gen_normal_bf16.argtypes = [u64, i32, i64, i64, i64, i64, i64, vp]
            L.gen_normal_f64.restype = None
            L.gen_normal_f64.argtypes = [u64, i32, i64, i64, i64, i64, i64, vp]
            L.gen_token_rows_bf16.restype = None
            L.gen_token_rows_bf16.argtypes = [u64, i32, i32, vp, vp, i64, i64, i32, i64, vp]
            L.gen_query_walk.restype = None
            L.gen_query_walk.argtypes = [u64, i32, i32, i64, i64, i64, dbl, i32, i32, vp]
            L.gen_f32_to_bf16.restype = ctypes.c_uint16
            L.gen_f32_to_bf16.argtypes = [ctypes.c_float]
            _lib = L
    return _lib


def normal_bf16(seed, kind, r, l, sub, j0, n):
    out = np.empty(n, dtype=np.uint16)
    lib().gen_normal_bf16(seed, kind, r, l, sub, j0, n, out.ctypes.data)
    return out


def normal_f64(seed, kind, r, l, sub, j0, n):
    out = np.empty(n, dtype=np.float64)
    lib().gen_normal_f64(seed, kind, r, l, sub, j0, n, out.ctypes.data)
    return out


def _rl(units_rl):
    rs = np.ascontiguousarray([u[0] for u in units_rl], dtype=np.int64)
    ls = np.ascontiguousarray([u[1] for u in units_rl], dtype=np.int64)
    return rs, ls


def token_rows(seed, kind, units_rl, t0, n_tok, width):
    """bf16 (as uint16) array [n_units][n_tok][width] of token rows t0..t0+n_tok-1."""
    rs, ls = _rl(units_rl)
    out = np.empty((len(units_rl), n_tok, width), dtype=np.uint16)
    if out.size:
        lib().gen_token_rows_bf16(seed, kind, len(units_rl), rs.ctypes.data, ls.ctypes.data,
                                  t0, n_tok, width, n_tok * width, out.ctypes.data)
    return out


def token_rows_into(ptr, unit_stride_elems, seed, kind, units_rl, t0, n_tok, width):
    """Write token rows straight into caller memory at integer address ptr."""
    rs, ls = _rl(units_rl)
    lib().gen_token_rows_bf16(seed, kind, len(units_rl), rs.ctypes.data, ls.ctypes.data,
                              t0, n_tok, width, unit_stride_elems, ctypes.c_void_p(ptr))


def query_walk(seed, r, l, sub, a, n_steps, dim=128):
    """bf16 (uint16) [n_steps][dim]: step s holds bf16(q_s) of the fp64 random walk."""
    out = np.empty((n_steps, dim), dtype=np.uint16)
    lib().gen_query_walk(seed, KIND_QINIT, KIND_QNOISE, r, l, sub, float(a), n_steps, dim,
                         out.ctypes.data)
    return out


def unit_queries(seed, units_rl, a, n_steps, n_pos, distinct=False, dim=128):
    """[n_steps][n_units][n_pos][dim] uint16.

    distinct=False: one walk per unit shared by all positions (sub = 0);
    distinct=True: an independent walk per position (sub = position)."""
    out = np.empty((n_steps, len(units_rl), n_pos, dim), dtype=np.uint16)
    for i, (r, l) in enumerate(units_rl):
        if distinct:
            for p in range(n_pos):
                out[:, i, p, :] = query_walk(seed, r, l, p, a, n_steps, dim)
        else:
            w = query_walk(seed, r, l, 0, a, n_steps, dim)
            out[:, i, :, :] = w[:, None, :]
    return out


def attention_queries(seed, units_rl, step, n_pos, n_heads, width=576):
    """bf16 (uint16) [n_units][n_pos][n_heads][width] attention queries of one decode step,
    N(0,1): rows step*n_pos*n_heads .. of the KIND_ATTN_Q stream of each unit."""
    q = token_rows(seed, KIND_ATTN_Q, units_rl, step * n_pos * n_heads, n_pos * n_heads, width)
    return q.reshape(len(units_rl), n_pos, n_heads, width)


def bf16_to_f32(a):
    """Exact bf16 (uint16 bit pattern) -> float32."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_np(x):
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)
