"""ctypes wrapper of the CPU oracle (kvo_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the library path never does.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

OK = 0
EINVAL = -1
ENOMEM = -2
ERANGE = -3
ECAPACITY = -6
PAD_PAYLOAD = -(2 ** 31)
DIM = 128

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvo_oracle.c")
_SO = os.path.join(_HERE, "libkvo_oracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src, out):
    """Compile an oracle source with plain gcc: no fast-math, no FP contraction."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)


def build(force=False):
    """Compile kvo_oracle.c into libkvo_oracle.so unless it is up to date."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + ".tmp%d" % os.getpid()
    compile_source(_SRC, tmp)
    os.replace(tmp, _SO)
    return _SO


def lib():
    """The oracle library, built on first use.

    KVO_ORACLE_LIB, when set, names an already compiled copy to load instead: the
    mutation test uses it to run the pins against copies with a planted mistake.
    """
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("KVO_ORACLE_LIB")
            if not path:
                path = build()
            L = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.oracle_unit_new.restype = vp
            L.oracle_unit_new.argtypes = [i64, i32, i32, i32, i32, i32, i32]
            L.oracle_unit_new2.restype = vp
            L.oracle_unit_new2.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32]
            u16, f32 = ctypes.c_uint16, ctypes.c_float
            L.oracle_f32_to_f16.restype = u16
            L.oracle_f32_to_f16.argtypes = [f32]
            L.oracle_f16_to_f32.restype = f32
            L.oracle_f16_to_f32.argtypes = [u16]
            L.oracle_fwht128.restype = None
            L.oracle_fwht128.argtypes = [vp, vp]
            L.oracle_quant_rotated.restype = None
            L.oracle_quant_rotated.argtypes = [vp, vp, vp]
            L.oracle_quant128.restype = None
            L.oracle_quant128.argtypes = [vp, vp, vp]
            L.oracle_score_i8.restype = f32
            L.oracle_score_i8.argtypes = [vp, u16, vp, u16]
            L.oracle_unit_free.restype = None
            L.oracle_unit_free.argtypes = [vp]
            L.oracle_append.restype = i32
            L.oracle_append.argtypes = [vp, i32, vp, vp]
            L.oracle_step.restype = i32
            L.oracle_step.argtypes = [vp] + [vp] * 9
            L.oracle_step_many.restype = i32
            L.oracle_step_many.argtypes = [vp, i32] + [vp] * 9
            L.oracle_score.restype = ctypes.c_float
            L.oracle_score.argtypes = [vp, vp]
            L.oracle_scores.restype = None
            L.oracle_scores.argtypes = [vp, vp, i64, vp]
            L.oracle_threads.restype = i32
            L.oracle_threads.argtypes = []
            f64 = ctypes.c_double
            L.oracle_attend_rows.restype = None
            L.oracle_attend_rows.argtypes = [vp, i32, i64, vp, i32, vp, i32, f64, vp, vp]
            L.oracle_attend.restype = i32
            L.oracle_attend.argtypes = [vp, vp, i32, vp, i32, f64, vp, vp]
            L.oracle_len.restype = i64
            L.oracle_len.argtypes = [vp]
            L.oracle_stamp.restype = ctypes.c_uint32
            L.oracle_stamp.argtypes = [vp]
            for name in ("oracle_cache_slots", "oracle_slot_token", "oracle_last_use",
                         "oracle_hot", "oracle_rows", "oracle_keys", "oracle_kcode",
                         "oracle_kscale"):
                getattr(L, name).restype = vp
                getattr(L, name).argtypes = [vp]
            _lib = L
    return _lib


def score(q, k):
    """Canonical fp32 score of one 128-element bf16 query/key pair (uint16 arrays)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    assert q.size == DIM and k.size == DIM
    return np.float32(lib().oracle_score(q.ctypes.data, k.ctypes.data))


# ---- int8 indexer (reading R12 of kvo_oracle.c) ------------------------------
def f32_to_f16(x):
    """fp16 bits (uint16) of an fp32 value, round to nearest even."""
    return int(lib().oracle_f32_to_f16(float(np.float32(x))))


def f16_to_f32(h):
    return np.float32(lib().oracle_f16_to_f32(int(h)))


def fwht128(x):
    """Unnormalised 128-point Walsh-Hadamard transform in fp32 (fixed stage order)."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(DIM)
    out = np.empty(DIM, np.float32)
    lib().oracle_fwht128(x.ctypes.data, out.ctypes.data)
    return out


def quant_rotated(y):
    """int8 codes and fp16 scale bits of an already rotated fp32 vector."""
    y = np.ascontiguousarray(y, dtype=np.float32).reshape(DIM)
    code = np.empty(DIM, np.int8)
    sc = np.zeros(1, np.uint16)
    lib().oracle_quant_rotated(y.ctypes.data, code.ctypes.data, sc.ctypes.data)
    return code, int(sc[0])


def quant128(x):
    """Rotate and quantize one bf16 vector (uint16[128]): (int8 codes, fp16 scale bits)."""
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(DIM)
    code = np.empty(DIM, np.int8)
    sc = np.zeros(1, np.uint16)
    lib().oracle_quant128(x.ctypes.data, code.ctypes.data, sc.ctypes.data)
    return code, int(sc[0])


def score_i8(qcode, qscale, kcode, kscale):
    q = np.ascontiguousarray(qcode, dtype=np.int8)
    k = np.ascontiguousarray(kcode, dtype=np.int8)
    return np.float32(lib().oracle_score_i8(q.ctypes.data, int(qscale), k.ctypes.data, int(kscale)))


class StepResult:
    __slots__ = ("tok", "score", "pay", "slot", "status", "miss_tok", "miss_slot", "n_miss")

    def misses(self):
        return list(zip(self.miss_tok[: self.n_miss].tolist(), self.miss_slot[: self.n_miss].tolist()))


class OracleUnit:
    """One (request, layer) unit: host rows, indexer keys, hot shelf, LRU table."""

    def __init__(self, max_tokens, topk, capacity, n_pos, row_elems=576, keep_rows=True,
                 idx_int8=False):
        self.L = lib()
        self.max_tokens, self.topk, self.capacity, self.n_pos = max_tokens, topk, capacity, n_pos
        self.row_elems, self.keep_rows, self.idx_int8 = row_elems, keep_rows, idx_int8
        self.h = self.L.oracle_unit_new2(max_tokens, DIM, row_elems, topk, capacity, n_pos,
                                         1 if keep_rows else 0, 1 if idx_int8 else 0)
        if not self.h:
            raise MemoryError("oracle_unit_new failed")

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.L.oracle_unit_free(h)
            self.h = None

    def append(self, keys, rows=None):
        keys = np.ascontiguousarray(keys, dtype=np.uint16).reshape(-1, DIM)
        n = keys.shape[0]
        rp = None
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.uint16).reshape(n, self.row_elems)
            rp = rows.ctypes.data
        return self.L.oracle_append(self.h, n, rp, keys.ctypes.data)

    def step(self, queries):
        q = np.ascontiguousarray(queries, dtype=np.uint16).reshape(self.n_pos, DIM)
        P, K = self.n_pos, self.topk
        r = StepResult()
        r.tok = np.empty((P, K), np.int32)
        r.score = np.empty((P, K), np.float32)
        r.pay = np.empty((P, K), np.int32)
        r.slot = np.empty((P, K), np.int32)
        st = np.zeros(1, np.int32)
        r.miss_tok = np.full(P * K, -1, np.int32)
        r.miss_slot = np.full(P * K, -1, np.int32)
        nm = np.zeros(1, np.int32)
        rc = self.L.oracle_step(self.h, q.ctypes.data, r.tok.ctypes.data, r.score.ctypes.data,
                                r.pay.ctypes.data, r.slot.ctypes.data, st.ctypes.data,
                                r.miss_tok.ctypes.data, r.miss_slot.ctypes.data, nm.ctypes.data)
        if rc != OK:
            raise RuntimeError("oracle_step failed: %d" % rc)
        r.status = int(st[0])
        r.n_miss = int(nm[0])
        return r

    def scores(self, query, n=None):
        n = self.length if n is None else n
        q = np.ascontiguousarray(query, dtype=np.uint16).reshape(DIM)
        out = np.empty(n, np.float32)
        self.L.oracle_scores(self.h, q.ctypes.data, n, out.ctypes.data)
        return out

    def _view(self, fn, n, dtype):
        p = getattr(self.L, fn)(self.h)
        if not p or n == 0:
            return np.empty(0, dtype)
        buf = (ctypes.c_char * (n * np.dtype(dtype).itemsize)).from_address(p)
        return np.frombuffer(buf, dtype=dtype, count=n).copy()

    @property
    def length(self):
        return int(self.L.oracle_len(self.h))

    @property
    def stamp(self):
        return int(self.L.oracle_stamp(self.h))

    def cache_slots(self):
        return self._view("oracle_cache_slots", self.max_tokens, np.int32)

    def slot_token(self):
        return self._view("oracle_slot_token", self.capacity, np.int32)

    def last_use(self):
        return self._view("oracle_last_use", self.capacity, np.uint32)

    def hot(self):
        assert self.keep_rows
        return self._view("oracle_hot", self.capacity * self.row_elems, np.uint16).reshape(
            self.capacity, self.row_elems)

    def key_codes(self):
        """int8 codes and fp16 scale bits of the cached keys (int8 indexer)."""
        assert self.idx_int8
        n = self.length
        return (self._view("oracle_kcode", n * DIM, np.int8).reshape(n, DIM),
                self._view("oracle_kscale", n, np.uint16))

    def rows(self):
        assert self.keep_rows
        return self._view("oracle_rows", self.max_tokens * self.row_elems, np.uint16).reshape(
            self.max_tokens, self.row_elems)

    def attend(self, tokens, queries, scale):
        """R13 attention of one position: tokens [k] int32 (< 0 = pad), queries [H][576]
        bf16 bits.  Returns (out [H][512] float64, lse [H] float64)."""
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        queries = np.ascontiguousarray(queries, dtype=np.uint16)
        H = queries.shape[0]
        out = np.zeros((H, 512), dtype=np.float64)
        lse = np.zeros(H, dtype=np.float64)
        rc = lib().oracle_attend(self.h, tokens.ctypes.data, len(tokens), queries.ctypes.data, H,
                                 float(scale), out.ctypes.data, lse.ctypes.data)
        assert rc == OK, rc
        return out, lse


def step_many(units, queries):
    """One step of many units in parallel (OpenMP).  queries: [n][P][128] uint16."""
    L = lib()
    n = len(units)
    P, K = units[0].n_pos, units[0].topk
    q = np.ascontiguousarray(queries, dtype=np.uint16).reshape(n, P, DIM)
    hs = (ctypes.c_void_p * n)(*[u.h for u in units])
    tok = np.empty((n, P, K), np.int32)
    sc = np.empty((n, P, K), np.float32)
    pay = np.empty((n, P, K), np.int32)
    sl = np.empty((n, P, K), np.int32)
    st = np.zeros(n, np.int32)
    mt = np.empty((n, P * K), np.int32)
    ms = np.empty((n, P * K), np.int32)
    nm = np.zeros(n, np.int32)
    rc = L.oracle_step_many(hs, n, q.ctypes.data, tok.ctypes.data, sc.ctypes.data,
                            pay.ctypes.data, sl.ctypes.data, st.ctypes.data, mt.ctypes.data,
                            ms.ctypes.data, nm.ctypes.data)
    if rc != OK:
        raise RuntimeError("oracle_step_many failed: %d" % rc)
    return tok, sc, pay, sl, st, nm


def attend_rows(rows, tokens, queries, scale):
    """R13 attention over explicit rows: rows [n][>=576] bf16 bits, tokens [k] int32
    (< 0 = pad), queries [H][576] bf16 bits.  Returns (out [H][512], lse [H]) in float64."""
    rows = np.ascontiguousarray(rows, dtype=np.uint16)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    queries = np.ascontiguousarray(queries, dtype=np.uint16)
    H = queries.shape[0]
    out = np.zeros((H, 512), dtype=np.float64)
    lse = np.zeros(H, dtype=np.float64)
    lib().oracle_attend_rows(rows.ctypes.data, rows.shape[1], rows.shape[0], tokens.ctypes.data,
                             len(tokens), queries.ctypes.data, H, float(scale), out.ctypes.data,
                             lse.ctypes.data)
    return out, lse


def threads():
    return int(lib().oracle_threads())
