"""Python binding of libkvo (the C ABI declared in include/kvo.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of libkvo.so.  PyTorch is used for device memory and streams.  There
is no CPU fallback: if the library is missing or cannot be loaded, every call
raises.
"""
import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libkvo.so")

KVO_OK = 0
KVO_EINVAL = -1
KVO_ENOMEM = -2
KVO_ERANGE = -3
KVO_ECUDA = -4
KVO_ETIMEOUT = -5
KVO_ECAPACITY = -6
KVO_PAD_PAYLOAD = -(2 ** 31)
KVO_SELECT_ERR_TIMEOUT = 1  # bits of the select calls' status word
KVO_SELECT_ERR_PLAN = 2

KVO_OPT_GATHER_MODE = 1
KVO_OPT_WAIT_LIMIT_NS = 2
KVO_OPT_PROFILE = 3
KVO_OPT_GROUPS = 4
KVO_OPT_SCORE_CTAS = 5
KVO_OPT_SPECULATE = 6
KVO_OPT_FUSED = 7
KVO_OPT_GATHER_CTAS = 8
KVO_OPT_PIECE_TOKENS = 9
KVO_OPT_HOST_HUGE_PAGE = 10
KVO_OPT_DEFER_FILL = 11
KVO_OPT_GROUP_GATHER_SMS = 12
KVO_OPT_PROFILE_KINDS = 13
PROF_KINDS = ("append", "plan", "score", "select", "residency", "gather", "reset", "rescore",
              "reselect", "fused", "attend")
KVO_IDX_BF16 = 0
KVO_IDX_INT8 = 1
KVO_GATHER_LDG = 0
KVO_GATHER_BULK = 1

EXPORTED = ("kvo_create", "kvo_destroy", "kvo_host_rows", "kvo_prefill", "kvo_append", "kvo_step",
            "kvo_select_workspace_size", "kvo_select", "kvo_reset", "kvo_profile_read",
            "kvo_set_option", "kvo_get_option", "kvo_get_stats", "kvo_export_state", "kvo_select_noalloc",
            "kvo_attend", "kvo_set_blocks", "kvo_host_block", "kvo_wait_selftest", "kvo_lw_create", "kvo_lw_destroy", "kvo_lw_plan", "kvo_lw_host_rows",
            "kvo_lw_set_length", "kvo_lw_begin", "kvo_lw_layer", "kvo_lw_layer_done", "kvo_lw_end",
            "kvo_lw_stats", "kvo_last_error")


class KvoConfig(ctypes.Structure):
    _fields_ = [("n_requests", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("max_tokens", ctypes.c_int64), ("idx_dim", ctypes.c_int32),
                ("row_elems", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("hot_capacity", ctypes.c_int32), ("n_positions", ctypes.c_int32),
                ("device", ctypes.c_int32), ("idx_dtype", ctypes.c_int32),
                ("host_block_tokens", ctypes.c_int32), ("host_blocks", ctypes.c_int64)]


class KvoLwConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_independent", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("lookahead", ctypes.c_int32),
                ("max_tokens", ctypes.c_int64), ("row_elems", ctypes.c_int32),
                ("device", ctypes.c_int32)]


class KvoStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("steps", "unit_steps", "capacity_errors", "hits", "misses", "rows_h2d",
                 "bytes_h2d", "rows_d2h", "bytes_d2h", "timeouts", "rescored", "fused_steps",
                 "block_errors", "fetch_dup_bytes", "split_steps", "launches", "rows_h2d_in_score")]


class KvoError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("kvo error %d: %s" % (code, msg))
        self.code = code


_lock = threading.Lock()
_lib = None


def library_path():
    return _SO


def lib():
    """Load libkvo.so (built by top_cache_gb300.build / __graft_entry__.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_SO):
                raise ImportError("libkvo.so is not built (run top_cache_gb300.build.build()); "
                                  "there is no fallback path")
            L = ctypes.CDLL(_SO)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.kvo_create.restype = ctypes.c_int
            L.kvo_create.argtypes = [ctypes.POINTER(KvoConfig), ctypes.POINTER(vp)]
            L.kvo_destroy.restype = ctypes.c_int
            L.kvo_destroy.argtypes = [vp]
            L.kvo_host_rows.restype = vp
            L.kvo_host_rows.argtypes = [vp, i32]
            L.kvo_prefill.restype = ctypes.c_int
            L.kvo_prefill.argtypes = [vp, i32, i64, vp, vp]
            L.kvo_append.restype = ctypes.c_int
            L.kvo_append.argtypes = [vp, vp, i32, i32, vp, vp, vp]
            L.kvo_step.restype = ctypes.c_int
            L.kvo_step.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
            L.kvo_select_workspace_size.restype = ctypes.c_size_t
            L.kvo_select_workspace_size.argtypes = [i32, i32, i32, i32]
            L.kvo_select.restype = ctypes.c_int
            L.kvo_select.argtypes = [vp, i64, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp,
                                     ctypes.c_size_t, vp, vp]
            L.kvo_select_noalloc.restype = ctypes.c_int
            L.kvo_select_noalloc.argtypes = [vp, i64, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
            L.kvo_attend.restype = ctypes.c_int
            L.kvo_attend.argtypes = [vp, vp, i32, vp, i32, ctypes.c_float, vp, vp, vp, vp]
            L.kvo_reset.restype = ctypes.c_int
            L.kvo_reset.argtypes = [vp, vp, i32, i64, vp]
            L.kvo_profile_read.restype = ctypes.c_int
            L.kvo_profile_read.argtypes = [vp, vp, vp, i32]
            L.kvo_set_option.restype = ctypes.c_int
            L.kvo_set_option.argtypes = [vp, i32, i64]
            L.kvo_get_option.restype = ctypes.c_int
            L.kvo_get_option.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64)]
            L.kvo_get_stats.restype = ctypes.c_int
            L.kvo_get_stats.argtypes = [vp, ctypes.POINTER(KvoStats)]
            L.kvo_export_state.restype = ctypes.c_int
            L.kvo_export_state.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
            L.kvo_last_error.restype = ctypes.c_char_p
            L.kvo_last_error.argtypes = []
            L.kvo_wait_selftest.restype = ctypes.c_int
            L.kvo_wait_selftest.argtypes = [i32, i64, ctypes.POINTER(ctypes.c_int64)]
            L.kvo_set_blocks.restype = ctypes.c_int
            L.kvo_set_blocks.argtypes = [vp, i32, i32, i32, vp, vp]
            L.kvo_host_block.restype = vp
            L.kvo_host_block.argtypes = [vp, i64]
            L.kvo_lw_create.restype = ctypes.c_int
            L.kvo_lw_create.argtypes = [ctypes.POINTER(KvoLwConfig), ctypes.POINTER(vp)]
            L.kvo_lw_destroy.restype = ctypes.c_int
            L.kvo_lw_destroy.argtypes = [vp]
            L.kvo_lw_plan.restype = ctypes.c_int
            L.kvo_lw_plan.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
            L.kvo_lw_host_rows.restype = vp
            L.kvo_lw_host_rows.argtypes = [vp, i32]
            L.kvo_lw_set_length.restype = ctypes.c_int
            L.kvo_lw_set_length.argtypes = [vp, i64]
            L.kvo_lw_begin.restype = ctypes.c_int
            L.kvo_lw_begin.argtypes = [vp, i64, vp]
            L.kvo_lw_layer.restype = ctypes.c_int
            L.kvo_lw_layer.argtypes = [vp, i32, ctypes.POINTER(vp), vp]
            L.kvo_lw_layer_done.restype = ctypes.c_int
            L.kvo_lw_layer_done.argtypes = [vp, i32, vp]
            L.kvo_lw_end.restype = ctypes.c_int
            L.kvo_lw_end.argtypes = [vp, vp]
            L.kvo_lw_stats.restype = ctypes.c_int
            L.kvo_lw_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]
            _lib = L
    return _lib


def _check(rc):
    if rc != KVO_OK:
        raise KvoError(rc, lib().kvo_last_error().decode())
    return rc


def _ptr(t):
    """Device/host address of a tensor or array, or None.

    The C ABI takes dense row-major buffers, so a strided view (a slice along an
    inner dimension, a transpose) is refused here rather than read as if dense.
    """
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        if not t.flags.c_contiguous:
            raise KvoError(KVO_EINVAL, "array is not C-contiguous")
        return t.ctypes.data
    if not t.is_contiguous():
        raise KvoError(KVO_EINVAL, "tensor is not contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _units(units):
    if units is None:
        return None, None
    arr = np.ascontiguousarray(units, dtype=np.int32)
    return arr, arr.ctypes.data


def kvo_create(n_requests, n_layers, max_tokens, topk, hot_capacity, n_positions=1,
               row_elems=576, idx_dim=128, device=0, idx_dtype=KVO_IDX_BF16, host_block_tokens=0,
               host_blocks=0):
    cfg = KvoConfig(n_requests, n_layers, max_tokens, idx_dim, row_elems, topk, hot_capacity,
                    n_positions, device, idx_dtype, host_block_tokens, host_blocks)
    h = ctypes.c_void_p()
    _check(lib().kvo_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def kvo_destroy(h):
    return _check(lib().kvo_destroy(h))


def kvo_host_rows(h, unit):
    """Integer host address of unit's row 0 in the pinned host pool."""
    p = lib().kvo_host_rows(h, unit)
    if not p:
        raise KvoError(KVO_ERANGE, "unit out of range")
    return p


def kvo_prefill(h, unit, n_tokens, idx_keys, stream=None):
    return _check(lib().kvo_prefill(h, unit, n_tokens, _ptr(idx_keys), _stream(stream)))


def kvo_append(h, units, n_units, n_tokens, main_rows, idx_keys, stream=None):
    arr, up = _units(units)
    return _check(lib().kvo_append(h, up, n_units, n_tokens, _ptr(main_rows), _ptr(idx_keys),
                                   _stream(stream)))


def kvo_step(h, units, n_units, queries, topk_tokens, topk_slots, topk_scores, topk_payload,
             unit_status, stream=None):
    arr, up = _units(units)
    return _check(lib().kvo_step(h, up, n_units, _ptr(queries), _ptr(topk_tokens),
                                 _ptr(topk_slots), _ptr(topk_scores), _ptr(topk_payload),
                                 _ptr(unit_status), _stream(stream)))


def kvo_attend(h, units, n_units, queries, n_heads, scale, topk_slots, out, lse=None, stream=None):
    arr, up = _units(units)
    return _check(lib().kvo_attend(h, up, n_units, _ptr(queries), n_heads, float(scale),
                                   _ptr(topk_slots), _ptr(out), _ptr(lse), _stream(stream)))


def kvo_select_workspace_size(n_units, n_pos, k, device=0):
    return int(lib().kvo_select_workspace_size(n_units, n_pos, k, device))


def kvo_select(keys, unit_stride, cache_slots, lengths, n_units, n_pos, k, queries, tokens,
               scores, payload, workspace, workspace_bytes, stream=None, status=None):
    ln = np.ascontiguousarray(lengths, dtype=np.int64)
    return _check(lib().kvo_select(_ptr(keys), unit_stride, _ptr(cache_slots), ln.ctypes.data,
                                   n_units, n_pos, k, _ptr(queries), _ptr(tokens), _ptr(scores),
                                   _ptr(payload), _ptr(workspace), workspace_bytes, _ptr(status),
                                   _stream(stream)))


def kvo_select_noalloc(keys, unit_stride, cache_slots, lengths, n_units, n_pos, k, queries,
                       tokens, scores, payload, stream=None, status=None):
    """kvo_select without a workspace (fixed scratch inside the library; allocates nothing).
    status: optional device uint32 tensor of one element that receives the kernels'
    completion word (0 = the outputs are valid)."""
    ln = np.ascontiguousarray(lengths, dtype=np.int64)
    return _check(lib().kvo_select_noalloc(_ptr(keys), unit_stride, _ptr(cache_slots),
                                           ln.ctypes.data, n_units, n_pos, k, _ptr(queries),
                                           _ptr(tokens), _ptr(scores), _ptr(payload),
                                           _ptr(status), _stream(stream)))


def kvo_reset(h, units, n_units, keep_tokens, stream=None):
    arr, up = _units(units)
    return _check(lib().kvo_reset(h, up, n_units, keep_tokens, _stream(stream)))


def kvo_profile_read(h):
    """{kind: (ms, launches)} accumulated since the last read (profiling option on)."""
    n = len(PROF_KINDS)
    ms = np.zeros(n, np.float64)
    cnt = np.zeros(n, np.uint64)
    _check(lib().kvo_profile_read(h, ms.ctypes.data, cnt.ctypes.data, n))
    return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(PROF_KINDS)}


def kvo_set_option(h, key, value):
    return _check(lib().kvo_set_option(h, key, value))


def kvo_get_option(h, key):
    v = ctypes.c_int64(0)
    _check(lib().kvo_get_option(h, key, ctypes.byref(v)))
    return v.value


def kvo_get_stats(h):
    s = KvoStats()
    _check(lib().kvo_get_stats(h, ctypes.byref(s)))
    return {n: int(getattr(s, n)) for n, _ in KvoStats._fields_}


def kvo_export_state(h, unit, max_tokens, capacity, row_elems=576, with_rows=False):
    cs = np.empty(max_tokens, np.int32)
    st = np.empty(capacity, np.int32)
    lu = np.empty(capacity, np.uint32)
    ln = ctypes.c_int64()
    sp = ctypes.c_uint32()
    hot = np.empty((capacity, row_elems), np.uint16) if with_rows else None
    _check(lib().kvo_export_state(h, unit, cs.ctypes.data, st.ctypes.data, lu.ctypes.data,
                                  ctypes.addressof(ln), ctypes.addressof(sp),
                                  hot.ctypes.data if with_rows else None))
    return {"cache_slots": cs, "slot_token": st, "last_use": lu, "length": ln.value,
            "stamp": sp.value, "hot": hot}


class Kvo:
    """A handle plus output buffers for all units (plumbing around the C ABI)."""

    def __init__(self, n_requests, n_layers, max_tokens, topk, hot_capacity, n_positions=1,
                 row_elems=576, device=0, idx_dtype=KVO_IDX_BF16, host_block_tokens=0, host_blocks=0):
        import torch
        self.n_requests, self.n_layers = n_requests, n_layers
        self.block_tokens = host_block_tokens
        self.U = n_requests * n_layers
        self.max_tokens, self.topk, self.C = max_tokens, topk, hot_capacity
        self.P, self.R, self.device = n_positions, row_elems, device
        self.idx_dtype = idx_dtype
        self.h = kvo_create(n_requests, n_layers, max_tokens, topk, hot_capacity, n_positions,
                            row_elems, 128, device, idx_dtype, host_block_tokens, host_blocks)
        dev = torch.device("cuda", device)
        shape = (self.U, self.P, self.topk)
        self.tokens = torch.empty(shape, dtype=torch.int32, device=dev)
        self.slots = torch.empty(shape, dtype=torch.int32, device=dev)
        self.scores = torch.empty(shape, dtype=torch.float32, device=dev)
        self.payload = torch.empty(shape, dtype=torch.int32, device=dev)
        self.status = torch.empty(self.U, dtype=torch.int32, device=dev)

    def close(self):
        if self.h:
            kvo_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def host_rows(self, unit):
        return kvo_host_rows(self.h, unit)

    def host_block(self, block):
        """Host address of physical block `block` of a paged pool ([B][row_elems] bf16)."""
        p = lib().kvo_host_block(self.h, block)
        if not p:
            raise KvoError(KVO_EINVAL, lib().kvo_last_error().decode())
        return p

    def set_blocks(self, unit, blocks, first_block=0, stream=None):
        """Entries first_block.. of unit's block table (-1 = unmapped)."""
        arr = np.ascontiguousarray(blocks, dtype=np.int32)
        return _check(lib().kvo_set_blocks(self.h, unit, first_block, len(arr), arr.ctypes.data,
                                           _stream(stream)))

    def prefill(self, unit, n_tokens, idx_keys, stream=None):
        return kvo_prefill(self.h, unit, n_tokens, idx_keys, stream)

    def append(self, main_rows, idx_keys, units=None, stream=None):
        n_units = self.U if units is None else len(units)
        n_tok = int(idx_keys.shape[-2])
        return kvo_append(self.h, units, n_units, n_tok, main_rows, idx_keys, stream)

    def step(self, queries, units=None, stream=None, out=None):
        n = self.U if units is None else len(units)
        if out is None:
            out = (self.tokens[:n], self.slots[:n], self.scores[:n], self.payload[:n],
                   self.status[:n])
        tok, sl, sc, pay, st = out
        kvo_step(self.h, units, n, queries, tok, sl, sc, pay, st, stream)
        return out

    def attend(self, queries, scale, out, lse=None, slots=None, units=None, stream=None):
        """Sparse attention of the last step's lists: queries [n][P][H][576] bf16 device,
        out [n][P][H][512] bf16 device, lse [n][P][H] float32 device or None."""
        n = self.U if units is None else len(units)
        if slots is None:
            slots = self.slots[:n]
        H = int(queries.shape[-2])
        return kvo_attend(self.h, units, n, queries, H, scale, slots, out, lse, stream)

    def reset(self, keep_tokens, units=None, stream=None):
        n_units = self.U if units is None else len(units)
        return kvo_reset(self.h, units, n_units, keep_tokens, stream)

    def profile_read(self):
        return kvo_profile_read(self.h)

    def set_option(self, key, value):
        return kvo_set_option(self.h, key, value)

    def get_option(self, key):
        return kvo_get_option(self.h, key)

    def stats(self):
        return kvo_get_stats(self.h)

    def export_state(self, unit, with_rows=False):
        return kvo_export_state(self.h, unit, self.max_tokens, self.C, self.R, with_rows)


class _DeviceRows:
    """__cuda_array_interface__ view of device rows (no copy), for torch.as_tensor."""

    def __init__(self, ptr, rows, row_elems):
        self.__cuda_array_interface__ = {"shape": (rows, row_elems), "typestr": "<i2",
                                         "data": (int(ptr), False), "version": 3, "strides": None}


class Layerwise:
    """Layerwise prefill offload (kvo_lw_*): host pool of every layer, device buffers by plan."""

    def __init__(self, n_layers, max_tokens, n_independent=1, n_shared=3, lookahead=1,
                 row_elems=576, device=0):
        cfg = KvoLwConfig(n_layers, n_independent, n_shared, lookahead, max_tokens, row_elems, device)
        h = ctypes.c_void_p()
        _check(lib().kvo_lw_create(ctypes.byref(cfg), ctypes.byref(h)))
        self.h = h.value
        self.n_layers, self.max_tokens, self.row_elems, self.device = n_layers, max_tokens, row_elems, device
        n = ctypes.c_int32()
        phys = np.zeros(n_layers, dtype=np.int32)
        _check(lib().kvo_lw_plan(self.h, ctypes.byref(n), phys.ctypes.data))
        self.n_phys, self.phys = int(n.value), phys
        self._views = {}

    def close(self):
        if getattr(self, "h", None):
            lib().kvo_lw_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def host_rows(self, layer):
        """numpy view [max_tokens][row_elems] uint16 of the layer's pinned host rows."""
        ptr = lib().kvo_lw_host_rows(self.h, layer)
        if not ptr:
            raise KvoError(KVO_EINVAL, lib().kvo_last_error().decode())
        n = self.max_tokens * self.row_elems
        return np.ctypeslib.as_array((ctypes.c_uint16 * n).from_address(ptr)).reshape(
            self.max_tokens, self.row_elems)

    def host_rows_ptr(self, layer):
        return lib().kvo_lw_host_rows(self.h, layer)

    def set_length(self, tokens):
        _check(lib().kvo_lw_set_length(self.h, tokens))

    def begin(self, chunk_tokens, stream=None):
        _check(lib().kvo_lw_begin(self.h, chunk_tokens, _stream(stream)))

    def layer(self, layer, stream=None):
        """The layer's device buffer as an int16 torch tensor [max_tokens][row_elems] (bf16 bits);
        `stream` waits until it holds the cached rows."""
        import torch
        p = ctypes.c_void_p()
        _check(lib().kvo_lw_layer(self.h, layer, ctypes.byref(p), _stream(stream)))
        ptr = int(p.value)
        if ptr not in self._views:
            self._views[ptr] = torch.as_tensor(_DeviceRows(ptr, self.max_tokens, self.row_elems),
                                               device="cuda:%d" % self.device)
        return self._views[ptr]

    def layer_done(self, layer, stream=None):
        _check(lib().kvo_lw_layer_done(self.h, layer, _stream(stream)))

    def end(self, stream=None):
        _check(lib().kvo_lw_end(self.h, _stream(stream)))

    def stats(self):
        a, b = ctypes.c_uint64(), ctypes.c_uint64()
        _check(lib().kvo_lw_stats(self.h, ctypes.byref(a), ctypes.byref(b)))
        return {"bytes_h2d": int(a.value), "bytes_d2h": int(b.value)}


def kvo_wait_selftest(device, limit_ns):
    """(return code, ns waited) of the bounded-wait self-test (KVO_ETIMEOUT expected)."""
    w = ctypes.c_int64()
    rc = lib().kvo_wait_selftest(device, int(limit_ns), ctypes.byref(w))
    return rc, int(w.value)
