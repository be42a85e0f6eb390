"""Thin Python binding of librx (the C ABI declared in include/rx.h).

Argument marshalling only: every function here forwards to the C entry point of the same name
(rx_store_kv -> store_kv, ...).  Tensors are torch CUDA tensors (their data_ptr() is passed) and
the stream defaults to torch's current stream.  There is no fallback: if the library has not been
built, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "librx.so")

RX_OK, RX_ERR_INVALID, RX_ERR_RANGE, RX_ERR_UNSUPPORTED, RX_ERR_CUDA, RX_ERR_TIMEOUT, \
    RX_ERR_WORKSPACE = range(7)
RX_EXTEND_TILES, RX_EXTEND_PAIR = 0, 1

EXPORTED = [
    "rx_status_string", "rx_last_error", "rx_store_kv", "rx_plan_create", "rx_plan_destroy",
    "rx_plan_set_extend_kernel",
    "rx_plan_workspace_size", "rx_plan_upload", "rx_plan_key_reads", "rx_plan_launches",
    "rx_plan_rows",
    "rx_extend_plan",
    "rx_extend_plan_tree", "rx_extend_attn", "rx_decode_plan", "rx_decode_plan_tree",
    "rx_decode_attn", "rx_decode_attn_noalloc", "rx_noalloc_read_status",
    "rx_noalloc_scratch_bytes", "rx_read_status", "rx_selftest_wait_timeout",
    "rx_selftest_pair_mma",
    "rx_check_slots", "rx_check_tables", "rx_radix_create", "rx_radix_destroy",
    "rx_radix_insert", "rx_radix_match", "rx_radix_stats", "rx_radix_acquire", "rx_radix_release",
    "rx_radix_evict", "rx_slot_pool_create", "rx_slot_pool_destroy", "rx_slot_pool_free_count",
    "rx_slot_pool_alloc", "rx_slot_pool_release", "rx_dfs_order", "rx_gain_groups",
    "rx_saved_tokens", "rx_token_saving", "rx_compute_reduction",
]


class RxError(RuntimeError):
    def __init__(self, status: int, msg: str, bad: int = -1):
        super().__init__(f"{msg} (status {status})")
        self.status = status
        self.bad = bad  # the offending index a check reported, else -1


class KVDesc(C.Structure):
    _fields_ = [("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("softmax_scale", C.c_float),
                ("pool_size", C.c_int64), ("req_to_token", C.c_void_p),
                ("req_to_token_rows", C.c_int64), ("req_to_token_stride", C.c_int64)]


_lib = None
_P = C.c_void_p
_I32P = C.POINTER(C.c_int32)
_I64P = C.POINTER(C.c_int64)


def lib():
    """Load librx.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -m prefix_shared_kv_gb300.build`")
    L = C.CDLL(LIB_PATH)
    sig = {
        "rx_status_string": (C.c_char_p, [C.c_int]),
        "rx_last_error": (C.c_char_p, []),
        "rx_store_kv": (C.c_int, [C.POINTER(KVDesc), _P, _P, _P, _P, _P, C.c_int64, _P]),
        "rx_plan_create": (C.c_int, [C.POINTER(_P)]),
        "rx_plan_destroy": (None, [_P]),
        "rx_plan_set_extend_kernel": (C.c_int, [_P, C.c_int32]),
        "rx_plan_workspace_size": (C.c_int, [_P, C.POINTER(C.c_size_t)]),
        "rx_plan_upload": (C.c_int, [_P, _P, C.c_size_t, _P]),
        "rx_plan_key_reads": (C.c_int, [_P, _I64P]),
        "rx_plan_launches": (C.c_int, [_P, _I32P]),
        "rx_plan_rows": (C.c_int, [_P, _I64P]),
        "rx_extend_plan": (C.c_int, [_P, C.POINTER(KVDesc), C.c_int32, _I32P, _I32P, _I32P,
                                     _I32P, C.c_int32, _I32P]),
        "rx_extend_plan_tree": (C.c_int, [_P, C.POINTER(KVDesc), C.c_int32, _I32P, _I32P, _I32P,
                                          _I32P, C.c_int32, _I32P, _I32P]),
        "rx_decode_plan_tree": (C.c_int, [_P, C.POINTER(KVDesc), C.c_int32, _I32P, _I32P, _I32P,
                                          C.c_int32, _I32P, _I32P]),
        "rx_extend_attn": (C.c_int, [_P, C.POINTER(KVDesc), _P, _P, _P, _P, _P, _P, C.c_size_t,
                                     _P]),
        "rx_decode_plan": (C.c_int, [_P, C.POINTER(KVDesc), C.c_int32, _I32P, _I32P, _I32P,
                                     C.c_int32, _I32P]),
        "rx_decode_attn": (C.c_int, [_P, C.POINTER(KVDesc), _P, _P, _P, _P, _P, _P, C.c_size_t,
                                     _P]),
        "rx_decode_attn_noalloc": (C.c_int, [_P, C.POINTER(KVDesc), _P, _P, _P, _P, _P, _P]),
        "rx_noalloc_read_status": (C.c_int, [_I32P, _P]),
        "rx_noalloc_scratch_bytes": (C.c_size_t, []),
        "rx_read_status": (C.c_int, [_P, _I32P, _P]),
        "rx_selftest_wait_timeout": (C.c_int, [_P, C.c_int64, _P]),
        "rx_selftest_pair_mma": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, _P]),
        "rx_radix_create": (C.c_int, [C.POINTER(_P)]),
        "rx_radix_destroy": (None, [_P]),
        "rx_radix_insert": (C.c_int, [_P, _I32P, _I32P, C.c_int64, _I64P]),
        "rx_radix_match": (C.c_int, [_P, _I32P, C.c_int64, C.c_int32, _I64P, _I32P]),
        "rx_radix_stats": (C.c_int, [_P, _I64P, _I64P]),
        "rx_radix_acquire": (C.c_int, [_P, _I32P, C.c_int64, C.c_int32, C.c_int32, _I64P, _I32P]),
        "rx_radix_release": (C.c_int, [_P, _I32P, C.c_int64]),
        "rx_radix_evict": (C.c_int, [_P, C.c_int64, _I32P, C.c_int64, _I64P]),
        "rx_slot_pool_create": (C.c_int, [C.c_int64, C.POINTER(_P)]),
        "rx_slot_pool_destroy": (None, [_P]),
        "rx_slot_pool_free_count": (C.c_int64, [_P]),
        "rx_slot_pool_alloc": (C.c_int, [_P, _P, C.c_int64, _I32P]),
        "rx_slot_pool_release": (C.c_int, [_P, _I32P, C.c_int64]),
        "rx_dfs_order": (C.c_int, [_I32P, _I64P, C.c_int32, _I32P]),
        "rx_gain_groups": (C.c_int, [_I32P, _I64P, C.c_int32, _I32P, _I32P, _I32P]),
        "rx_saved_tokens": (C.c_int64, [C.c_int64, C.c_int32]),
        "rx_token_saving": (C.c_double, [C.c_int64, C.c_int64]),
        "rx_compute_reduction": (C.c_double, [C.c_int64, C.c_int64]),
        "rx_check_slots": (C.c_int, [_I32P, C.c_int64, C.c_int64, _I64P]),
        "rx_check_tables": (C.c_int, [_I32P, C.c_int64, C.c_int64, C.c_int64, C.c_int32, _I32P,
                                      _I32P, _I32P, C.c_int32, _I32P, _I32P, _I64P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(status: int, bad: int = -1):
    if status != RX_OK:
        L = lib()
        raise RxError(status, f"{L.rx_status_string(status).decode()}: {L.rx_last_error().decode()}",
                      bad)


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host_i32(a):
    """Host int32 array (numpy, list or CPU tensor) -> (numpy array kept alive, pointer)."""
    if a is None:
        return None, None
    if hasattr(a, "cpu") and not isinstance(a, np.ndarray):
        a = a.cpu().numpy()
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, arr.ctypes.data_as(_I32P)


def _same_length(*arrays):
    """The C calls take one count per group of arrays: arrays given (not None) must agree."""
    n = {int(a.shape[0]) for a in arrays if a is not None}
    if len(n) > 1:
        raise ValueError(f"array lengths differ: {sorted(n)}")


def kv_desc(num_q_heads: int, num_kv_heads: int, pool_size: int, req_to_token,
            softmax_scale: Optional[float] = None, head_dim: int = 128) -> KVDesc:
    """Descriptor of the pool and of req_to_token (a [rows, stride] int32 CUDA tensor)."""
    if softmax_scale is None:
        softmax_scale = head_dim ** -0.5
    rows, stride = (req_to_token.shape if req_to_token is not None else (0, 0))
    if req_to_token is not None and req_to_token.numel() > 0 and req_to_token.stride(1) != 1:
        raise ValueError("req_to_token rows must be contiguous")
    return KVDesc(num_q_heads, num_kv_heads, head_dim, softmax_scale, pool_size,
                  _ptr(req_to_token), rows, req_to_token.stride(0) if req_to_token is not None else 0)


def store_kv(desc: KVDesc, k_pool, v_pool, k_new, v_new, slots, stream=None):
    n = int(slots.shape[0]) if slots is not None else 0
    row = desc.num_kv_heads * desc.head_dim
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if n > 0 and hasattr(t, "numel") and t.numel() != n * row:
            raise ValueError(f"{name} holds {t.numel()} elements, slots ask for {n} x {row}")
    _check(lib().rx_store_kv(C.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
                             _ptr(slots), n, _stream(stream)))


class Plan:
    """rx_plan: host-built work list for one batch (extend or decode)."""

    def __init__(self):
        h = _P()
        _check(lib().rx_plan_create(C.byref(h)))
        self._h = h

    def close(self):
        if self._h:
            lib().rx_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def set_extend_kernel(self, kernel: int):
        """rx_plan_set_extend_kernel: RX_EXTEND_TILES (default) or RX_EXTEND_PAIR for the extend
        plans built from now on."""
        _check(lib().rx_plan_set_extend_kernel(self._h, int(kernel)))

    def workspace_size(self) -> int:
        n = C.c_size_t(0)
        _check(lib().rx_plan_workspace_size(self._h, C.byref(n)))
        return n.value

    def rows(self) -> int:
        """Rows of q / o / lse an attention call with the plan touches (rx_plan_rows)."""
        n = np.zeros(1, np.int64)
        _check(lib().rx_plan_rows(self._h, n.ctypes.data_as(_I64P)))
        return int(n[0])

    def launches(self) -> int:
        """Kernels one attention call with the plan launches (rx_plan_launches)."""
        n = np.zeros(1, np.int32)
        _check(lib().rx_plan_launches(self._h, n.ctypes.data_as(_I32P)))
        return int(n[0])

    def key_reads(self) -> int:
        """(key, KV head) rows of the pool the plan's kernels read (rx_plan_key_reads)."""
        n = np.zeros(1, np.int64)
        _check(lib().rx_plan_key_reads(self._h, n.ctypes.data_as(_I64P)))
        return int(n[0])

    def upload(self, workspace, nbytes: Optional[int] = None, stream=None):
        if nbytes is None:
            nbytes = workspace.numel() * workspace.element_size()
        _check(lib().rx_plan_upload(self._h, _ptr(workspace), nbytes, _stream(stream)))


def extend_plan(plan: Plan, desc: KVDesc, req_idx, prefix_len, extend_len, group_of_req=None,
                group_prefix_len=None, group_parent=None):
    """rx_extend_plan, or rx_extend_plan_tree when group_parent is given."""
    ri, rip = _host_i32(req_idx)
    pl, plp = _host_i32(prefix_len)
    el, elp = _host_i32(extend_len)
    g, gp_ = _host_i32(group_of_req)
    gl, glp = _host_i32(group_prefix_len)
    pa, pap = _host_i32(group_parent)
    ng = 0 if gl is None else int(gl.shape[0])
    _same_length(ri, pl, el, g)
    _same_length(gl, pa)
    if pa is None:
        _check(lib().rx_extend_plan(plan.handle, C.byref(desc), int(ri.shape[0]), rip, plp, elp,
                                    gp_, ng, glp))
    else:
        _check(lib().rx_extend_plan_tree(plan.handle, C.byref(desc), int(ri.shape[0]), rip, plp,
                                         elp, gp_, ng, glp, pap))


def decode_plan(plan: Plan, desc: KVDesc, req_idx, seq_len, group_of_req=None,
                group_prefix_len=None, group_parent=None):
    """rx_decode_plan, or rx_decode_plan_tree when group_parent is given."""
    ri, rip = _host_i32(req_idx)
    sl, slp = _host_i32(seq_len)
    g, gp_ = _host_i32(group_of_req)
    gl, glp = _host_i32(group_prefix_len)
    pa, pap = _host_i32(group_parent)
    ng = 0 if gl is None else int(gl.shape[0])
    _same_length(ri, sl, g)
    _same_length(gl, pa)
    if pa is None:
        _check(lib().rx_decode_plan(plan.handle, C.byref(desc), int(ri.shape[0]), rip, slp, gp_,
                                    ng, glp))
    else:
        _check(lib().rx_decode_plan_tree(plan.handle, C.byref(desc), int(ri.shape[0]), rip, slp,
                                         gp_, ng, glp, pap))


def _nbytes(t) -> int:
    if t is None or isinstance(t, int):
        return 0
    return t.numel() * t.element_size()


def check_io(plan: Plan, desc: KVDesc, q, o, lse):
    """The kernels write o and lse by row index, so buffers smaller than the plan's rows would be
    written past their end: tensors (anything with numel / dtype) must hold exactly the plan's
    rows -- q, o bf16 [rows, Hq, head_dim], lse float32 [rows, Hq].  Raw addresses (ints) are
    the caller's responsibility."""
    n = plan.rows()
    per = desc.num_q_heads * desc.head_dim
    for name, t, want, dt in (("q", q, n * per, "bfloat16"), ("o", o, n * per, "bfloat16"),
                              ("lse", lse, n * desc.num_q_heads, "float32")):
        if hasattr(t, "numel") and t.numel() != want:
            raise ValueError(f"{name} holds {t.numel()} elements; the plan's {n} rows need {want}")
        if hasattr(t, "dtype") and not str(t.dtype).endswith(dt):
            raise ValueError(f"{name} is {t.dtype}, {dt} expected")


def extend_attn(plan: Plan, desc: KVDesc, k_pool, v_pool, q, o, lse, workspace, stream=None):
    check_io(plan, desc, q, o, lse)
    _check(lib().rx_extend_attn(plan.handle, C.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(q),
                                _ptr(o), _ptr(lse), _ptr(workspace), _nbytes(workspace),
                                _stream(stream)))


def decode_attn(plan: Plan, desc: KVDesc, k_pool, v_pool, q, o, lse, workspace, stream=None):
    check_io(plan, desc, q, o, lse)
    _check(lib().rx_decode_attn(plan.handle, C.byref(desc), _ptr(k_pool), _ptr(v_pool), _ptr(q),
                                _ptr(o), _ptr(lse), _ptr(workspace), _nbytes(workspace),
                                _stream(stream)))


def decode_attn_noalloc(plan: Plan, desc: KVDesc, k_pool, v_pool, q, o, lse, stream=None):
    """rx_decode_attn_noalloc: decode without a workspace (the library's own scratch is used)."""
    check_io(plan, desc, q, o, lse)
    _check(lib().rx_decode_attn_noalloc(plan.handle, C.byref(desc), _ptr(k_pool), _ptr(v_pool),
                                        _ptr(q), _ptr(o), _ptr(lse), _stream(stream)))


def noalloc_scratch_bytes() -> int:
    """rx_noalloc_scratch_bytes: the largest plan rx_decode_attn_noalloc takes."""
    return int(lib().rx_noalloc_scratch_bytes())


def noalloc_read_status(stream=None) -> int:
    """rx_noalloc_read_status: the status word of the last rx_decode_attn_noalloc call on the
    current device (waits for `stream`; clears the word)."""
    s = C.c_int32(0)
    _check(lib().rx_noalloc_read_status(C.byref(s), _stream(stream)))
    return s.value


def read_status(workspace, stream=None) -> int:
    s = C.c_int32(0)
    _check(lib().rx_read_status(_ptr(workspace), C.byref(s), _stream(stream)))
    return s.value


class Radix:
    """rx_radix: host radix cache of token sequences -> pool slots."""

    def __init__(self):
        h = _P()
        _check(lib().rx_radix_create(C.byref(h)))
        self._h = h

    def __del__(self):
        try:
            if self._h:
                lib().rx_radix_destroy(self._h)
                self._h = None
        except Exception:
            pass

    def insert(self, tokens, slots) -> int:
        t, tp = _host_i32(tokens)
        s, sp = _host_i32(slots)
        if t.shape != s.shape:
            raise ValueError("tokens and slots differ in length")
        n = C.c_int64(0)
        _check(lib().rx_radix_insert(self._h, tp, sp, int(t.shape[0]), C.byref(n)))
        return n.value

    def match(self, tokens, match_unit: int = 1, want_slots: bool = True):
        t, tp = _host_i32(tokens)
        saved = C.c_int64(0)
        out = np.zeros(max(1, t.shape[0]), np.int32) if want_slots else None
        _check(lib().rx_radix_match(self._h, tp, int(t.shape[0]), match_unit, C.byref(saved),
                                    out.ctypes.data_as(_I32P) if want_slots else None))
        return (saved.value, out[:saved.value].copy()) if want_slots else saved.value

    def stats(self):
        a, b = C.c_int64(0), C.c_int64(0)
        _check(lib().rx_radix_stats(self._h, C.byref(a), C.byref(b)))
        return a.value, b.value

    def acquire(self, tokens, match_unit: int = 1, lock: bool = True):
        """(saved tokens, their slots); with lock the saved prefix is held until release()."""
        t, tp = _host_i32(tokens)
        saved = C.c_int64(0)
        out = np.zeros(max(1, t.shape[0]), np.int32)
        _check(lib().rx_radix_acquire(self._h, tp, int(t.shape[0]), match_unit, int(bool(lock)),
                                      C.byref(saved), out.ctypes.data_as(_I32P)))
        return saved.value, out[:saved.value].copy()

    def release(self, tokens):
        t, tp = _host_i32(tokens)
        _check(lib().rx_radix_release(self._h, tp, int(t.shape[0])))

    def evict(self, n_tokens: int) -> np.ndarray:
        """Slots freed by evicting least recently used unheld leaves (>= n_tokens if possible)."""
        total, _ = self.stats()
        out = np.zeros(max(1, total), np.int32)
        n = C.c_int64(0)
        _check(lib().rx_radix_evict(self._h, int(n_tokens), out.ctypes.data_as(_I32P), total,
                                    C.byref(n)))
        return out[:n.value].copy()


class SlotPool:
    """rx_slot_pool: free pool slots shared by the cache and the running requests."""

    def __init__(self, pool_size: int):
        h = _P()
        _check(lib().rx_slot_pool_create(int(pool_size), C.byref(h)))
        self._h = h

    def __del__(self):
        try:
            if self._h:
                lib().rx_slot_pool_destroy(self._h)
                self._h = None
        except Exception:
            pass

    def free_count(self) -> int:
        return int(lib().rx_slot_pool_free_count(self._h))

    def alloc(self, n: int, tree: Optional["Radix"] = None) -> np.ndarray:
        out = np.zeros(max(1, n), np.int32)
        _check(lib().rx_slot_pool_alloc(self._h, tree._h if tree is not None else None, int(n),
                                        out.ctypes.data_as(_I32P)))
        return out[:n].copy()

    def release(self, slots):
        s, sp = _host_i32(slots)
        _check(lib().rx_slot_pool_release(self._h, sp, int(s.shape[0])))


def dfs_order(sequences) -> np.ndarray:
    """rx_dfs_order: the depth-first order of the batch's radix tree (a permutation)."""
    seqs = [np.asarray(q, np.int32) for q in sequences]
    offs = np.zeros(len(seqs) + 1, np.int64)
    offs[1:] = np.cumsum([len(q) for q in seqs])
    toks = np.ascontiguousarray(np.concatenate(seqs) if seqs else np.zeros(1, np.int32))
    order = np.zeros(max(1, len(seqs)), np.int32)
    _check(lib().rx_dfs_order(toks.ctypes.data_as(_I32P), offs.ctypes.data_as(_I64P), len(seqs),
                              order.ctypes.data_as(_I32P)))
    return order[:len(seqs)].copy()


def gain_groups(sequences):
    """rx_gain_groups: (group_of_req, group_prefix_len) under BatchLLM's gain rule."""
    seqs = [np.asarray(q, np.int32) for q in sequences]
    offs = np.zeros(len(seqs) + 1, np.int64)
    offs[1:] = np.cumsum([len(q) for q in seqs])
    toks = np.ascontiguousarray(np.concatenate(seqs) if seqs else np.zeros(1, np.int32))
    grp = np.zeros(max(1, len(seqs)), np.int32)
    gpl = np.zeros(max(1, len(seqs)), np.int32)
    ng = np.zeros(1, np.int32)
    _check(lib().rx_gain_groups(toks.ctypes.data_as(_I32P), offs.ctypes.data_as(_I64P), len(seqs),
                                grp.ctypes.data_as(_I32P), gpl.ctypes.data_as(_I32P),
                                ng.ctypes.data_as(_I32P)))
    return grp[:len(seqs)].copy(), gpl[:int(ng[0])].copy()


def selftest_pair_mma(q, k, v, p, s_out, o_out, info, stream=None):
    """rx_selftest_pair_mma: s_out = q k^T, o_out = p v on one SM pair (see rx.h)."""
    for t, shape in ((q, (256, 128)), (k, (128, 128)), (v, (128, 128)), (p, (256, 128))):
        if tuple(t.shape) != shape or t.dtype.itemsize != 2 or not t.is_contiguous():
            raise ValueError(f"bf16 operand of shape {shape} expected")
    for t in (s_out, o_out):
        if tuple(t.shape) != (256, 128) or t.dtype.itemsize != 4 or not t.is_contiguous():
            raise ValueError("fp32 output of shape (256, 128) expected")
    if info.numel() < 3 or info.dtype.itemsize != 4:
        raise ValueError("int32 info of 3 elements expected")
    _check(lib().rx_selftest_pair_mma(_ptr(q), _ptr(k), _ptr(v), _ptr(p), _ptr(s_out),
                                      _ptr(o_out), _ptr(info), _stream(stream)))


def selftest_wait_timeout(status, limit_ns: int, stream=None):
    """rx_selftest_wait_timeout: a bounded wait that runs out; writes RX_ERR_TIMEOUT to `status`."""
    _check(lib().rx_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)))


def saved_tokens(matched: int, unit: int) -> int:
    return lib().rx_saved_tokens(matched, unit)


def token_saving(n_processed: int, n_logical: int) -> float:
    return lib().rx_token_saving(n_processed, n_logical)


def compute_reduction(l_prefix: int, l_new: int) -> float:
    return lib().rx_compute_reduction(l_prefix, l_new)


def check_slots(slots, pool_size: int):
    """rx_check_slots: raises RxError (with .bad = the token) unless the host slots are distinct
    and inside the pool."""
    a, ap = _host_i32(slots)
    bad = C.c_int64(-1)
    st = lib().rx_check_slots(ap, int(a.shape[0]), int(pool_size), C.byref(bad))
    _check(st, bad.value)


def check_tables(req_to_token, pool_size: int, req_idx, key_len, group_of_req=None,
                 group_prefix_len=None, group_parent=None):
    """rx_check_tables on a host copy of req_to_token ([rows, stride] int32): raises RxError
    (with .bad = the request) unless every slot a request reads is inside the pool and every
    declared shared prefix is the same in all rows that declare it."""
    t = req_to_token.cpu().numpy() if hasattr(req_to_token, "cpu") else req_to_token
    t = np.ascontiguousarray(np.asarray(t, dtype=np.int32))
    if t.ndim != 2:
        raise ValueError("req_to_token must be [rows, stride]")
    ri, rip = _host_i32(req_idx)
    kl, klp = _host_i32(key_len)
    g, gp_ = _host_i32(group_of_req)
    gl, glp = _host_i32(group_prefix_len)
    pa, pap = _host_i32(group_parent)
    ng = 0 if gl is None else int(gl.shape[0])
    _same_length(ri, kl, g)
    _same_length(gl, pa)
    bad = C.c_int64(-1)
    st = lib().rx_check_tables(t.ctypes.data_as(_I32P), int(t.shape[0]), int(t.shape[1]),
                               int(pool_size), int(ri.shape[0]), rip, klp, gp_, ng, glp, pap,
                               C.byref(bad))
    _check(st, bad.value)
