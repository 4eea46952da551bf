"""ctypes binding of libzerogr.so: the C ABI declared in include/zerogr.h.

Argument marshalling only.  Every step of the decode runs in the library's
CUDA kernels; if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzerogr.so")

ZG_MAX_STEPS = 8
ZG_MAX_BEAM = 512
ZG_OK = 0
STATUS_NAMES = {0: "ZG_OK", 1: "ZG_ERR_INVALID_ARG", 2: "ZG_ERR_OUT_OF_MEMORY", 3: "ZG_ERR_CUDA",
                4: "ZG_ERR_UNSUPPORTED", 5: "ZG_ERR_TIMEOUT", 6: "ZG_ERR_DEVICE_STATUS", 7: "ZG_ERR_IO"}
ZG_F32, ZG_BF16, ZG_F16 = 0, 1, 2
DTYPES = {"f32": ZG_F32, "bf16": ZG_BF16, "f16": ZG_F16}
ZG_FMT_SPARSE, ZG_FMT_DENSE = 0, 1
ZG_SELECTIVE, ZG_FULL, ZG_NAIVE = 0, 1, 2
ZG_RESIDENT_DEVICE, ZG_RESIDENT_HOST = 0, 1
ZG_FORMAT_AUTO, ZG_FORMAT_ALL_SPARSE, ZG_FORMAT_ALL_DENSE = 0, 1, 2
ZG_ORDER_FILTER_FIRST, ZG_ORDER_SCORE_FIRST = 0, 1
ZG_HIDDEN_SPLIT, ZG_HIDDEN_SINGLE = 0, 1
ZG_SCORES_AUTO, ZG_SCORES_WRITTEN, ZG_SCORES_CHUNK_TOPS = 0, 1, 2


class ZgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


ZG_MAX_DECO_LAYERS = 4


class zg_deco(C.Structure):
    _fields_ = [("M", C.c_int32), ("heads", C.c_int32), ("ffn", C.c_int32), ("layers", C.c_int32),
                ("E", C.c_void_p * ZG_MAX_STEPS), ("P", C.c_void_p)] + \
               [(n, C.c_void_p * ZG_MAX_DECO_LAYERS) for n in ("Wq", "Wk", "Wv", "Wo", "W1", "W2")]


class zg_model(C.Structure):
    _fields_ = [("L", C.c_int32), ("V", C.c_int32), ("d", C.c_int32), ("w_dtype", C.c_int32),
                ("C", C.c_void_p * ZG_MAX_STEPS), ("W", C.c_void_p * ZG_MAX_STEPS),
                ("deco", C.POINTER(zg_deco))]


class zg_build_opts(C.Structure):
    _fields_ = [("n_threads", C.c_int32), ("format_mode", C.c_int32), ("reserved", C.c_int32),
                ("residency", C.c_int32), ("pinned_chunk_bytes", C.c_uint64)]


class zg_step_stats(C.Structure):
    _fields_ = [("format", C.c_int32), ("rows", C.c_uint32), ("nnz", C.c_uint32),
                ("words_per_row", C.c_uint32), ("max_fanout", C.c_uint32), ("reserved", C.c_uint32),
                ("mean_fanout", C.c_double), ("legal_fraction", C.c_double), ("bytes", C.c_uint64)]


class zg_index_info(C.Structure):
    _fields_ = [("L", C.c_int32), ("V", C.c_int32), ("residency", C.c_int32), ("reserved", C.c_int32),
                ("n_input", C.c_int64), ("n_unique", C.c_int64), ("bytes", C.c_uint64),
                ("dense_trie_bytes", C.c_uint64), ("ms_sort", C.c_double), ("ms_count", C.c_double),
                ("ms_fill", C.c_double), ("ms_total", C.c_double)]


class zg_step_trace(C.Structure):
    _fields_ = [("variant", C.c_int32), ("live_beams", C.c_int32), ("legal_slots", C.c_int64),
                ("chunks", C.c_int64), ("unique_tokens", C.c_int64), ("index_bytes", C.c_int64),
                ("ms_gather", C.c_float), ("ms_project", C.c_float), ("ms_select", C.c_float),
                ("ms_model", C.c_float)]


class zg_trace(C.Structure):
    _fields_ = [("L", C.c_int32), ("fused_from", C.c_int32), ("step", zg_step_trace * ZG_MAX_STEPS),
                ("ms_fused", C.c_float), ("ms_total", C.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (nvcc, sm_103a)")
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64, u64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_size_t
    P = C.POINTER
    sigs = {
        "zg_index_build": [vp, i64, i32, i32, P(zg_build_opts), vp, P(vp)],
        "zg_index_stats": [vp, i32, P(zg_step_stats)],
        "zg_index_info_get": [vp, P(zg_index_info)],
        "zg_index_export": [vp, i32, vp, P(sz)],
        "zg_index_save": [vp, C.c_char_p],
        "zg_index_load": [C.c_char_p, i32, vp, P(vp)],
        "zg_tune": [vp, P(zg_model), vp, i32, i32, i32, i32, vp, P(vp)],
        "zg_plan_force": [vp, i32, i32, vp, P(vp)],
        "zg_plan_describe": [vp, vp, vp, vp, vp],
        "zg_plan_set_fusion": [vp, i32],
        "zg_plan_set_order": [vp, i32],
        "zg_plan_set_full_projection": [vp, i32, i32],
        "zg_decode_workspace_size": [vp, vp, P(zg_model), i32, i32, i32, P(sz)],
        "zg_decode": [vp, vp, P(zg_model), vp, i32, i32, i32, vp, vp, vp, sz, vp],
        "zg_decode_host_workspace_size": [vp, vp, P(zg_model), i32, i32, i32, P(sz)],
        "zg_decode_host": [vp, vp, P(zg_model), vp, i32, i32, i32, vp, vp, vp, sz, vp],
        "zg_decode_trace": [vp, vp, P(zg_model), vp, i32, i32, i32, vp, vp, vp, sz, vp, P(zg_trace)],
        "zg_decode_static": [vp, vp, P(zg_model), vp, i32, i32, i32, vp, vp, vp],
        "zg_check_device_status": [vp],
        "zg_plan_save": [vp, C.c_char_p],
        "zg_plan_load": [C.c_char_p, P(vp)],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = C.c_int
    lib.zg_index_free.argtypes = [vp]
    lib.zg_index_free.restype = None
    lib.zg_plan_free.argtypes = [vp]
    lib.zg_plan_free.restype = None
    lib.zg_last_error.argtypes = []
    lib.zg_last_error.restype = C.c_char_p
    lib.zg_version.argtypes = []
    lib.zg_version.restype = C.c_char_p
    lib.zg_static_scratch_bytes.argtypes = []
    lib.zg_static_scratch_bytes.restype = C.c_size_t
    lib.zg_debug_set_wait_limit.argtypes = [C.c_uint32]
    lib.zg_debug_set_wait_limit.restype = None
    lib.zg_debug_inject_build_failure.argtypes = [C.c_int32, C.c_int32]
    lib.zg_debug_inject_build_failure.restype = None
    return lib


lib = _load()


def _check(status: int):
    if status != ZG_OK:
        raise ZgError(status, lib.zg_last_error().decode(errors="replace"))


def _ptr(x) -> int | None:
    """Device/host address of a torch tensor, numpy array or int (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(type(x))


class Index:
    """Owner of a zg_index handle."""

    def __init__(self, handle: int):
        self.handle = handle

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            lib.zg_index_free(h)
            self.handle = None

    @property
    def _as_parameter_(self):
        return self.handle


class Plan:
    """Owner of a zg_plan handle."""

    def __init__(self, handle: int, L: int):
        self.handle = handle
        self.L = L

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            lib.zg_plan_free(h)
            self.handle = None

    @property
    def _as_parameter_(self):
        return self.handle


def zg_version() -> str:
    return lib.zg_version().decode()


def zg_index_build(sids: np.ndarray, V: int, *, n_threads: int = 0, format_mode: int = ZG_FORMAT_AUTO,
                   residency: int = ZG_RESIDENT_DEVICE, pinned_chunk_bytes: int = 0, stream: int = 0) -> Index:
    sids = np.ascontiguousarray(sids, dtype=np.int32)
    if sids.ndim != 2:
        raise ValueError("sids must be [n, L]")
    opts = zg_build_opts(n_threads, format_mode, 0, residency, pinned_chunk_bytes)
    h = C.c_void_p()
    _check(lib.zg_index_build(sids.ctypes.data, sids.shape[0], sids.shape[1], V, C.byref(opts),
                              stream or None, C.byref(h)))
    return Index(h.value)


def zg_index_stats(idx: Index, step: int) -> dict:
    st = zg_step_stats()
    _check(lib.zg_index_stats(idx, step, C.byref(st)))
    return {f: getattr(st, f) for f, _ in zg_step_stats._fields_ if f != "reserved"}


def zg_index_info_get(idx: Index) -> dict:
    info = zg_index_info()
    _check(lib.zg_index_info_get(idx, C.byref(info)))
    return {f: getattr(info, f) for f, _ in zg_index_info._fields_ if f != "reserved"}


def zg_index_export(idx: Index, step: int) -> bytes:
    n = C.c_size_t(0)
    _check(lib.zg_index_export(idx, step, None, C.byref(n)))
    buf = (C.c_uint8 * n.value)()
    _check(lib.zg_index_export(idx, step, buf, C.byref(n)))
    return bytes(buf)


def zg_index_save(idx: Index, path: str):
    _check(lib.zg_index_save(idx, path.encode()))


def zg_index_load(path: str, residency: int = ZG_RESIDENT_DEVICE, stream: int = 0) -> Index:
    h = C.c_void_p()
    _check(lib.zg_index_load(path.encode(), residency, stream or None, C.byref(h)))
    return Index(h.value)


def make_model(L: int, V: int, d: int, w_dtype: int, C_ptrs, W_ptrs, deco: zg_deco | None = None) -> zg_model:
    m = zg_model()
    m.L, m.V, m.d, m.w_dtype = L, V, d, w_dtype
    for s, p in enumerate(C_ptrs):
        m.C[s] = _ptr(p)
    for s, p in enumerate(W_ptrs):
        m.W[s] = _ptr(p)
    if deco is not None:
        m.deco = C.pointer(deco)
        m._deco_ref = deco          # keeps the struct alive with the model
    return m


def make_deco(M: int, heads: int, ffn: int, E_ptrs, P_ptr, Wq, Wk, Wv, Wo, W1, W2) -> zg_deco:
    """zg_deco from device pointers (per layer lists for the matrices)."""
    t = zg_deco()
    t.M, t.heads, t.ffn, t.layers = M, heads, ffn, len(Wq)
    for s, p in enumerate(E_ptrs):
        t.E[s] = _ptr(p)
    t.P = _ptr(P_ptr)
    for name, ptrs in (("Wq", Wq), ("Wk", Wk), ("Wv", Wv), ("Wo", Wo), ("W1", W1), ("W2", W2)):
        arr = getattr(t, name)
        for l, p in enumerate(ptrs):
            arr[l] = _ptr(p)
    return t


def zg_plan_force(idx: Index, B: int, beam: int, variant) -> Plan:
    v = np.ascontiguousarray(variant, dtype=np.uint8)
    h = C.c_void_p()
    _check(lib.zg_plan_force(idx, B, beam, v.ctypes.data, C.byref(h)))
    return Plan(h.value, v.size)


def zg_tune(idx: Index, model: zg_model, warm_u, B: int, beam: int, K: int, reps: int = 10,
            stream: int = 0) -> Plan:
    h = C.c_void_p()
    _check(lib.zg_tune(idx, C.byref(model), _ptr(warm_u), B, beam, K, reps, stream or None, C.byref(h)))
    return Plan(h.value, model.L)


def zg_plan_describe(plan: Plan):
    """(variant [L], step_ms [L, 2], cluster_ctas, fused_ms [5])."""
    v = np.zeros(plan.L, np.uint8)
    ms = np.zeros((plan.L, 2), np.float32)
    g = C.c_int32(0)
    fms = np.zeros(5, np.float32)
    _check(lib.zg_plan_describe(plan, v.ctypes.data, ms.ctypes.data, C.byref(g), fms.ctypes.data))
    return v, ms, g.value, fms


def zg_decode_workspace_size(idx: Index | None, plan: Plan | None, model: zg_model, B: int, beam: int,
                             K: int) -> int:
    n = C.c_size_t(0)
    _check(lib.zg_decode_workspace_size(idx, plan, C.byref(model), B, beam, K, C.byref(n)))
    return n.value


def zg_decode_host_workspace_size(idx: Index | None, plan: Plan | None, model: zg_model, B: int, beam: int,
                                  K: int) -> int:
    n = C.c_size_t(0)
    _check(lib.zg_decode_host_workspace_size(idx, plan, C.byref(model), B, beam, K, C.byref(n)))
    return n.value


def zg_decode(idx: Index | None, plan: Plan | None, model: zg_model, u, B: int, beam: int, K: int, out_sids,
              out_scores, workspace, ws_bytes: int, stream: int = 0):
    _check(lib.zg_decode(idx, plan, C.byref(model), _ptr(u), B, beam, K, _ptr(out_sids), _ptr(out_scores),
                         _ptr(workspace), ws_bytes, stream or None))


def zg_decode_host(idx: Index | None, plan: Plan | None, model: zg_model, u_host, B: int, beam: int, K: int,
                   out_sids_host, out_scores_host, workspace, ws_bytes: int, stream: int = 0):
    _check(lib.zg_decode_host(idx, plan, C.byref(model), _ptr(u_host), B, beam, K, _ptr(out_sids_host),
                              _ptr(out_scores_host), _ptr(workspace), ws_bytes, stream or None))


ZG_STATIC_SCRATCH_BYTES = int(lib.zg_static_scratch_bytes())   # as compiled into the library


def zg_decode_static(idx: Index | None, plan: Plan | None, model: zg_model, u, B: int, beam: int, K: int,
                     out_sids, out_scores, stream: int = 0):
    """zg_decode without a workspace: scratch from the library's static device array."""
    _check(lib.zg_decode_static(idx, plan, C.byref(model), _ptr(u), B, beam, K, _ptr(out_sids),
                                _ptr(out_scores), stream or None))


ZG_INJECT_PINNED_ALLOC, ZG_INJECT_COPY = 1, 2


def zg_debug_inject_build_failure(point: int = 0, after: int = 0):
    """Make the index builder's (after+1)-th next pinned allocation or copy fail once (0: disarm)."""
    lib.zg_debug_inject_build_failure(int(point), int(after))


def zg_plan_save(plan: Plan, path: str):
    _check(lib.zg_plan_save(plan, path.encode()))


def zg_plan_load(path: str) -> Plan:
    h = C.c_void_p()
    _check(lib.zg_plan_load(path.encode(), C.byref(h)))
    with open(path, "rb") as f:                 # steps: the int32 after the 8-byte magic
        L = int.from_bytes(f.read(12)[8:12], "little")
    return Plan(h.value, L)


def zg_debug_set_wait_limit(polls: int = 0):
    """Polls before a tensor-core pipeline wait gives up (0: the default)."""
    lib.zg_debug_set_wait_limit(int(polls))


def zg_check_device_status(stream: int = 0):
    _check(lib.zg_check_device_status(stream or None))


def zg_decode_trace(idx: Index | None, plan: Plan | None, model: zg_model, u, B: int, beam: int, K: int,
                    out_sids, out_scores, workspace, ws_bytes: int, stream: int = 0) -> dict:
    """Kernel times (ms) of zg_decode's launch sequence and, per step, of the
    stand-alone step kernels with their work counts."""
    t = zg_trace()
    _check(lib.zg_decode_trace(idx, plan, C.byref(model), _ptr(u), B, beam, K, _ptr(out_sids),
                               _ptr(out_scores), _ptr(workspace), ws_bytes, stream or None, C.byref(t)))
    steps = [{f: getattr(t.step[i], f) for f, _ in zg_step_trace._fields_ if f != "reserved"}
             for i in range(t.L)]
    return {"fused_from": t.fused_from, "ms_fused": t.ms_fused, "ms_total": t.ms_total, "steps": steps}


def zg_plan_set_order(plan: Plan, order: int):
    """ZG_ORDER_FILTER_FIRST (default) or ZG_ORDER_SCORE_FIRST (every step full,
    log-softmax over the whole codebook, then the mask)."""
    _check(lib.zg_plan_set_order(plan, int(order)))


def zg_plan_set_full_projection(plan: Plan, hidden_rounding: int = ZG_HIDDEN_SPLIT, scores: int = ZG_SCORES_AUTO):
    """How full steps run: the hidden as two half operands or one rounding;
    scores written out or handed to the select as chunk tops (auto by size)."""
    _check(lib.zg_plan_set_full_projection(plan, int(hidden_rounding), int(scores)))


def zg_plan_set_fusion(plan: Plan, cluster_ctas):
    """cluster_ctas: 0 (stand-alone step kernels) or 1, 2, 4, 8, 16; True = 8."""
    if cluster_ctas is True:
        cluster_ctas = 8
    _check(lib.zg_plan_set_fusion(plan, int(cluster_ctas)))
