"""GB300 offloaded-MoE expert slot cache: Python binding of libmoecache.so.

Every function here has the name of the C entry point it calls (see
``include/moe_cache.h`` for the meaning, layout, ownership and errors of each
argument) and only marshals arguments: tensors become device or host
addresses, streams become ``cudaStream_t`` handles, error codes become
:class:`MoeError`.  All of the hot path runs in the library's CUDA kernels.
There is no fallback: if the shared library is missing this import fails.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoecache.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
        "or python expert_slot_cache_lru_gb300/build.py); there is no CPU fallback")

_lib = C.CDLL(LIB_PATH)

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_CONFIG = -2
MOE_ERR_CUDA = -3
MOE_ERR_CAPACITY = -4
MOE_ERR_UNSUPPORTED = -5
MOE_ERR_STATE = -6
MOE_ERR_INJECTED = -7
MOE_ERR_SCRATCH = -8
MOE_NOALLOC_SCRATCH_BYTES = 1 << 20
MOE_W_BF16 = 0
MOE_W_NVFP4 = 1
MOE_W_MXFP4 = 2
MOE_W_Q4_0 = 3
MOE_POOL_SHARED = 0
MOE_POOL_PER_LAYER = 1
MOE_PLAN_DEMAND = 0
MOE_PLAN_PREFETCH = 1
MOE_OVERLAP = 1
MOE_FUSED = 2
MOE_HYBRID = 4
MOE_STATUS_INVALID_ID = 1
MOE_STATUS_CAPACITY = 2
MOE_STATUS_TIMEOUT = 4
MOE_WIDE_AUTO = 0
MOE_WIDE_CUDA_CORES = 1
MOE_WIDE_TENSOR_CORES = 2


class moe_cache_desc(C.Structure):
    _fields_ = [
        ("n_layers", C.c_int), ("n_experts", C.c_int), ("n_slots", C.c_int),
        ("pool_mode", C.c_int), ("hidden", C.c_int), ("inter", C.c_int), ("wfmt", C.c_int),
        ("shared_inter", C.c_int), ("slot_bytes", C.c_size_t), ("slot_stride", C.c_size_t),
        ("slot_storage", C.c_void_p), ("host_experts", C.c_void_p), ("max_routes", C.c_int),
        ("max_rows", C.c_int), ("max_pred", C.c_int), ("gather_ctas", C.c_int),
    ]


STAT_FIELDS = (
    "calls", "lookups", "hits", "misses", "fetched", "overflow_routes", "evictions",
    "invalid_routes", "pf_requests", "pf_invalid", "pf_resident", "pf_filled",
    "pf_dropped_guard", "pf_no_victim", "pf_evictions", "status_bits",
)


class moe_stats(C.Structure):
    _fields_ = [(f, C.c_uint64) for f in STAT_FIELDS]

    def as_dict(self) -> dict:
        return {f: int(getattr(self, f)) for f in STAT_FIELDS}


class moe_views(C.Structure):
    _fields_ = [(f, C.c_void_p) for f in (
        "map", "slot_key", "stamp", "pinned", "clock", "decode_freq", "demand_freq",
        "last_demand", "stats", "plan_demand", "plan_prefetch", "groups")] + [("n_pools", C.c_int)]


_vp, _i, _u = C.c_void_p, C.c_int, C.c_uint
_SIGS = {
    "moe_cache_create": [C.POINTER(moe_cache_desc), C.POINTER(C.c_void_p)],
    "moe_cache_destroy": [_vp],
    "moe_cache_prefill": [_vp, _i, _vp, _i, _vp],
    "moe_cache_pin": [_vp, _i, _i, _i, _vp],
    "moe_admit": [_vp, _i, _vp, _vp, _i, _i, _vp],
    "moe_prefetch": [_vp, _i, _vp, _i, _vp],
    "moe_gather_missing": [_vp, _i, _vp],
    "moe_rollback_plan": [_vp, _i, _vp],
    "moe_routed_experts": [_vp, _i, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp],
    "moe_routed_experts_noalloc": [_i, _i, _i, _vp, C.c_size_t, _i, _vp, _vp, _vp, _i, _i, _vp,
                                   _vp, _vp],
    "moe_decode_layer": [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _vp,
                         _vp, _u],
    "moe_read_stats": [_vp, _i, C.POINTER(moe_stats)],
    "moe_device_views": [_vp, C.POINTER(moe_views)],
    "moe_cache_fail_next_gather": [_vp, _i],
    "moe_cache_set_wide_path": [_vp, _i],
    "moe_hybrid_start": [_vp, _i],
    "moe_hybrid_stop": [_vp],
    "moe_hybrid_counters": [_vp, _vp],
    "moe_hybrid_pause": [_vp, _i],
    "moe_schedule_trace": [_i, _i, _i, _i, _i, _i, _i, _vp, _i],
    "moe_decode_layer_plan": [_vp, _i, _i, _i, _i, _u, _vp, _i],
    "moe_lookahead_predict": [_vp, _vp, _vp, _i, _i, _vp, _vp],
    "moe_hybrid_selftest": [_i, _i, _i, _vp, _i, _i, _i, _i, _i, _u, _vp],
    "moe_cpu_experts": [_i, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _vp],
    "moe_strerror": [_i],
    "moe_last_cuda_error": [],
    "moe_abi_version": [],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = C.c_char_p if _name in ("moe_strerror", "moe_last_cuda_error") else C.c_int


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        msg = _lib.moe_strerror(code).decode()
        if code == MOE_ERR_CUDA or code == MOE_ERR_CONFIG:
            extra = _lib.moe_last_cuda_error().decode()
            if extra:
                msg += f" ({extra})"
        super().__init__(f"{fn}: {msg} [{code}]")


def _check(fn: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def _ptr(t) -> int | None:
    """Address of a tensor / array, an int address, or None (NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(s) -> int | None:
    """cudaStream_t of a torch stream; None means torch's current stream."""
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def abi_version() -> int:
    return _lib.moe_abi_version()


def moe_strerror(code: int) -> str:
    return _lib.moe_strerror(code).decode()


def moe_cache_create(desc: moe_cache_desc) -> int:
    h = C.c_void_p()
    _check("moe_cache_create", _lib.moe_cache_create(C.byref(desc), C.byref(h)))
    return h.value


def moe_cache_destroy(cache: int) -> None:
    _check("moe_cache_destroy", _lib.moe_cache_destroy(cache))


def moe_cache_prefill(cache: int, layer: int, h_ids, n: int, stream=None) -> None:
    _check("moe_cache_prefill", _lib.moe_cache_prefill(cache, layer, _ptr(h_ids), n, _stream(stream)))


def moe_cache_pin(cache: int, layer: int, slot: int, pinned: int, stream=None) -> None:
    _check("moe_cache_pin", _lib.moe_cache_pin(cache, layer, slot, pinned, _stream(stream)))


def moe_admit(cache: int, layer: int, d_ids, d_slot_ids, n_routes: int, fetch_cap: int = -1,
              stream=None) -> None:
    _check("moe_admit", _lib.moe_admit(cache, layer, _ptr(d_ids), _ptr(d_slot_ids), n_routes,
                                       fetch_cap, _stream(stream)))


def moe_prefetch(cache: int, layer: int, d_pred, n: int, stream=None) -> None:
    _check("moe_prefetch", _lib.moe_prefetch(cache, layer, _ptr(d_pred), n, _stream(stream)))


def moe_lookahead_predict(cache: int, d_x, d_router, n_rows: int, k_pred: int, d_pred,
                          stream=None) -> None:
    """Predicted ids of the next layer (see moe_cache.h)."""
    _check("moe_lookahead_predict", _lib.moe_lookahead_predict(
        cache, _ptr(d_x), _ptr(d_router), n_rows, k_pred, _ptr(d_pred), _stream(stream)))


def moe_gather_missing(cache: int, which: int = MOE_PLAN_DEMAND, stream=None) -> None:
    _check("moe_gather_missing", _lib.moe_gather_missing(cache, which, _stream(stream)))


def moe_rollback_plan(cache: int, which: int = MOE_PLAN_DEMAND, stream=None) -> None:
    _check("moe_rollback_plan", _lib.moe_rollback_plan(cache, which, _stream(stream)))


def moe_routed_experts(cache: int, layer: int, d_x, d_slot_ids, d_w, n_rows: int, k: int,
                       d_shared_blob, d_shared_gate, d_out, stream=None) -> None:
    _check("moe_routed_experts", _lib.moe_routed_experts(
        cache, layer, _ptr(d_x), _ptr(d_slot_ids), _ptr(d_w), n_rows, k, _ptr(d_shared_blob),
        _ptr(d_shared_gate), _ptr(d_out), _stream(stream)))


def moe_routed_experts_noalloc(wfmt: int, hidden: int, inter: int, d_slots, slot_stride: int,
                               n_slots: int, d_x, d_slot_ids, d_w, n_rows: int, k: int, d_out,
                               d_status=None, stream=None) -> None:
    """Routed FFNs + combine over a caller-owned slot pool; allocates nothing
    (scratch is a fixed 1 MiB device array, see include/moe_cache.h)."""
    _check("moe_routed_experts_noalloc", _lib.moe_routed_experts_noalloc(
        wfmt, hidden, inter, _ptr(d_slots), slot_stride, n_slots, _ptr(d_x), _ptr(d_slot_ids),
        _ptr(d_w), n_rows, k, _ptr(d_out), _ptr(d_status), _stream(stream)))


def moe_decode_layer(cache: int, layer: int, d_x, d_ids, d_w, d_slot_ids, n_rows: int, k: int,
                     fetch_cap: int, d_pred, n_pred: int, d_shared_blob, d_shared_gate, d_out,
                     compute_stream=None, side_stream=None, flags: int = MOE_OVERLAP) -> None:
    _check("moe_decode_layer", _lib.moe_decode_layer(
        cache, layer, _ptr(d_x), _ptr(d_ids), _ptr(d_w), _ptr(d_slot_ids), n_rows, k, fetch_cap,
        _ptr(d_pred), n_pred, _ptr(d_shared_blob), _ptr(d_shared_gate), _ptr(d_out),
        _stream(compute_stream), None if side_stream is None else _stream(side_stream), flags))


def moe_read_stats(cache: int, layer: int) -> dict:
    st = moe_stats()
    _check("moe_read_stats", _lib.moe_read_stats(cache, layer, C.byref(st)))
    return st.as_dict()


def moe_device_views(cache: int) -> moe_views:
    v = moe_views()
    _check("moe_device_views", _lib.moe_device_views(cache, C.byref(v)))
    return v


def moe_cache_fail_next_gather(cache: int, n: int = 1) -> None:
    _check("moe_cache_fail_next_gather", _lib.moe_cache_fail_next_gather(cache, n))


def moe_cache_set_wide_path(cache: int, mode: int) -> None:
    """MOE_WIDE_AUTO, MOE_WIDE_CUDA_CORES or MOE_WIDE_TENSOR_CORES: which
    kernels run wide steps' routed experts (see moe_cache.h)."""
    _check("moe_cache_set_wide_path", _lib.moe_cache_set_wide_path(cache, int(mode)))


def moe_hybrid_start(cache: int, n_threads: int) -> None:
    _check("moe_hybrid_start", _lib.moe_hybrid_start(cache, n_threads))


def moe_hybrid_stop(cache: int) -> None:
    _check("moe_hybrid_stop", _lib.moe_hybrid_stop(cache))


def moe_hybrid_pause(cache: int, paused: bool) -> None:
    _check("moe_hybrid_pause", _lib.moe_hybrid_pause(cache, int(paused)))


def moe_hybrid_selftest(wfmt: int, hidden: int, inter: int, blob_ptrs, max_rows: int, k: int,
                        n_threads: int, n_jobs: int, seed: int = 0) -> int:
    """Host-only stress test of the executor's job protocol; returns the number
    of jobs whose answer differed from moe_cpu_experts (see moe_cache.h)."""
    import numpy as np
    ptrs = np.ascontiguousarray(np.asarray(blob_ptrs, dtype=np.uint64))
    bad = C.c_longlong(0)
    _check("moe_hybrid_selftest", _lib.moe_hybrid_selftest(
        wfmt, hidden, inter, ptrs.ctypes.data, len(ptrs), max_rows, k, n_threads, n_jobs, seed,
        C.byref(bad)))
    return bad.value


def moe_schedule_trace(one_launch: bool = False, fused: bool = False, overlap: bool = True,
                       pf: bool = False, shared: bool = False, hybrid: bool = False,
                       fail_at: int = -1) -> tuple[int, list[str]]:
    """(return code, ["c:admit", "s:gather_demand", ...]) of a layer plan (see moe_cache.h)."""
    buf = C.create_string_buffer(4096)
    rc = _lib.moe_schedule_trace(int(one_launch), int(fused), int(overlap), int(pf), int(shared),
                                 int(hybrid), fail_at, buf, len(buf))
    return rc, buf.value.decode().split()


def moe_decode_layer_plan(cache: int, n_rows: int, k: int, shared: bool = False,
                          pf: bool = False, flags: int = 0) -> list[str]:
    """The operations moe_decode_layer would enqueue on this cache for the
    shape and flags, as moe_schedule_trace tokens (see moe_cache.h)."""
    buf = C.create_string_buffer(4096)
    _check("moe_decode_layer_plan", _lib.moe_decode_layer_plan(
        cache, n_rows, k, int(shared), int(pf), flags, buf, len(buf)))
    return buf.value.decode().split()


def moe_hybrid_counters(cache: int) -> dict:
    import numpy as np
    out = np.zeros(4, np.uint64)
    _check("moe_hybrid_counters", _lib.moe_hybrid_counters(cache, out.ctypes.data))
    return {"jobs": int(out[0]), "cpu_routes": int(out[1]), "busy_ns": int(out[2]),
            "busy_route_ns": int(out[3])}


def moe_cpu_experts(wfmt: int, hidden: int, inter: int, blob_ptrs, x_bf16, ids, slot_ids, w,
                    n_threads: int = 1):
    """The hybrid executor's CPU partial as a host call: ``blob_ptrs`` [E] host
    blob addresses of one layer, ``x_bf16`` uint16 [B, H], ``ids`` /
    ``slot_ids`` int32 and ``w`` float32 [B, k]; returns float32 [B, H]."""
    import numpy as np
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    B = x.shape[0]
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(B, -1)
    k = ids.shape[1]
    slot_ids = np.ascontiguousarray(slot_ids, dtype=np.int32).reshape(B, k)
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(B, k)
    ptrs = np.ascontiguousarray(np.asarray(blob_ptrs, dtype=np.uint64))
    out = np.empty((B, hidden), np.float32)
    _check("moe_cpu_experts", _lib.moe_cpu_experts(
        wfmt, hidden, inter, ptrs.ctypes.data, len(ptrs), x.ctypes.data, ids.ctypes.data,
        slot_ids.ctypes.data, w.ctypes.data, B, k, n_threads, out.ctypes.data))
    return out


def blob_bytes(wfmt: int, hidden: int, inter: int) -> int:
    """Bytes of one expert blob in the layout of moe_cache.h."""
    if wfmt == MOE_W_BF16:
        return 6 * hidden * inter
    if wfmt == MOE_W_MXFP4:
        return 3 * hidden * inter // 2 + 3 * hidden * inter // 32
    if wfmt == MOE_W_Q4_0:
        return 3 * hidden * inter // 2 + 3 * hidden * inter // 16
    return 3 * hidden * inter // 2 + 3 * hidden * inter // 16 + 16


def split_routes(ids, slot_ids, weights):
    """Complementary CPU / GPU views of a hybrid step, as the hybrid executor
    of FreeToken PR #491 ("refactor(moe): extract hybrid decode
    orchestration", section 5) hands them to its two sides: the CPU side gets
    the original id where the cache returned -1 (else -1), the GPU side the
    slot id with -1 replaced by 0 and that route's weight set to 0.  The GPU
    kernels of this library skip -1 routes directly and do not need the GPU
    view; it is provided for callers that feed another kernel."""
    import torch
    ids = torch.as_tensor(ids)
    slot_ids = torch.as_tensor(slot_ids)
    weights = torch.as_tensor(weights)
    cpu = slot_ids < 0
    cpu_ids = torch.where(cpu, ids, torch.full_like(ids, -1))
    gpu_slots = torch.where(cpu, torch.zeros_like(slot_ids), slot_ids)
    gpu_w = torch.where(cpu, torch.zeros_like(weights), weights)
    return cpu_ids, gpu_slots, gpu_w


class SlotCache:
    """Owner of one ``moe_cache`` plus the buffers it points at.

    ``slot_storage`` (device tensor) and ``host_blob_ptrs`` (addresses of
    pinned host blobs) are kept referenced so they outlive the cache."""

    def __init__(self, *, n_layers: int, n_experts: int, n_slots: int, pool_mode: int,
                 hidden: int = 0, inter: int = 0, wfmt: int = MOE_W_BF16, shared_inter: int = 0,
                 slot_storage=None, slot_stride: int = 0, host_blob_ptrs=None,
                 max_routes: int = 1, max_rows: int = 1, max_pred: int = 0, gather_ctas: int = 0,
                 keepalive=()):
        import numpy as np
        self._keep = [slot_storage, *keepalive]
        d = moe_cache_desc()
        d.n_layers, d.n_experts, d.n_slots, d.pool_mode = n_layers, n_experts, n_slots, pool_mode
        d.hidden, d.inter, d.wfmt, d.shared_inter = hidden, inter, wfmt, shared_inter
        d.slot_bytes = blob_bytes(wfmt, hidden, inter) if (slot_storage is not None and hidden) else 0
        d.slot_stride = slot_stride
        d.slot_storage = _ptr(slot_storage)
        if host_blob_ptrs is not None:
            arr = np.ascontiguousarray(np.asarray(host_blob_ptrs, dtype=np.uint64))
            self._keep.append(arr)
            d.host_experts = arr.ctypes.data
        d.max_routes, d.max_rows, d.max_pred, d.gather_ctas = max_routes, max_rows, max_pred, gather_ctas
        self.desc = d
        self.n_pools = n_layers if pool_mode == MOE_POOL_PER_LAYER else 1
        self.handle = moe_cache_create(d)

    def close(self) -> None:
        if getattr(self, "handle", None):
            moe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stats(self, layer: int) -> dict:
        return moe_read_stats(self.handle, layer)

    def views(self) -> moe_views:
        return moe_device_views(self.handle)
