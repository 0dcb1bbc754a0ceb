"""CPU oracle of the offloaded-MoE slot cache and layer math (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``expert_slot_cache_lru_gb300``) never imports it and shares no code with it.

The model itself is ``oracle.cpp`` (plain single-threaded C++); this module
only loads it and converts arguments.  See ``oracle.h`` for the citations of
each function.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = [os.path.join(_HERE, "oracle.cpp")]
_HDR = os.path.join(_HERE, "oracle.h")

STAT_FIELDS = (
    "calls", "lookups", "hits", "misses", "fetched", "overflow_routes", "evictions",
    "invalid_routes", "pf_requests", "pf_invalid", "pf_resident", "pf_filled",
    "pf_dropped_guard", "pf_no_victim", "pf_evictions", "status_bits",
)
STATUS_INVALID_ID = 1
STATUS_CAPACITY = 2
FMT_BF16 = 0
FMT_NVFP4 = 1
FMT_MXFP4 = 2
FMT_Q4_0 = 3


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (plain C++17, -O2, no CPU-specific flags)."""
    newest = max(os.path.getmtime(p) for p in _SRC + [_HDR])
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-Wall", "-o", tmp] + _SRC
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_SO)
        p = C.c_void_p
        i32p = C.POINTER(C.c_int32)
        u64p = C.POINTER(C.c_uint64)
        L.oc_create.restype = p
        L.oc_create.argtypes = [C.c_int] * 4
        L.oc_destroy.argtypes = [p]
        L.oc_prefill.argtypes = [p, C.c_int, i32p, C.c_int]
        L.oc_pin.argtypes = [p, C.c_int, C.c_int, C.c_int]
        L.oc_admit.argtypes = [p, C.c_int, i32p, C.c_int, C.c_int, C.c_int, i32p, i32p, i32p, i32p]
        L.oc_prefetch.argtypes = [p, C.c_int, i32p, C.c_int, i32p]
        L.oc_rollback.argtypes = [p, i32p]
        L.oc_stats.argtypes = [p, C.c_int, u64p]
        L.oc_n_pools.argtypes = [p]
        L.oc_state.argtypes = [p] + [C.c_void_p] * 8
        L.oc_lru_order.argtypes = [p, C.c_int, i32p]
        L.om_e2m1.restype = C.c_double
        L.om_e2m1.argtypes = [C.c_int]
        L.om_e4m3.restype = C.c_double
        L.om_e4m3.argtypes = [C.c_int]
        L.om_e8m0.restype = C.c_double
        L.om_e8m0.argtypes = [C.c_int]
        L.om_f16.restype = C.c_double
        L.om_f16.argtypes = [C.c_uint16]
        L.om_bf16.restype = C.c_double
        L.om_bf16.argtypes = [C.c_uint16]
        L.om_blob_bytes.restype = C.c_uint64
        L.om_blob_bytes.argtypes = [C.c_int, C.c_int, C.c_int]
        L.om_dequant.argtypes = [C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p]
        L.om_expert_ffn.argtypes = [C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        L.om_lookahead_predict.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                           C.c_int, C.c_void_p, C.c_void_p]
        L.om_layer.argtypes = [C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                               C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
        _lib = L
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray, t=C.c_int32):
    return a.ctypes.data_as(C.POINTER(t))


def parse_plan(buf: np.ndarray) -> list[tuple[int, int, int]]:
    n = int(buf[0])
    return [tuple(int(v) for v in buf[1 + 3 * i: 4 + 3 * i]) for i in range(n)]


def parse_groups(buf: np.ndarray) -> list[tuple[int, list[int]]]:
    G = int(buf[0])
    slots = buf[1:1 + G]
    starts = buf[1 + G:2 + 2 * G]
    lst = buf[2 + 2 * G:]
    return [(int(slots[g]), [int(r) for r in lst[starts[g]:starts[g + 1]]]) for g in range(G)]


class OracleCache:
    """The slot cache, admission and prefetch, one explicit LRU list per pool."""

    def __init__(self, n_layers: int, n_experts: int, n_slots: int, per_layer: bool = False):
        self.L, self.E, self.S = n_layers, n_experts, n_slots
        self.per_layer = per_layer
        self._h = lib().oc_create(n_layers, n_experts, n_slots, 1 if per_layer else 0)
        if not self._h:
            raise ValueError("oc_create: bad arguments")
        self.n_pools = lib().oc_n_pools(self._h)

    def __del__(self):
        if getattr(self, "_h", None):
            lib().oc_destroy(self._h)
            self._h = None

    def prefill(self, layer: int, ids) -> None:
        a = _i32(ids)
        rc = lib().oc_prefill(self._h, layer, _ptr(a), len(a))
        if rc != 0:
            raise ValueError(f"oc_prefill rc={rc}")

    def pin(self, layer: int, slot: int, pinned: bool = True) -> None:
        if lib().oc_pin(self._h, layer, slot, int(bool(pinned))) != 0:
            raise ValueError("oc_pin: bad arguments")

    def admit(self, layer: int, ids, cap: int = -1, split_width: int = 0) -> dict:
        a = _i32(ids).ravel()
        R = len(a)
        out = np.empty(max(R, 1), np.int32)
        plan = np.zeros(1 + 3 * max(R, 1), np.int32)
        groups = np.zeros(2 + 3 * max(R, 1), np.int32)
        widths = np.zeros(R + 2, np.int32)
        rc = lib().oc_admit(self._h, layer, _ptr(a), R, cap, split_width, _ptr(out), _ptr(plan),
                            _ptr(groups), _ptr(widths))
        if rc != 0:
            raise ValueError(f"oc_admit rc={rc}")
        return {
            "slots": out[:R].copy(),
            "plan": parse_plan(plan),
            "groups": parse_groups(groups),
            "widths": [int(w) for w in widths[1:1 + widths[0]]],
        }

    def prefetch(self, layer: int, pred) -> list[tuple[int, int, int]]:
        a = _i32(pred).ravel()
        plan = np.zeros(1 + 3 * max(len(a), 1), np.int32)
        if lib().oc_prefetch(self._h, layer, _ptr(a), len(a), _ptr(plan)) != 0:
            raise ValueError("oc_prefetch: bad arguments")
        return parse_plan(plan)

    def rollback(self, plan: list[tuple[int, int, int]]) -> None:
        buf = np.zeros(1 + 3 * max(len(plan), 1), np.int32)
        buf[0] = len(plan)
        for i, t in enumerate(plan):
            buf[1 + 3 * i:4 + 3 * i] = t
        if lib().oc_rollback(self._h, _ptr(buf)) != 0:
            raise ValueError("oc_rollback: bad plan")

    def stats(self, layer: int) -> dict:
        out = np.zeros(len(STAT_FIELDS), np.uint64)
        if lib().oc_stats(self._h, layer, _ptr(out, C.c_uint64)) != 0:
            raise ValueError("oc_stats: bad layer")
        return {k: int(v) for k, v in zip(STAT_FIELDS, out)}

    def state(self) -> dict:
        K = self.L * self.E
        P = self.n_pools * self.S
        st = {
            "map": np.zeros(K, np.int32),
            "slot_key": np.zeros(P, np.int32),
            "stamp": np.zeros(P, np.uint64),
            "pinned": np.zeros(P, np.uint8),
            "clock": np.zeros(self.n_pools, np.uint64),
            "decode_freq": np.zeros(K, np.uint32),
            "demand_freq": np.zeros(K, np.uint32),
            "last_demand": np.zeros(K, np.uint64),
        }
        order = ["map", "slot_key", "stamp", "pinned", "clock", "decode_freq", "demand_freq",
                 "last_demand"]
        lib().oc_state(self._h, *[C.c_void_p(st[k].ctypes.data) for k in order])
        return st

    def lru_order(self, pool: int = 0) -> list[int]:
        out = np.zeros(max(self.S, 1), np.int32)
        n = lib().oc_lru_order(self._h, pool, _ptr(out))
        return [int(v) for v in out[:n]]


# ---------------------------------------------------------------- layer math

def e2m1(code: int) -> float:
    return lib().om_e2m1(code)


def e4m3(byte: int) -> float:
    return lib().om_e4m3(byte)


def e8m0(byte: int) -> float:
    return lib().om_e8m0(byte)


def f16(bits: int) -> float:
    return lib().om_f16(bits)


def bf16(bits: int) -> float:
    return lib().om_bf16(bits)


def blob_bytes(fmt: int, hidden: int, inter: int) -> int:
    return int(lib().om_blob_bytes(fmt, hidden, inter))


def _addr(a) -> int:
    """Address of a numpy array or a (pinned) CPU torch tensor."""
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        assert not a.is_cuda and a.is_contiguous()
        return a.data_ptr()
    if isinstance(a, int):
        return a
    raise TypeError(type(a))


def dequant(fmt: int, blob, hidden: int, inter: int, which: int) -> np.ndarray:
    rows, cols = (hidden, inter) if which == 2 else (inter, hidden)
    out = np.empty((rows, cols), np.float64)
    if lib().om_dequant(fmt, _addr(blob), hidden, inter, which, out.ctypes.data) != 0:
        raise ValueError("om_dequant: bad arguments")
    return out


def expert_ffn(fmt: int, blob, hidden: int, inter: int, x_bf16: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    y = np.empty(hidden, np.float64)
    if lib().om_expert_ffn(fmt, _addr(blob), hidden, inter, x.ctypes.data, y.ctypes.data) != 0:
        raise ValueError("om_expert_ffn: bad arguments")
    return y


def layer(fmt: int, blobs, n_experts: int, hidden: int, inter: int, x_bf16, ids, w,
          mask=None, shared_blob=None, shared_inter: int = 0, shared_gate_w=None) -> np.ndarray:
    """fp64 layer output [B, H]; ``blobs[e]`` is expert e's blob (array, tensor or address)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    B = x.shape[0]
    ids = _i32(ids).reshape(B, -1)
    k = ids.shape[1]
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(B, k)
    ptrs = (C.c_void_p * n_experts)(*[_addr(b) if b is not None else 0 for b in blobs])
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8).reshape(B, k)
    gw = None if shared_gate_w is None else np.ascontiguousarray(shared_gate_w, dtype=np.uint16)
    out = np.empty((B, hidden), np.float64)
    rc = lib().om_layer(fmt, ptrs, n_experts, hidden, inter, x.ctypes.data, ids.ctypes.data,
                        w.ctypes.data, None if m is None else m.ctypes.data, B, k,
                        None if shared_blob is None else _addr(shared_blob), shared_inter,
                        None if gw is None else gw.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"om_layer rc={rc}")
    return out


def lookahead_predict(x_bf16, router_bf16, k: int) -> tuple[np.ndarray, np.ndarray]:
    """(pred int32 [B, k], z fp64 [B, E]): layer L+1's router on layer L's hidden
    state, each row's k largest logits (see oracle.h)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    r = np.ascontiguousarray(router_bf16, dtype=np.uint16)
    B, H = x.shape
    E = r.shape[0]
    if r.shape[1] != H:
        raise ValueError("router and x widths differ")
    pred = np.empty((B, k), np.int32)
    z = np.empty((B, E), np.float64)
    rc = lib().om_lookahead_predict(x.ctypes.data, r.ctypes.data, B, E, H, k, pred.ctypes.data,
                                    z.ctypes.data)
    if rc != 0:
        raise ValueError(f"om_lookahead_predict rc={rc}")
    return pred, z
