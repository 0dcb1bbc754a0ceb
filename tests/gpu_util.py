"""Helpers for the GPU tests: a workload's cache on the device beside its
oracle twin, and copies of the device state for bit-exact comparison."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

TOL = {synth.FMT_NVFP4: (2e-2, 1e-2), synth.FMT_MXFP4: (2e-2, 1e-2), synth.FMT_Q4_0: (2e-2, 1e-2),
       synth.FMT_BF16: (5e-3, 1e-2)}  # (atol, rtol); the 4-bit formats take the fp4 tolerance


class _Dev:
    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3}


def dev_copy(ptr: int, n: int, dtype) -> np.ndarray:
    """Host copy of n elements of a device array owned by the library."""
    dt = np.dtype(dtype)
    if n == 0:
        return np.zeros(0, dt)
    t = torch.as_tensor(_Dev(ptr, n, dt.str), device="cuda")
    return t.cpu().numpy().copy()


def gpu_state(sc) -> dict:
    """Copies of the cache state behind a SlotCache (same keys as OracleCache.state())."""
    torch.cuda.synchronize()
    v = sc.views()
    d = sc.desc
    K = d.n_layers * d.n_experts
    P = sc.n_pools * d.n_slots
    return {
        "map": dev_copy(v.map, K, np.int32),
        "slot_key": dev_copy(v.slot_key, P, np.int32),
        "stamp": dev_copy(v.stamp, P, np.uint64),
        "pinned": dev_copy(v.pinned, P, np.uint8),
        "clock": dev_copy(v.clock, sc.n_pools, np.uint64),
        "decode_freq": dev_copy(v.decode_freq, K, np.uint32),
        "demand_freq": dev_copy(v.demand_freq, K, np.uint32),
        "last_demand": dev_copy(v.last_demand, K, np.uint64),
    }


def gpu_plan(sc, which: int = 0) -> list[tuple[int, int, int]]:
    v = sc.views()
    ptr = v.plan_demand if which == 0 else v.plan_prefetch
    n = int(dev_copy(ptr, 1, np.int32)[0])
    a = dev_copy(ptr, 1 + 3 * n, np.int32)
    return [tuple(int(x) for x in a[1 + 3 * i:4 + 3 * i]) for i in range(n)]


def assert_state_equal(sc, oc: oracle.OracleCache, layers=None, what="") -> None:
    g = gpu_state(sc)
    o = oc.state()
    for k in g:
        if not np.array_equal(g[k], o[k]):
            bad = np.nonzero(g[k] != o[k])[0][:8]
            raise AssertionError(f"{what} state '{k}' differs at {bad.tolist()}: "
                                 f"gpu {g[k][bad].tolist()} oracle {o[k][bad].tolist()}")
    for layer in (range(oc.L) if layers is None else layers):
        gs, os_ = sc.stats(layer), oc.stats(layer)
        assert gs == os_, f"{what} layer {layer} stats: gpu {gs} oracle {os_}"


def assert_close(out_bf16: torch.Tensor, ref: np.ndarray, fmt: int, what="") -> dict:
    """Elementwise |gpu - ref| <= atol + rtol*|ref|; returns max-abs / max-rel."""
    atol, rtol = TOL[fmt]
    got = out_bf16.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    err = np.abs(got - ref)
    ok = err <= atol + rtol * np.abs(ref)
    rel = err / np.maximum(np.abs(ref), 1e-30)
    info = {"max_abs": float(err.max()) if err.size else 0.0,
            "max_rel": float(rel.max()) if rel.size else 0.0}
    if not ok.all():
        i = np.argwhere(~ok)[:5].tolist()
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside atol={atol} "
                             f"rtol={rtol}; first {i}; {info}")
    return info


class Rig:
    """A workload's slot cache on cuda:0 with its pinned host blobs, plus the
    oracle cache fed the same calls."""

    def __init__(self, w: synth.Workload, *, storage: bool = True, max_routes: int | None = None,
                 max_rows: int | None = None, max_pred: int | None = None, blobs=None,
                 gather_ctas: int = 0):
        import expert_slot_cache_lru_gb300 as m
        self.m = m
        self.w = w
        self.P = w.n_layers if w.per_layer_pools else 1
        compute = storage and w.hidden > 0
        self.blobs = (blobs or synth.HostBlobs(w, pinned=True)) if compute else None
        self.storage = None
        stride = 0
        if compute:
            stride = self.blobs.stride
            self.storage = torch.empty(self.P * w.n_slots * stride, dtype=torch.uint8, device="cuda")
        mr = max_routes or max(w.routes, max(w.batches or (1,)) * w.top_k, 1)
        self.sc = m.SlotCache(
            n_layers=w.n_layers, n_experts=w.n_experts, n_slots=w.n_slots,
            pool_mode=m.MOE_POOL_PER_LAYER if w.per_layer_pools else m.MOE_POOL_SHARED,
            hidden=w.hidden if compute else 0, inter=w.inter if compute else 0, wfmt=w.fmt,
            shared_inter=w.shared_inter if compute else 0, slot_storage=self.storage,
            slot_stride=stride, host_blob_ptrs=self.blobs.addrs() if compute else None,
            max_routes=mr, max_rows=max_rows or max(w.batch, 1),
            max_pred=w.n_pred if max_pred is None else max_pred, gather_ctas=gather_ctas)
        self.oc = oracle.OracleCache(w.n_layers, w.n_experts, w.n_slots, w.per_layer_pools)
        # one shared expert per layer (host copy for the oracle, device copy for the GPU)
        self.h_shared = [(None, None)] * w.n_layers
        self.d_shared = [(None, None)] * w.n_layers
        if compute and w.shared_inter:
            self.h_shared = [synth.make_shared(w, l) for l in range(w.n_layers)]
            self.d_shared = [(torch.from_numpy(b).cuda(), torch.from_numpy(g.view(np.int16)).cuda())
                             for b, g in self.h_shared]

    def prefill(self, layer: int, ids) -> None:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        self.m.moe_cache_prefill(self.sc.handle, layer, ids, len(ids))
        self.oc.prefill(layer, ids)

    def slot_bytes(self, layer: int, slot: int) -> np.ndarray:
        p = layer if self.w.per_layer_pools else 0
        off = (p * self.w.n_slots + slot) * self.blobs.stride
        return self.storage[off:off + self.blobs.nbytes].cpu().numpy()

    def oracle_layer(self, layer: int, x: np.ndarray, ids: np.ndarray, wts: np.ndarray,
                     mask=None) -> np.ndarray:
        w = self.w
        return oracle.layer(w.fmt, [self.blobs.addr(layer * w.n_experts + e) for e in range(w.n_experts)],
                            w.n_experts, w.hidden, w.inter, x, ids, wts, mask=mask,
                            shared_blob=self.h_shared[layer][0], shared_inter=w.shared_inter,
                            shared_gate_w=self.h_shared[layer][1])
