"""Benchmark of one GPU's offloaded-MoE decode on the Qwen3-MoE-like workload.

A step is one decode token through all 40 MoE layers: per layer the slot-cache
admission, the miss gather from pinned host memory (side stream, event
fork/join), the sigmoid-gated shared expert, the routed NVFP4 expert FFNs and
the weighted combine -- the whole layer captured as one CUDA graph per token,
as in FreeToken issue #753 ("[Perf] Offloaded decode: overlap the
expert-miss gather with the same layer's shared expert, event-ordered inside
the CUDA graph").  Inputs are synthetic (synth/: Zipf(1.1) routing with
temporal reuse, ~28 misses per token on the 3,164-slot LRU cache, random NVFP4
weights); the cache is warmed with 64 tokens before the warm-up steps.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the slow, obviously-correct model the tests compare against).
With torchrun, N>1 ranks run independent replicas (one GPU each; there is
no collective on the data path) and ``value`` is the sum of their tokens over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes as C
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "admission µs/layer vs routes; offloaded MoE decode tok/s; GEMV GB/s vs HBM peak"
WORKLOAD = "qwen3moe_decode"
WARM_TOKENS = 64


# ---------------------------------------------------------------- environment

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# DRAM bytes per launch of the routed FFN kernel from an ncu capture, kept
# beside the kernel source's hash: the figure is reported only while the
# source is unchanged since the capture.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ffn_fused_kernel_routed_traffic.txt")
FFN_SOURCE = os.path.join(ROOT, "expert_slot_cache_lru_gb300", "csrc", "ffn_stream.cu")


def replica_rate(local_s: float, units: int, ws: int, device="cpu") -> tuple[float, float]:
    """Whole-job rate of ws independent replicas: every rank processed `units`
    in `local_s` seconds; the job took the slowest rank's time (max over
    ranks), so the rate is ws * units / max_s.  Returns (rate, max_s)."""
    if ws > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([local_s], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        local_s = float(t.item())
    return ws * units / local_s, local_s


def source_hash(path: str) -> str:
    import hashlib
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def routed_traffic() -> dict | None:
    """{"bytes_per_launch": ..., "source": ...} from the traffic file, or None
    when it is missing or the kernel source changed since the capture."""
    try:
        kv = dict(line.split("=", 1) for line in open(TRAFFIC_FILE).read().split("\n")
                  if "=" in line and not line.startswith("#"))
        if kv.get("source_sha256_16") != source_hash(FFN_SOURCE):
            return None
        return {"bytes_per_launch": float(kv["dram_bytes_per_launch"]),
                "source": os.path.relpath(TRAFFIC_FILE, ROOT)}
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "_source": "fallback"}


def host_numa(addr: int, dev: int) -> dict:
    """Where the pinned host blobs live and which node the GPU hangs off:
    the NUMA nodes the host shows, the GPU's PCI numa_node, and the per-node
    page counts of the memory mapping that holds `addr` (/proc/self/numa_maps)."""
    out = {}
    try:
        out["host_nodes"] = sorted(n for n in os.listdir("/sys/devices/system/node")
                                   if n.startswith("node"))
    except OSError:
        out["host_nodes"] = None
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        bus = (f"{getattr(p, 'pci_domain_id', 0):04x}:{getattr(p, 'pci_bus_id', 0):02x}:"
               f"{getattr(p, 'pci_device_id', 0):02x}.0")
        out["gpu_numa_node"] = int(open(f"/sys/bus/pci/devices/{bus}/numa_node").read())
    except Exception:
        out["gpu_numa_node"] = None
    try:
        for line in open("/proc/self/numa_maps"):
            f = line.split()
            if f and int(f[0], 16) <= addr:
                best = f
        out["blob_mapping"] = " ".join(x for x in best[1:] if x.startswith(("N", "default", "bind",
                                                                            "interleave", "prefer")))
    except Exception:
        out["blob_mapping"] = None
    return out


class ClockSampler:
    """SM clock and clock-event reasons sampled through NVML (read-only)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str, index: int = 0, period_s: float = 0.005):
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self.err = None
        self._stop = threading.Event()
        self._period = period_s
        try:
            self.nvml = C.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            self.h = C.c_void_p()
            bus = pci_bus_id.encode()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(C.c_char_p(bus), C.byref(self.h)) != 0:
                if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, C.byref(self.h)) != 0:
                    raise RuntimeError("no NVML handle for " + pci_bus_id)
            mx = C.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, C.byref(mx)) == 0:
                self.max_mhz = mx.value
        except Exception as ex:  # pragma: no cover - depends on the machine
            self.err = str(ex)
            self.nvml = None

    def _run(self):
        clk = C.c_uint()
        rs = C.c_ulonglong()
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, C.byref(clk)) == 0 and \
                    get_reasons(self.h, C.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(self._period)

    def __enter__(self):
        if self.nvml:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.nvml:
            self._stop.set()
            self._t.join()

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "note": self.err or "no samples"}
        bits = 0
        for _, r in self.samples:
            bits |= r
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if bits & b],
                "samples": len(self.samples)}


# ---------------------------------------------------------------- native arm

class Decode:
    """The benchmark workload on one GPU: cache, inputs, one-token graph."""

    def __init__(self, dev: int, overlap: bool = True, warm_tokens: int = WARM_TOKENS,
                 total_tokens: int = 512, n_layers: int | None = None, n_slots: int | None = None,
                 fused: bool = True):
        import torch

        import expert_slot_cache_lru_gb300 as m
        import synth
        self.torch, self.m, self.synth = torch, m, synth
        torch.cuda.set_device(dev)
        w = synth.workloads()[WORKLOAD]
        if n_layers or n_slots:  # a smaller case of the same layer, for profiler captures
            w = synth.scaled(w, n_layers=n_layers or w.n_layers, n_slots=n_slots or w.n_slots)
        self.w = w
        self.overlap = overlap
        self.fused = fused
        t0 = time.time()
        self.blobs = synth.HostBlobs(w, pinned=True)
        self.setup_s = {"host_blobs": time.time() - t0}
        self.storage = torch.empty(w.n_slots * self.blobs.stride, dtype=torch.uint8, device="cuda")
        self.cache = m.SlotCache(
            n_layers=w.n_layers, n_experts=w.n_experts, n_slots=w.n_slots,
            pool_mode=m.MOE_POOL_SHARED, hidden=w.hidden, inter=w.inter, wfmt=w.fmt,
            shared_inter=w.shared_inter, slot_storage=self.storage, slot_stride=self.blobs.stride,
            host_blob_ptrs=self.blobs.addrs(), max_routes=w.routes, max_rows=w.batch)
        sh = [synth.make_shared(w, l) for l in range(w.n_layers)]
        self.shared = [(torch.from_numpy(b).cuda(), torch.from_numpy(g.view(np.int16)).cuda())
                       for b, g in sh]
        T = max(total_tokens, 1)
        ids, wts = synth.make_routing(synth.scaled(w, steps=min(T, w.steps)))
        self.T = ids.shape[0]
        x = np.stack([synth.make_hidden(w, t) for t in range(self.T)])  # [T, L, B, H]
        L, R = w.n_layers, w.routes
        # staged inputs (device and pinned host), one slice per token
        self.d_ids = torch.from_numpy(ids.reshape(self.T, L, R)).cuda()
        self.d_w = torch.from_numpy(wts.reshape(self.T, L, R)).cuda()
        self.d_x = torch.from_numpy(x.view(np.int16)).cuda()
        self.h_ids = torch.from_numpy(ids.reshape(self.T, L, R)).pin_memory()
        self.h_w = torch.from_numpy(wts.reshape(self.T, L, R)).pin_memory()
        self.h_x = torch.from_numpy(x.view(np.int16)).pin_memory()
        # the graph's fixed input / output buffers
        self.b_ids = torch.empty(L, R, dtype=torch.int32, device="cuda")
        self.b_w = torch.empty(L, R, dtype=torch.float32, device="cuda")
        self.b_x = torch.empty(L, w.batch, w.hidden, dtype=torch.int16, device="cuda")
        self.b_slots = torch.empty(L, R, dtype=torch.int32, device="cuda")
        self.b_out = torch.empty(L, w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
        self.h_out = torch.empty(L, w.batch, w.hidden, dtype=torch.bfloat16).pin_memory()
        self.cs = torch.cuda.Stream()
        self.side = torch.cuda.Stream()
        self.t = 0
        t0 = time.time()
        with torch.cuda.stream(self.cs):
            for _ in range(warm_tokens):  # eager warm-up of the cache
                self.load_device(self.t)
                self.enqueue()
                self.t += 1
        torch.cuda.synchronize()
        self.setup_s["warm_cache"] = time.time() - t0
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.cs):
            self.enqueue()
        torch.cuda.synchronize()

    def enqueue(self):
        m, w = self.m, self.w
        flags = (m.MOE_OVERLAP if self.overlap else 0) | (m.MOE_FUSED if self.fused else 0)
        for layer in range(w.n_layers):
            sb, sg = self.shared[layer]
            m.moe_decode_layer(self.cache.handle, layer, self.b_x[layer], self.b_ids[layer],
                               self.b_w[layer], self.b_slots[layer], w.batch, w.top_k, -1, None, 0,
                               sb, sg, self.b_out[layer], self.cs, self.side, flags)

    def load_device(self, t):
        t %= self.T
        self.b_ids.copy_(self.d_ids[t], non_blocking=True)
        self.b_w.copy_(self.d_w[t], non_blocking=True)
        self.b_x.copy_(self.d_x[t], non_blocking=True)

    def load_host(self, t):
        t %= self.T
        self.b_ids.copy_(self.h_ids[t], non_blocking=True)
        self.b_w.copy_(self.h_w[t], non_blocking=True)
        self.b_x.copy_(self.h_x[t], non_blocking=True)

    def step(self):
        """One token: its inputs into the graph's buffers (device to device), replay."""
        with self.torch.cuda.stream(self.cs):
            self.load_device(self.t)
            self.graph.replay()
        self.t += 1

    def step_e2e(self):
        """One token end to end: pinned host inputs -> device, replay, output -> pinned host."""
        with self.torch.cuda.stream(self.cs):
            self.load_host(self.t)
            self.graph.replay()
            self.h_out.copy_(self.b_out, non_blocking=True)
        self.cs.synchronize()
        self.t += 1

    def totals(self) -> dict:
        """Statistics summed over the layers (synchronises the device)."""
        tot = {}
        for layer in range(self.w.n_layers):
            for k, v in self.cache.stats(layer).items():
                tot[k] = tot.get(k, 0) + v
        return tot

    def layer_kernel_roofline(self, t_first: int, steps: int, ms: float, timed: dict,
                              hbm_gbs: float, gather_peak=None) -> dict:
        """The decode's own kernel (one launch per layer: admission, miss
        staging, shared and routed experts, combine), from the timed region:
        its average launch time is the timed region over steps x layers (the
        graph holds nothing else).  HBM algorithmic bytes per launch: each
        step's distinct experts' blobs (the misses read back from staging),
        the shared expert's blob, activations and ids; host-link bytes: the
        misses' blobs."""
        w = self.w
        L = w.n_layers
        ids = self.d_ids.cpu().numpy()
        hbm_bytes = 0
        for i in range(steps):
            t = (t_first + i) % self.T
            for layer in range(L):
                nd = len(set(int(v) for v in ids[t, layer] if 0 <= v < w.n_experts))
                hbm_bytes += ((nd + (1 if w.shared_inter else 0)) * w.blob_bytes +
                              w.batch * w.hidden * 2 * 2 + w.routes * 12)
        launches = steps * L
        per_launch_s = ms * 1e-3 / launches
        hbm_per = hbm_bytes / launches
        host_per = timed["fetched"] / L * w.blob_bytes
        return {"kernel": "ffn_fused_kernel<NVFP4, layerAdmit> (moe_decode_layer, MOE_FUSED: "
                          "the whole layer in one launch)",
                "bound": "hbm", "launches": launches, "avg_launch_us": round(per_launch_s * 1e6, 3),
                "bytes_per_launch": round(hbm_per), "achieved": round(hbm_per / per_launch_s / 1e9, 1),
                "peak": hbm_gbs, "unit": "GB/s",
                "frac": round(hbm_per / per_launch_s / 1e9 / hbm_gbs, 4),
                "host_link": {"bytes_per_launch": round(host_per),
                              "achieved": round(host_per / per_launch_s / 1e9, 1),
                              "unit": "GB/s", "peak": gather_peak, "frac": None}}

    def h2d_bytes(self) -> int:
        return (self.b_ids.numel() * 4 + self.b_w.numel() * 4 + self.b_x.numel() * 2)

    def d2h_bytes(self) -> int:
        return self.b_out.numel() * 2

    # ------------------------------------------------------------ sub-measurements

    def routed_gemv_roofline(self, steps: int) -> dict:
        """The routed expert GEMV (gate/up + down + combine, moe_routed_experts
        without the shared expert) for every layer of `steps` tokens, captured as
        a graph of back-to-back launches and timed with CUDA events on its
        stream.  Algorithmic bytes per launch: the distinct resident routes'
        expert blobs plus activations."""
        torch, m, w = self.torch, self.m, self.w
        L, R = w.n_layers, w.routes
        steps = max(1, min(steps, 16))
        # slot ids as the decode left them for the last `steps` tokens, replayed eagerly
        slots, xs, ws, nbytes = [], [], [], 0
        for i in range(steps):
            with torch.cuda.stream(self.cs):
                self.load_device(self.t)
                self.graph.replay()
            self.cs.synchronize()
            self.t += 1
            slots.append(self.b_slots.clone())
            xs.append(self.b_x.clone())
            ws.append(self.b_w.clone())
        out = torch.empty_like(self.b_out)
        for s in slots:
            for layer in range(L):
                nd = len(set(int(v) for v in s[layer].tolist() if v >= 0))
                nbytes += nd * w.blob_bytes + w.batch * w.hidden * 2 * 2 + R * 8
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.cs):
            for i in range(steps):
                for layer in range(L):
                    m.moe_routed_experts(self.cache.handle, layer, xs[i][layer], slots[i][layer],
                                         ws[i][layer], w.batch, w.top_k, None, None, out[layer],
                                         self.cs)
        with torch.cuda.stream(self.cs):
            g.replay()  # warm-up
        self.cs.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        with torch.cuda.stream(self.cs):
            e0.record(self.cs)
            for _ in range(reps):
                g.replay()
            e1.record(self.cs)
        self.cs.synchronize()
        ms = e0.elapsed_time(e1)
        launches = reps * steps * L
        per_launch_s = ms * 1e-3 / launches
        per_launch_bytes = nbytes / (steps * L)
        return {"kernel": "ffn_fused_kernel<NVFP4, routed> (moe_routed_experts: gate/up, "
                          "grid barrier, down + combine in one cooperative launch)",
                "launches": launches, "avg_launch_us": per_launch_s * 1e6,
                "bytes_per_launch": per_launch_bytes,
                "achieved_gbs": per_launch_bytes / per_launch_s / 1e9}

    def gather_bandwidth(self) -> dict:
        """The SM-driven gather alone: two cold caches over the same pinned host
        blobs (a region of the same slot storage) admit the same n
        never-resident experts, and each gathers that plan, timed with CUDA
        events.  The first gather is the first GPU read of those host pages in a
        while (`..._first_read`); the second reads them again right after, as a
        decode's repeated misses of the same experts do, and is the gather's
        figure against the host link.  Next to it the copy engine's pinned host
        -> device bandwidth (cudaMemcpyAsync, the host link's reference)."""
        torch, m, w = self.torch, self.m, self.w
        n_slots = 64
        caches = [m.SlotCache(
            n_layers=w.n_layers, n_experts=w.n_experts, n_slots=n_slots,
            pool_mode=m.MOE_POOL_SHARED, hidden=w.hidden, inter=w.inter, wfmt=w.fmt,
            shared_inter=0, slot_storage=self.storage, slot_stride=self.blobs.stride,
            host_blob_ptrs=self.blobs.addrs(), max_routes=64, max_rows=1) for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        res = {}
        key = 0
        for n in (1, 8, 28):
            best = [None, None]  # first read, second read
            for rep in range(4):
                # n experts of one layer never admitted to these caches before
                layer, first = divmod(key, w.n_experts - n)
                layer %= w.n_layers
                key += n
                ids = torch.arange(first, first + n, dtype=torch.int32, device="cuda")
                for i, c in enumerate(caches):
                    out = torch.empty_like(ids)
                    with torch.cuda.stream(self.cs):
                        m.moe_admit(c.handle, layer, ids, out, n, -1, self.cs)
                        e0.record(self.cs)
                        m.moe_gather_missing(c.handle, m.MOE_PLAN_DEMAND, self.cs)
                        e1.record(self.cs)
                    self.cs.synchronize()
                    assert c.stats(layer)["fetched"] >= n
                    ms = e0.elapsed_time(e1)
                    best[i] = ms if best[i] is None else min(best[i], ms)
            res[f"sm_gather_gbs_{n}_experts"] = n * w.blob_bytes / (best[1] * 1e-3) / 1e9
            res[f"sm_gather_gbs_{n}_experts_first_read"] = n * w.blob_bytes / (best[0] * 1e-3) / 1e9
        for c in caches:
            c.close()
        nbytes = 28 * w.blob_bytes
        src = self.blobs.buf[:nbytes]
        dst = self.storage[:nbytes]
        ce = []
        for _ in range(5):
            with torch.cuda.stream(self.cs):
                e0.record(self.cs)
                dst.copy_(src, non_blocking=True)
                e1.record(self.cs)
            self.cs.synchronize()
            ce.append(e0.elapsed_time(e1))
        res["copy_engine_gbs_28_experts"] = nbytes / (min(ce) * 1e-3) / 1e9
        big = 1 << 30
        ce = []
        for _ in range(3):
            with torch.cuda.stream(self.cs):
                e0.record(self.cs)
                self.storage[:big].copy_(self.blobs.buf[:big], non_blocking=True)
                e1.record(self.cs)
            self.cs.synchronize()
            ce.append(e0.elapsed_time(e1))
        res["copy_engine_gbs_1GiB"] = big / (min(ce) * 1e-3) / 1e9
        # four 256 MiB copies on four streams at once, from four regions of the blobs
        streams = [torch.cuda.Stream() for _ in range(4)]
        part = big // 4
        ce = []
        for _ in range(3):
            self.cs.synchronize()
            with torch.cuda.stream(self.cs):
                e0.record(self.cs)
            for i, st in enumerate(streams):
                st.wait_event(e0)
                with torch.cuda.stream(st):
                    self.storage[i * part:(i + 1) * part].copy_(
                        self.blobs.buf[(2 * i + 1) * part:(2 * i + 2) * part], non_blocking=True)
            for st in streams:
                ev = torch.cuda.Event()
                ev.record(st)
                self.cs.wait_event(ev)
            with torch.cuda.stream(self.cs):
                e1.record(self.cs)
            self.cs.synchronize()
            ce.append(e0.elapsed_time(e1))
        res["copy_engine_gbs_4_streams_1GiB"] = big / (min(ce) * 1e-3) / 1e9
        res["numa"] = host_numa(self.blobs.buf.data_ptr(), self.torch.cuda.current_device())
        res["host_link_peak_gbs"] = max(res["copy_engine_gbs_1GiB"],
                                        res["copy_engine_gbs_4_streams_1GiB"],
                                        res["sm_gather_gbs_28_experts"])
        res["frac_of_host_link_peak"] = res["sm_gather_gbs_28_experts"] / res["host_link_peak_gbs"]
        return res


def admission_sweep(dev: int) -> dict:
    """Wide all-hit admission: 48 per-layer 2,100-slot pools holding all 512
    experts, top-10, uniform ids; 48 admissions captured in one CUDA graph,
    replayed 40 times; microseconds per admission by route count [FreeToken
    PR #680, Measurement]."""
    import torch

    import expert_slot_cache_lru_gb300 as m
    import synth
    w = synth.workloads()["wide_admission"]
    res = {}
    cache = m.SlotCache(n_layers=w.n_layers, n_experts=w.n_experts, n_slots=w.n_slots,
                        pool_mode=m.MOE_POOL_PER_LAYER, max_routes=max(w.batches) * w.top_k,
                        max_rows=1)
    pre = synth.prefill_ids(w)
    for layer in range(w.n_layers):
        m.moe_cache_prefill(cache.handle, layer, pre, len(pre))
    s = torch.cuda.Stream()
    # empty-kernel graph of 48 nodes: the launch cost the admissions ride on
    for batch in w.batches:
        ids = torch.from_numpy(synth.uniform_ids(w, batch, salt=batch)).cuda()
        out = torch.empty_like(ids)
        R = ids.shape[1]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for layer in range(w.n_layers):
                m.moe_admit(cache.handle, layer, ids[layer], out[layer], R, -1, s)
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
        s.synchronize()
        meds = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                for _ in range(40):
                    g.replay()
                e1.record(s)
            s.synchronize()
            meds.append(e0.elapsed_time(e1) * 1e3 / (48 * 40))
        res[str(R)] = round(statistics.median(meds), 3)
    cache.close()
    return res


def _admission_inputs(name: str, tokens: int):
    """(workload, ids [T, L, R], predictions [T, L, n_pred] or None) of a
    workload's first tokens."""
    import synth
    w = synth.workloads()[name]
    ids, _ = synth.make_routing(w, steps=tokens)
    ids = ids.reshape(tokens, w.n_layers, -1).astype(np.int32)
    pred = None
    if w.n_pred:
        pred = np.zeros((tokens, w.n_layers, w.n_pred), np.int32)
        for t in range(tokens):
            for l in range(w.n_layers - 1):
                pred[t, l] = synth.make_predictions(w, ids[t, l + 1], t, l)
    return w, ids, pred


ADMISSION_CASES = {"tiny": 64, "hybrid_prefetch": 8}  # workload -> tokens timed


def admission_small(dev: int) -> dict:
    """GPU admission on the tiny workload (1 layer, 16 experts, 6 slots, top-2,
    64 steps) and the hybrid one (48 layers, 1,024 slots, fetch cap 4, plus the
    look-ahead prefetch of 8 ids for the next layer), as the workloads' first
    tokens captured in one CUDA graph of admissions (and prefetches) on an
    admission-only cache.  The graph is replayed 5 times (the cache state
    carries over), each replay timed with CUDA events; median µs per call."""
    import torch

    import expert_slot_cache_lru_gb300 as m
    res = {}
    for name, tokens in ADMISSION_CASES.items():
        w, ids, pred = _admission_inputs(name, tokens)
        L, R = w.n_layers, ids.shape[2]
        cache = m.SlotCache(n_layers=L, n_experts=w.n_experts, n_slots=w.n_slots,
                            pool_mode=m.MOE_POOL_SHARED, max_routes=R, max_rows=w.batch,
                            max_pred=w.n_pred)
        d_ids = torch.from_numpy(ids).cuda()
        d_out = torch.empty_like(d_ids)
        d_pred = torch.from_numpy(pred).cuda() if pred is not None else None
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        calls = 0
        with torch.cuda.graph(g, stream=s):
            for t in range(tokens):
                for l in range(L):
                    m.moe_admit(cache.handle, l, d_ids[t, l], d_out[t, l], R, w.fetch_cap, s)
                    calls += 1
                    if d_pred is not None and l + 1 < L:
                        m.moe_prefetch(cache.handle, l + 1, d_pred[t, l], w.n_pred, s)
                        calls += 1
        times = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                g.replay()
                e1.record(s)
            s.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / calls)
        res[name] = {"calls_per_graph": calls, "us_per_call": round(statistics.median(times), 3)}
        del g
        cache.close()
    return res


def admission_oracle(seconds: float = 6.0) -> dict:
    """The oracle's admission (single-threaded, the caller's thread) on the
    same inputs as admission_small and admission_sweep: µs per call."""
    import oracle
    import synth
    res = {}
    for name, tokens in ADMISSION_CASES.items():
        w, ids, pred = _admission_inputs(name, tokens)
        oc = oracle.OracleCache(w.n_layers, w.n_experts, w.n_slots)
        calls, t0 = 0, time.perf_counter()
        for t in range(tokens):
            for l in range(w.n_layers):
                oc.admit(l, ids[t, l], w.fetch_cap)
                calls += 1
                if pred is not None and l + 1 < w.n_layers:
                    oc.prefetch(l + 1, pred[t, l])
                    calls += 1
        res[name] = {"calls": calls, "us_per_call": round((time.perf_counter() - t0) * 1e6 / calls, 2)}
    w = synth.workloads()["wide_admission"]
    pre = synth.prefill_ids(w)
    for batch in (1, 128):
        oc = oracle.OracleCache(w.n_layers, w.n_experts, w.n_slots, per_layer=True)
        for layer in range(w.n_layers):
            oc.prefill(layer, pre)
        ids = synth.uniform_ids(w, batch, salt=batch)
        calls, t0 = 0, time.perf_counter()
        while True:
            for layer in range(w.n_layers):
                oc.admit(layer, ids[layer])
                calls += 1
            if time.perf_counter() - t0 > seconds / 4:
                break
        res[f"wide_admission_{ids.shape[1]}_routes"] = {
            "calls": calls, "us_per_call": round((time.perf_counter() - t0) * 1e6 / calls, 2)}
    return res


def wide_step(dev: int, reps: int = 5, routing: str = "uniform") -> dict:
    """The wide decode step: 600 rows x top-2 = 1,200 routes over 1,024 NVFP4
    experts (H 2048, I 768) with a 1,100-slot cache, 30% of the experts
    pre-resident.  The first step admits ~495 misses; its admission, gather and
    routed FFNs + combine are timed with CUDA events on one stream.  The FFN is
    then re-timed `reps` times on the resident slots (the same step again: all
    hits), which is the grouped-FFN figure.  Algorithmic bytes of the FFN: the
    distinct resident experts' blobs plus activations."""
    import torch

    import expert_slot_cache_lru_gb300 as m
    import synth
    w = synth.workloads()["wide_decode"]
    if routing != w.routing:
        w = synth.scaled(w, routing=routing)
    blobs = synth.HostBlobs(w, pinned=True)
    storage = torch.empty(w.n_slots * blobs.stride, dtype=torch.uint8, device="cuda")
    cache = m.SlotCache(n_layers=1, n_experts=w.n_experts, n_slots=w.n_slots,
                        pool_mode=m.MOE_POOL_SHARED, hidden=w.hidden, inter=w.inter, wfmt=w.fmt,
                        shared_inter=0, slot_storage=storage, slot_stride=blobs.stride,
                        host_blob_ptrs=blobs.addrs(), max_routes=w.routes, max_rows=w.batch)
    pre = synth.prefill_ids(w)
    m.moe_cache_prefill(cache.handle, 0, pre, len(pre))
    ids, wts = synth.make_routing(w, steps=1)
    d_ids = torch.from_numpy(ids[0, 0].ravel().copy()).cuda()
    d_w = torch.from_numpy(wts[0, 0].ravel().copy()).cuda()
    d_x = torch.from_numpy(synth.make_hidden(w, 0)[0].view(np.int16)).cuda()
    d_slots = torch.empty_like(d_ids)
    out = torch.empty(w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    R = w.routes
    with torch.cuda.stream(s):
        ev[0].record(s)
        m.moe_admit(cache.handle, 0, d_ids, d_slots, R, -1, s)
        ev[1].record(s)
        m.moe_gather_missing(cache.handle, m.MOE_PLAN_DEMAND, s)
        ev[2].record(s)
        m.moe_routed_experts(cache.handle, 0, d_x, d_slots, d_w, w.batch, w.top_k, None, None,
                             out, s)
        ev[3].record(s)
    s.synchronize()
    st = cache.stats(0)
    t_adm, t_gat, t_ffn = (ev[i].elapsed_time(ev[i + 1]) for i in range(3))
    slots = d_slots.cpu().numpy()
    distinct = len(set(int(v) for v in slots if v >= 0))
    _, counts = np.unique(slots[slots >= 0], return_counts=True)
    dense_groups = int((counts >= 4).sum())
    ffn_bytes = distinct * w.blob_bytes + w.batch * w.hidden * 2 * 2 + R * 8
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            m.moe_routed_experts(cache.handle, 0, d_x, d_slots, d_w, w.batch, w.top_k, None, None,
                                 out, s)
            e1.record(s)
        s.synchronize()
        times.append(e0.elapsed_time(e1))
    t_ffn_hot = statistics.median(times)
    # the same FFN with every group forced onto one kernel family, for comparison
    forced = {}
    for name, mode in (("cuda_cores", m.MOE_WIDE_CUDA_CORES), ("tensor_cores", m.MOE_WIDE_TENSOR_CORES)):
        m.moe_cache_set_wide_path(cache.handle, mode)
        tt = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                m.moe_routed_experts(cache.handle, 0, d_x, d_slots, d_w, w.batch, w.top_k, None,
                                     None, out, s)
                e1.record(s)
            s.synchronize()
            tt.append(e0.elapsed_time(e1))
        forced[name] = statistics.median(tt)
    m.moe_cache_set_wide_path(cache.handle, m.MOE_WIDE_AUTO)
    # the admission again in a graph, repeated: the same 1,200 routes each time
    # on a fresh cache holding the same 307 experts (so every replay admits the
    # ~479 misses into empty slots, as the first step did).  Two such graphs on
    # two sets of caches: the first replayed as the warm-up, the second timed.
    adm_graph = None
    try:
        n_rep = 8
        graphs, outs_all, caches = [], [], []
        for _ in range(2):
            g = torch.cuda.CUDAGraph()
            cs_ = []
            for _ in range(n_rep):
                c2 = m.SlotCache(n_layers=1, n_experts=w.n_experts, n_slots=w.n_slots,
                                 pool_mode=m.MOE_POOL_SHARED, max_routes=w.routes,
                                 max_rows=w.batch)
                m.moe_cache_prefill(c2.handle, 0, pre, len(pre))
                cs_.append(c2)
            outs = [torch.empty_like(d_ids) for _ in range(n_rep)]
            with torch.cuda.graph(g, stream=s):
                for c2, o2 in zip(cs_, outs):
                    m.moe_admit(c2.handle, 0, d_ids, o2, R, -1, s)
            graphs.append(g)
            outs_all.append(outs)
            caches += cs_
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            graphs[0].replay()  # warm-up: the same miss-heavy admissions on other caches
            e0.record(s)
            graphs[1].replay()
            e1.record(s)
        s.synchronize()
        assert all(torch.equal(o2, d_slots) for outs in outs_all for o2 in outs)
        adm_graph = round(e0.elapsed_time(e1) * 1e3 / n_rep, 2)
        del g
        for c2 in caches:
            c2.close()
    except Exception as ex:  # reported, never fatal to the bench line
        adm_graph = f"failed: {ex}"
    cache.close()
    return {"routing": routing, "routes": R, "distinct_experts": distinct,
            "misses": int(st["misses"]),
            "admission_us": round(t_adm * 1e3, 2),
            "gather_ms": round(t_gat, 3),
            "gather_gbs": round(st["fetched"] * w.blob_bytes / (t_gat * 1e-3) / 1e9, 1),
            "admission_us_graph": adm_graph,
            "ffn_path": "automatic: expert groups of >= 4 routes on the tensor cores (tcgen05), "
                        "the rest on the CUDA cores",
            "groups_ge_4_routes": dense_groups,
            "ffn_ms_first": round(t_ffn, 3), "ffn_ms": round(t_ffn_hot, 3),
            "ffn_bytes": ffn_bytes, "ffn_gbs": round(ffn_bytes / (t_ffn_hot * 1e-3) / 1e9, 1),
            "ffn_ms_all_cuda_cores": round(forced["cuda_cores"], 3),
            "ffn_ms_all_tensor_cores": round(forced["tensor_cores"], 3),
            "ffn_gbs_all_tensor_cores": round(ffn_bytes / (forced["tensor_cores"] * 1e-3) / 1e9, 1),
            "step_ms": round(t_adm + t_gat + t_ffn, 3)}


def hybrid_step(dev: int, warm: int = 4, tokens: int = 8) -> dict:
    """The hybrid decode: 48 bf16 layers (H 4096, I 1024, 256 experts, top-8),
    a 1,024-slot shared pool, fetch cap 4 and 8 look-ahead predictions per
    layer, host blobs aliased onto 96.  Each layer is moe_decode_layer with
    MOE_FUSED | MOE_HYBRID: the routes the capped admission leaves at -1 run
    on the host's cores (the hybrid CPU executor) and are added to the GPU's
    output.  Timed with CUDA events over `tokens` tokens after `warm`; the same
    pipeline without MOE_HYBRID (the GPU partial alone) is timed beside it on a
    second cache.  The executor's figure is the expert bytes its -1 routes
    stream per second of its busy time."""
    import torch

    import expert_slot_cache_lru_gb300 as m
    import synth
    w = synth.workloads()["hybrid_prefetch"]
    blobs = synth.HostBlobs(w, pinned=True)
    ids, wts = synth.make_routing(w, steps=warm + tokens)
    L, R = w.n_layers, w.routes
    s = torch.cuda.Stream()
    n_threads = max(1, min(16, os.cpu_count() or 1))
    res = {"threads": n_threads, "tokens": tokens}
    # the host-read reference for the executor: a plain multi-threaded read of
    # the same pinned blobs (torch's fp32 sum over the bytes viewed as fp32,
    # whatever values they hold), with as many threads as the pool, best of 3
    prev = torch.get_num_threads()
    torch.set_num_threads(n_threads)
    flat = blobs.buf[:blobs.buf.numel() // 4 * 4].view(torch.float32)
    times = []
    for _ in range(3):
        t0 = time.perf_counter()
        flat.sum()
        times.append(time.perf_counter() - t0)
    torch.set_num_threads(prev)
    host_gbs = flat.numel() * 4 / min(times) / 1e9
    for hybrid in (True, False):
        storage = torch.empty(w.n_slots * blobs.stride, dtype=torch.uint8, device="cuda")
        cache = m.SlotCache(n_layers=L, n_experts=w.n_experts, n_slots=w.n_slots,
                            pool_mode=m.MOE_POOL_SHARED, hidden=w.hidden, inter=w.inter,
                            wfmt=w.fmt, slot_storage=storage, slot_stride=blobs.stride,
                            host_blob_ptrs=blobs.addrs(), max_routes=R, max_rows=w.batch,
                            max_pred=w.n_pred)
        if hybrid:
            m.moe_hybrid_start(cache.handle, n_threads)
        flags = m.MOE_FUSED | (m.MOE_HYBRID if hybrid else 0)
        d_x = torch.empty(L, w.batch, w.hidden, dtype=torch.int16, device="cuda")
        d_ids = torch.empty(L, R, dtype=torch.int32, device="cuda")
        d_w = torch.empty(L, R, dtype=torch.float32, device="cuda")
        d_pred = torch.empty(L, w.n_pred, dtype=torch.int32, device="cuda")
        d_slots = torch.empty(L, R, dtype=torch.int32, device="cuda")
        out = torch.empty(L, w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
        inputs = []
        for t in range(warm + tokens):
            pred = np.stack([synth.make_predictions(w, ids[t, l + 1], t, l) if l + 1 < L else
                             np.zeros(w.n_pred, np.int32) for l in range(L)]).astype(np.int32)
            inputs.append((synth.make_hidden(w, t).view(np.int16), ids[t].reshape(L, -1),
                           wts[t].reshape(L, -1), pred))

        def load(t):
            x, i, wt, pr = inputs[t]
            d_x.copy_(torch.from_numpy(x))
            d_ids.copy_(torch.from_numpy(np.ascontiguousarray(i)))
            d_w.copy_(torch.from_numpy(np.ascontiguousarray(wt)))
            d_pred.copy_(torch.from_numpy(pr))

        def layers():
            for l in range(L):
                has = l + 1 < L
                m.moe_decode_layer(cache.handle, l, d_x[l], d_ids[l], d_w[l], d_slots[l], w.batch,
                                   w.top_k, w.fetch_cap, d_pred[l] if has else None,
                                   w.n_pred if has else 0, None, None, out[l], s, None, flags)

        with torch.cuda.stream(s):
            for t in range(warm):
                load(t)
                layers()
        s.synchronize()
        c0 = m.moe_hybrid_counters(cache.handle) if hybrid else None
        ms = 0.0
        for t in range(warm, warm + tokens):  # input copies stay outside the timed region
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                load(t)
                e0.record(s)
                layers()
                e1.record(s)
            s.synchronize()
            ms += e0.elapsed_time(e1)
        st = [cache.stats(l) for l in range(L)]
        key = "hybrid" if hybrid else "gpu_partial_only"
        res[key] = {"tok_s": round(tokens / (ms * 1e-3), 2), "ms_per_token": round(ms / tokens, 3),
                    "timeouts": int(any(x["status_bits"] & 4 for x in st))}
        if hybrid:
            c1 = m.moe_hybrid_counters(cache.handle)
            jobs = c1["jobs"] - c0["jobs"]
            routes = c1["cpu_routes"] - c0["cpu_routes"]
            busy = (c1["busy_ns"] - c0["busy_ns"]) * 1e-9
            busy_r = (c1["busy_route_ns"] - c0["busy_route_ns"]) * 1e-9
            gbs = routes * w.blob_bytes / max(busy_r, 1e-9) / 1e9
            res[key].update({"jobs": jobs, "cpu_routes": routes,
                             "cpu_routes_per_token": round(routes / tokens, 2),
                             "cpu_busy_us_per_job": round(busy / max(jobs, 1) * 1e6, 1),
                             "cpu_expert_gbs": round(gbs, 1),
                             "host_read_gbs": round(host_gbs, 1),
                             "frac_of_host_read": round(gbs / host_gbs, 3)})
            m.moe_hybrid_stop(cache.handle)
        cache.close()
        del storage
        torch.cuda.empty_cache()
    return res


def cpu_baseline(seconds: float = 15.0) -> dict:
    """The oracle as it stands, single-threaded on one host core (the process
    is pinned to one CPU with sched_setaffinity while it runs): admission plus
    fp64 layer math for as many layers of the benchmark's tokens as fit in
    ~`seconds`, extrapolated to tokens/s (40 layers per token); then the
    oracle's µs per admission on the tiny, hybrid and wide-admission inputs.
    Reports the host's core count beside it."""
    prev = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    cpu = min(prev) if prev else None
    if prev:
        os.sched_setaffinity(0, {cpu})
    try:
        res = _cpu_baseline(seconds)
    finally:
        if prev:
            os.sched_setaffinity(0, prev)
    res["pinned_cpu"] = cpu
    res["host_cores"] = os.cpu_count()
    return res


def _cpu_baseline(seconds: float) -> dict:
    import oracle
    import synth
    w = synth.workloads()[WORKLOAD]
    wl = synth.scaled(w, steps=8)
    ids, wts = synth.make_routing(wl)
    oc = oracle.OracleCache(w.n_layers, w.n_experts, w.n_slots)
    # lazily generated blobs of the experts the sample touches (not timed)
    blobs = {}
    shared = {}

    def blob(key):
        if key not in blobs:
            b = np.empty(w.blob_bytes, np.uint8)
            synth.fill_blob(b, w.fmt, w.hidden, w.inter, synth.Rng(w.seed, synth.S_WEIGHTS, key))
            blobs[key] = b
        return blobs[key]

    layers_done = 0
    elapsed = 0.0
    t = 0
    while elapsed < seconds and t < wl.steps:
        x = synth.make_hidden(w, t)
        for layer in range(w.n_layers):
            lb = [blob(layer * w.n_experts + e) if e in set(ids[t, layer].ravel().tolist()) else None
                  for e in range(w.n_experts)]
            if layer not in shared:
                shared[layer] = synth.make_shared(w, layer)
            sb, sg = shared[layer]
            t0 = time.perf_counter()
            oc.admit(layer, ids[t, layer].ravel())
            oracle.layer(w.fmt, lb, w.n_experts, w.hidden, w.inter, x[layer], ids[t, layer],
                         wts[t, layer], shared_blob=sb, shared_inter=w.shared_inter,
                         shared_gate_w=sg)
            elapsed += time.perf_counter() - t0
            layers_done += 1
            if elapsed >= seconds:
                break
        t += 1
    tok_s = layers_done / w.n_layers / elapsed
    adm = admission_oracle()
    return {"value": tok_s, "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"{layers_done} layers (admission + fp64 dequantised layer math, "
                      f"shared expert included) of the first tokens, {elapsed:.1f} s of CPU, "
                      f"extrapolated at 40 layers per token",
            "admission_us_per_call": adm}


def run_native(args) -> None:
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo",
                                device_id=torch.device("cuda", local))
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    if args.wide_only:  # profiler runs: the wide decode step alone
        if rank == 0:
            print(json.dumps({"wide_only": True, **wide_step(local, routing=args.wide_routing)}),
                  flush=True)
        return
    if args.hybrid_only:
        if rank == 0:
            print(json.dumps({"hybrid_only": True, **hybrid_step(local)}), flush=True)
        return
    dec = Decode(local, overlap=not args.serial, warm_tokens=args.warm_tokens,
                 n_layers=args.layers, n_slots=args.slots, fused=not args.unfused)
    L = dec.w.n_layers
    props = torch.cuda.get_device_properties(local)
    # settle: decode for a few seconds first.  Host reads over the CPU link
    # (the miss gathers) are slower for the first seconds of activity after an
    # idle period; the timed tokens then measure the steady state.
    t_settle = time.perf_counter()
    settle_tokens = 0
    while time.perf_counter() - t_settle < args.settle_s:
        for _ in range(50):
            dec.step()
        settle_tokens += 50
        torch.cuda.synchronize()
    settle_s = time.perf_counter() - t_settle
    for _ in range(args.warmup):
        dec.step()
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    barrier()
    torch.cuda.synchronize()
    st0 = dec.totals()
    t_first = dec.t
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bus = (f"{getattr(props, 'pci_domain_id', 0):08x}:{getattr(props, 'pci_bus_id', 0):02x}:"
           f"{getattr(props, 'pci_device_id', 0):02x}.0")
    sampler = ClockSampler(bus, index=local)
    with sampler:
        torch.cuda.nvtx.range_push("timed")
        e0.record(dec.cs)
        for _ in range(args.steps):
            dec.step()
        e1.record(dec.cs)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
    barrier()
    st1 = dec.totals()
    timed = {k: (st1[k] - st0[k]) / args.steps for k in st0}
    local_ms = e0.elapsed_time(e1)
    tok_s, max_s = replica_rate(local_ms * 1e-3, args.steps, ws, "cuda")
    ms = max_s * 1e3
    if args.routed_only:  # profiler runs: the routed FFN kernel's roofline graph only
        if rank == 0:
            roof = dec.routed_gemv_roofline(steps=2)
            print(json.dumps({"routed_only": True, "layers": L, **roof}), flush=True)
        return
    if args.prefill_only:
        if rank == 0:
            print(json.dumps({"prefill_only": True, "on_demand": prefill_chunks(dec),
                              "layer_major": prefill_chunks(dec, (128,), layer_major=True)}),
                  flush=True)
        return
    if args.lookahead_only:
        if rank == 0:
            print(json.dumps({"lookahead_only": True, **lookahead_producer(dec)}), flush=True)
        return
    if args.decode_only:  # profiler runs: the timed decode only, no sub-measurements
        if rank == 0:
            print(json.dumps({"decode_only": True, "layers": L, "slots": dec.w.n_slots,
                              "settle_tokens": settle_tokens,
                              "misses_per_token": round(timed["misses"], 2),
                              "tok_s": round(tok_s, 2), "ms_per_step": round(ms / args.steps, 4)}),
                  flush=True)
        return

    # end to end through the public API: pinned host inputs in, output back, per token
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dec.step_e2e()
    e2e_rate, _ = replica_rate(time.perf_counter() - t0, args.steps, ws, "cuda")
    e2e = {"value": e2e_rate, "unit": "tok/s",
           "h2d_bytes_per_step": dec.h2d_bytes(), "d2h_bytes_per_step": dec.d2h_bytes()}

    layer_roof = dec.layer_kernel_roofline(t_first, args.steps, local_ms, timed, hbm,
                                           gather_peak=None)
    roof = dec.routed_gemv_roofline(steps=8)
    gather = dec.gather_bandwidth()
    layer_roof["host_link"]["peak"] = round(gather["host_link_peak_gbs"], 1)
    layer_roof["host_link"]["frac"] = round(layer_roof["host_link"]["achieved"] /
                                            gather["host_link_peak_gbs"], 4)
    adm = admission_sweep(local)
    adm_small = admission_small(local)
    wide = wide_step(local)
    wide_zipf = wide_step(local, reps=3, routing="zipf")
    hyb = hybrid_step(local) if not args.no_hybrid else None
    look = lookahead_producer(dec)
    pre = {"on_demand": prefill_chunks(dec),
           "layer_major": prefill_chunks(dec, (128,), layer_major=True)}
    tr = routed_traffic()
    line = {
        "metric": METRIC,
        "value": round(tok_s, 2),
        "unit": "tok/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 weights (e2m1 + e4m3/16 + fp32), bf16 activations, fp32 accumulate; int32 cache",
        "data": "synthetic",
        "config": {"workload": "Qwen3-MoE-like offloaded decode: 40 MoE layers x 256 NVFP4 experts, "
                               "top-8, H 2048, I 512, gated shared expert I 512, 3164-slot LRU, "
                               "batch 1, Zipf(1.1) routing with reuse (~28 misses/token)",
                   "global_batch": ws, "graph": "one CUDA graph per token (40 layers)",
                   "layer": ("one launch: CTA 0 admits while the others copy the misses into "
                             "staging, run the shared and routed experts and combine"
                             if not args.unfused else
                             "four launches: admission, gather on a side stream (events), "
                             "shared expert, routed experts" if not args.serial else
                             "four launches on one stream"),
                   "overlap": not args.serial, "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2: each token streams ~637 MB of expert weights",
                   "cache_warmup_tokens": args.warm_tokens,
                   "settle": f"{settle_tokens} untimed tokens ({settle_s:.1f} s) before the "
                             f"{args.warmup} warm-up steps: host-link reads reach their steady "
                             f"rate only after seconds of activity"},
        # per layer: one launch (admission, gathers, shared + routed experts);
        # unfused: admission, demand gather, shared-expert FFN, routed FFN + combine
        "gpu_launches": args.steps * (4 if args.unfused else 1) * L,
        "e2e": e2e,
        "roofline": {"bound": "hbm", "achieved": round(roof["achieved_gbs"], 1),
                     "peak": hbm, "unit": "GB/s",
                     "frac": round(roof["achieved_gbs"] / hbm, 4),
                     "traffic": round(tr["bytes_per_launch"]) if tr else None,
                     "traffic_source": tr["source"] if tr else
                     "null: no capture of the current kernel source",
                     "kernel": roof["kernel"], "avg_launch_us": round(roof["avg_launch_us"], 3),
                     "bytes_per_launch": round(roof["bytes_per_launch"]),
                     "peak_source": f"{peaks['_source']} (MEASURED_PEAKS.json hbm_gbs)"},
        "timed_tokens": {"misses_per_token": round(timed["misses"], 2),
                         "fetched_per_token": round(timed["fetched"], 2),
                         "lookups_per_token": round(timed["lookups"], 2),
                         "hits_per_token": round(timed["hits"], 2)},
        "roofline_layer_kernel": layer_roof,
        "admission_us_per_layer": adm,
        "admission_us_per_call_small": adm_small,
        "wide_decode_step": wide,
        "wide_decode_step_zipf": wide_zipf,
        "hybrid_decode": hyb,
        "lookahead_producer": look,
        "prefill_chunks": pre,
        "gather": {k: (round(v, 3) if isinstance(v, float) else v) for k, v in gather.items()},
        "setup_s": {k: round(v, 1) for k, v in dec.setup_s.items()},
        "clocks": sampler.summary(),
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_reference(args) -> None:
    """The oracle timed as it stands: each step is one layer of one token (a
    bounded sample); tokens/s extrapolated at 40 layers per token."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    w = synth.workloads()[WORKLOAD]
    n = args.warmup + args.steps
    ids, wts = synth.make_routing(synth.scaled(w, steps=max(1, n // w.n_layers + 1)))
    oc = oracle.OracleCache(w.n_layers, w.n_experts, w.n_slots)
    shared = {}
    samples = []
    for i in range(n):
        t, layer = divmod(i, w.n_layers)
        x = synth.make_hidden(w, t)
        lb = [None] * w.n_experts
        for e in set(ids[t, layer].ravel().tolist()):
            b = np.empty(w.blob_bytes, np.uint8)
            synth.fill_blob(b, w.fmt, w.hidden, w.inter,
                            synth.Rng(w.seed, synth.S_WEIGHTS, layer * w.n_experts + e))
            lb[e] = b
        if layer not in shared:
            shared[layer] = synth.make_shared(w, layer)
        sb, sg = shared[layer]
        t0 = time.perf_counter()
        oc.admit(layer, ids[t, layer].ravel())
        oracle.layer(w.fmt, lb, w.n_experts, w.hidden, w.inter, x[layer], ids[t, layer],
                     wts[t, layer], shared_blob=sb, shared_inter=w.shared_inter,
                     shared_gate_w=sg)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            samples.append(dt)
    total = sum(samples)
    tok_s = len(samples) / w.n_layers / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tok_s, 5), "unit": "tok/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / len(samples) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": "Qwen3-MoE-like offloaded decode (as the native arm); one step = "
                               "one layer of one token", "parallelism": "single host thread"},
        "cpu_baseline": {"value": round(tok_s, 5), "unit": "tok/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(samples)} layers, extrapolated at 40 layers per token"},
        "e2e": {"value": round(tok_s, 5), "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def prefill_chunks(dec, tokens=(16, 128), chunks: int = 4, layer_major: bool = False) -> dict:
    """Prefill chunks through the decode workload's 40 layers [FreeToken PR
    #680, Problem: DeepSeek-V4's on-demand prefill chunks, taken while
    T * top_k < num_experts; Solution: one admission per layer, graph-capturable]:
    a chunk of T tokens is one wide step per layer (admission, gather on the side
    stream, grouped FFN with the tensor cores for dense groups, shared expert,
    combine), on its own 3,164-slot cache over the decode's pinned blobs.  Chunk
    0 starts cold; the median of the later chunks is the steady figure.  Each
    chunk is timed with CUDA events around its 40 layer calls.  layer_major: a
    chunk with more routes than experts also prefetches every expert of the next
    layer (the look-ahead prefetch with all E ids as predictions), so that layer
    l + 1's copies cross the host link while layer l computes."""
    import torch

    import synth
    m, w0 = dec.m, dec.w
    L, k = w0.n_layers, w0.top_k
    out = {}
    for T in tokens:
        w = synth.scaled(w0, batch=T, steps=chunks)
        storage = torch.empty(w.n_slots * dec.blobs.stride, dtype=torch.uint8, device="cuda")
        cache = m.SlotCache(n_layers=L, n_experts=w.n_experts, n_slots=w.n_slots,
                            pool_mode=m.MOE_POOL_SHARED, hidden=w.hidden, inter=w.inter,
                            wfmt=w.fmt, shared_inter=w.shared_inter, slot_storage=storage,
                            slot_stride=dec.blobs.stride, host_blob_ptrs=dec.blobs.addrs(),
                            max_routes=T * k, max_rows=T, max_pred=w.n_experts)
        lm = layer_major and T * k >= w.n_experts
        every = torch.arange(w.n_experts, dtype=torch.int32, device="cuda")
        ids, wts = synth.make_routing(w, steps=chunks)
        slots = torch.empty(L, T * k, dtype=torch.int32, device="cuda")
        y = torch.empty(L, T, w.hidden, dtype=torch.bfloat16, device="cuda")
        cs, side = torch.cuda.Stream(), torch.cuda.Stream()
        flags = m.MOE_FUSED | m.MOE_OVERLAP
        rows = []
        for c in range(chunks):
            d_x = torch.from_numpy(synth.make_hidden(w, c).view(np.int16)).cuda()
            d_ids = torch.from_numpy(ids[c].reshape(L, -1).copy()).cuda()
            d_w = torch.from_numpy(wts[c].reshape(L, -1).copy()).cuda()
            def counts():
                st = [cache.stats(l) for l in range(L)]
                return sum(x["misses"] for x in st), sum(x["pf_filled"] for x in st)
            before = counts()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(cs):
                e0.record(cs)
                for l in range(L):
                    sb, sg = dec.shared[l]
                    pf = lm and l + 1 < L
                    m.moe_decode_layer(cache.handle, l, d_x[l], d_ids[l], d_w[l], slots[l], T, k, -1,
                                       every if pf else None, w.n_experts if pf else 0, sb, sg,
                                       y[l], cs, side, flags)
                e1.record(cs)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            after = counts()
            rows.append((ms, after[0] - before[0], after[1] - before[1]))
        plan = m.moe_decode_layer_plan(cache.handle, T, k, shared=True, pf=lm, flags=flags)
        cache.close()
        del storage
        steady = rows[1:]
        ms = statistics.median(r[0] for r in steady)
        mi = statistics.median(r[1] for r in steady)
        pfi = statistics.median(r[2] for r in steady)
        out[str(T)] = {"routes_per_layer": T * k, "cold_chunk_ms": round(rows[0][0], 3),
                       "cold_chunk_misses": rows[0][1], "ms_per_chunk": round(ms, 3),
                       "tok_s": round(T / (ms * 1e-3), 1), "misses_per_chunk": mi,
                       "prefetch_fills_per_chunk": pfi,
                       "host_link_gbs": round((mi + pfi) * w.blob_bytes / (ms * 1e6), 1),
                       "layer_major_prefetch": lm, "launches_per_layer": plan}
    return out


def lookahead_producer(dec, steps: int = 12, drifts=(0.25, 0.5, 1.0)) -> dict:
    """The look-ahead producer (moe_lookahead_predict): layer L+1's router on
    layer L's hidden state, at the decode's shape (256 experts, H 2048, one
    row, top 8).  Its time per launch in a graph of one launch per layer (each
    with its own 1 MiB router, so the routers stream from HBM), and its recall
    of the next layer's true top 8 when the hidden states drift from layer to
    layer (synth.drift_stream: x_{l+1} = (x_l + s n) / sqrt(1 + s^2)), the true
    routing of layer l+1 being its router's top 8 on x_{l+1}."""
    import torch

    import synth
    m, w = dec.m, dec.w
    L, E, H, k = w.n_layers, w.n_experts, w.hidden, w.top_k
    h = dec.cache.handle
    routers = torch.stack([torch.from_numpy(synth.make_router(w, l).view(np.int16))
                           for l in range(L)]).cuda()
    x = torch.from_numpy(np.ascontiguousarray(synth.make_hidden(w, 0)[:, :1]).view(np.int16)).cuda()
    pred = torch.zeros(L, k, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def enqueue():
        for l in range(L):
            m.moe_lookahead_predict(h, x[l], routers[(l + 1) % L], 1, k, pred[l], s)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        enqueue()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        enqueue()
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):  # replays run on the current stream: make it s
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * L)
    nbytes = E * H * 2 + H * 2 + k * 4
    recall = {}
    truth = torch.zeros(L, k, dtype=torch.int32, device="cuda")
    guess = torch.zeros(L, k, dtype=torch.int32, device="cuda")
    for sd in drifts:
        hit = tot = 0
        for t in range(steps):
            xs = torch.from_numpy(synth.drift_stream(w, t, sd, batch=1).view(np.int16)).cuda()
            for l in range(L - 1):
                m.moe_lookahead_predict(h, xs[l + 1], routers[l + 1], 1, k, truth[l], s)
                m.moe_lookahead_predict(h, xs[l], routers[l + 1], 1, k, guess[l], s)
            torch.cuda.synchronize()
            tr, gu = truth.cpu().numpy(), guess.cpu().numpy()
            for l in range(L - 1):
                hit += len(set(tr[l].tolist()) & set(gu[l].tolist()))
                tot += k
        recall[str(sd)] = round(hit / tot, 4)
    return {"us_per_launch": round(us, 3), "launches_per_token": L,
            "bytes_per_launch": nbytes, "achieved_gbs": round(nbytes / (us * 1e3), 1),
            "recall_of_next_layer_top8_by_drift": recall, "steps_per_drift": steps,
            "shape": f"{E} experts x H {H}, 1 row, top {k}"}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--serial", action="store_true", help="gather on the compute stream (ncu mode)")
    ap.add_argument("--unfused", action="store_true",
                    help="four launches per layer (side-stream gather joined by events) instead of "
                         "the fused layer")
    ap.add_argument("--settle-s", type=float, default=3.0,
                    help="seconds of untimed decode before the warm-up steps (steady state)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hybrid", action="store_true", help="skip the hybrid-executor decode")
    ap.add_argument("--hybrid-only", action="store_true",
                    help="run only the hybrid-executor decode and print it")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--warm-tokens", type=int, default=WARM_TOKENS,
                    help="eager tokens that warm the cache before the graph is captured")
    ap.add_argument("--layers", type=int, default=None, help="profiler case: fewer layers")
    ap.add_argument("--slots", type=int, default=None, help="profiler case: fewer slots")
    ap.add_argument("--decode-only", action="store_true",
                    help="time the decode only and print a short line (profiler runs)")
    ap.add_argument("--wide-only", action="store_true",
                    help="run only the wide decode step sub-measurement (profiler runs)")
    ap.add_argument("--wide-routing", choices=["uniform", "zipf"], default="uniform",
                    help="routing of the --wide-only step")
    ap.add_argument("--prefill-only", action="store_true",
                    help="after the decode set-up, only the prefill-chunk line")
    ap.add_argument("--lookahead-only", action="store_true",
                    help="after the decode set-up, only the look-ahead producer's line")
    ap.add_argument("--routed-only", action="store_true",
                    help="after the decode, run only the routed FFN kernel's roofline graph "
                         "(profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
