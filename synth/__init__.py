"""Seeded synthetic inputs for the offloaded-MoE decode layer.

This module is shared by the tests, the benchmark and the smoke check, and by
both sides of every parity comparison (the CUDA library and the CPU oracle
read the very same bytes).  It holds no cache policy and no expert
arithmetic: only random draws, the workload shapes, and the byte layout of an
expert blob (where the code, scale and global-scale banks sit), which it needs
to put valid scale bytes in the scale banks.

Recipe (all streams derived from ``numpy.random.SeedSequence([seed, stream,
...])`` over the PCG64 raw stream, which is stable across numpy versions):

* router ids: Zipf(1.1) over expert rank, P(rank r) ~ r^-1.1, mapped to expert
  ids by a fixed per-layer random permutation; top-k distinct per row by
  rejection; optional temporal reuse (each route position keeps the previous
  step's id with probability ``reuse`` if still distinct in the row);
  "uniform" routing draws ids uniformly instead;
* routing weights: k standard-normal logits per row, softmax over the k (the
  renormalised top-k softmax);
* hidden states: N(0, 1) rounded to bf16, independent per (step, layer, row);
* bf16 expert weights: N(0, 0.02) rounded to bf16;
* NVFP4 expert weights: uniform random e2m1 codes, e4m3 block scales drawn
  uniformly from the 16 codes 0x28..0x37 (0.25 .. 0.9375), one fp32 global
  scale per matrix uniform in [0.008, 0.014] -- about 0.02 rms per weight;
* look-ahead predictions: each true next-layer id kept with probability 0.7,
  else uniform over the experts;
* router weights (the look-ahead producer's input): N(0, 1 / H) rounded to
  bf16, one [E][H] matrix per layer;
* a drifting hidden stream (the producer's accuracy): x of layer l + 1 is
  (x_l + s n_l) / sqrt(1 + s^2) with n_l ~ N(0, 1), rounded to bf16 -- a
  stand-in for a residual stream whose consecutive layers' inputs correlate.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

FMT_BF16 = 0
FMT_NVFP4 = 1
FMT_MXFP4 = 2
FMT_Q4_0 = 3

# stream ids of the seed sequence
S_WEIGHTS, S_PERM, S_ROUTING, S_HIDDEN, S_PRED, S_RWEIGHTS, S_SHARED, S_PREFILL, S_ALIAS = range(1, 10)
S_ROUTER, S_DRIFT = 10, 11


# ----------------------------------------------------------------------------- RNG

class Rng:
    """Counter-style access to a PCG64 stream identified by a tuple of ints."""

    def __init__(self, *key: int):
        ss = np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in key])
        self.bg = np.random.PCG64(ss)

    def raw(self, n: int) -> np.ndarray:
        return self.bg.random_raw(n).astype(np.uint64, copy=False)

    def uniform(self, n: int) -> np.ndarray:
        """Doubles in [0, 1): the top 53 bits of each raw draw."""
        return (self.raw(n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)

    def normal(self, n: int) -> np.ndarray:
        """Box-Muller on pairs of uniforms."""
        m = (n + 1) // 2
        u1 = self.uniform(m)
        u2 = self.uniform(m)
        r = np.sqrt(-2.0 * np.log1p(-u1))  # 1-u1 in (0, 1]
        z = np.concatenate([r * np.cos(2 * math.pi * u2), r * np.sin(2 * math.pi * u2)])
        return z[:n]

    def below(self, hi: int, n: int) -> np.ndarray:
        """Integers uniform in [0, hi)."""
        return np.minimum((self.uniform(n) * hi).astype(np.int64), hi - 1)

    def bytes(self, n: int) -> np.ndarray:
        w = self.raw((n + 7) // 8)
        return w.view(np.uint8)[:n]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bfloat16 bit patterns (round to nearest even), via torch."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# ---------------------------------------------------------------------- workloads

@dataclasses.dataclass
class Workload:
    name: str
    n_layers: int
    n_experts: int
    top_k: int
    hidden: int
    inter: int
    fmt: int
    n_slots: int
    per_layer_pools: bool
    batch: int
    steps: int
    seed: int
    routing: str = "zipf"          # "zipf" or "uniform"
    zipf_s: float = 1.1
    reuse: float = 0.0             # temporal reuse probability per route position
    shared_inter: int = 0          # 0: no shared expert
    fetch_cap: int = -1
    n_pred: int = 0                # look-ahead predictions per layer
    pred_keep: float = 0.7
    prefill_frac: float = 0.0      # fraction of experts pre-resident (layer 0)
    prefill_all: bool = False      # every layer's pool holds all its experts
    n_blob_alias: int = 0          # >0: keys share this many distinct host blobs
    batches: tuple = ()            # batch sweep (admission-only workload)

    @property
    def routes(self) -> int:
        return self.batch * self.top_k

    @property
    def blob_bytes(self) -> int:
        return blob_bytes(self.fmt, self.hidden, self.inter)

    @property
    def n_keys(self) -> int:
        return self.n_layers * self.n_experts


def workloads() -> dict[str, Workload]:
    return {
        # Tiny single layer, bf16, 6 slots, 64 decode steps.
        "tiny": Workload("tiny", 1, 16, 2, 64, 128, FMT_BF16, 6, False, 1, 64, 1001),
        # Qwen3-MoE-like offloaded decode: 40 layers x 256 experts, top-8, NVFP4,
        # one 3,164-slot pool, gated shared expert, temporal reuse tuned so the
        # LRU misses about 28 experts per token in steady state.
        "qwen3moe_decode": Workload("qwen3moe_decode", 40, 256, 8, 2048, 512, FMT_NVFP4, 3164,
                                    False, 1, 512, 1002, reuse=C2_REUSE, shared_inter=512),
        # Wide all-hit admission sweep: 48 per-layer pools of 2,100 slots holding
        # all 512 experts, top-10, uniform ids, 10..1,280 routes.
        "wide_admission": Workload("wide_admission", 48, 512, 10, 0, 0, FMT_BF16, 2100, True, 1,
                                   1, 1003, routing="uniform", prefill_all=True,
                                   batches=(1, 4, 8, 12, 13, 16, 24, 32, 48, 128)),
        # Wide decode step with misses: 600 rows x top-2 over 1,024 experts,
        # 1,100 slots, 30% of experts pre-resident, NVFP4.
        "wide_decode": Workload("wide_decode", 1, 1024, 2, 2048, 768, FMT_NVFP4, 1100, False, 600,
                                1, 1004, routing="uniform", prefill_frac=0.3),
        # Hybrid capped fetch + look-ahead prefetch: 48 layers x 256 experts,
        # bf16, 1,024 slots, cap 4, 8 predictions per layer; host blobs aliased.
        "hybrid_prefetch": Workload("hybrid_prefetch", 48, 256, 8, 4096, 1024, FMT_BF16, 1024,
                                    False, 1, 256, 1005, fetch_cap=4, n_pred=8, n_blob_alias=96),
    }


# Temporal-reuse probability of the Qwen3-MoE-like decode routing.  Chosen so
# that the steady-state LRU miss count is about 28 experts per token with 3,164
# slots; tests/test_synth.py checks that figure against the oracle.
C2_REUSE = 0.69


def scaled(w: Workload, **kw) -> Workload:
    return dataclasses.replace(w, **kw)


# --------------------------------------------------------------------- blob layout

def nvfp4_banks(hidden: int, inter: int) -> dict:
    """Byte offsets of the six banks and the global scales of an NVFP4 blob.

    gate/up codes [I, H/2], down codes [H, I/2] (two e2m1 per byte, even
    element in the low nibble); gate/up scales [I, H/16], down scales
    [H, I/16] (e4m3, one per 16 consecutive elements of a row); then three fp32
    global scales (gate, up, down) padded to 16 bytes.
    """
    ih = inter * hidden
    o = {"code": [0, ih // 2, ih], "scale": [3 * ih // 2, 3 * ih // 2 + ih // 16,
                                             3 * ih // 2 + 2 * (ih // 16)]}
    o["glob"] = 3 * ih // 2 + 3 * (ih // 16)
    o["total"] = o["glob"] + 16
    return o


def mxfp4_banks(hidden: int, inter: int) -> dict:
    """Byte offsets of an MXFP4 blob: the same code banks as NVFP4, then
    gate/up scales [I, H/32] and down scales [H, I/32] (E8M0, one per 32
    consecutive elements of a row); no global scales; padded to 16 bytes."""
    ih = inter * hidden
    o = {"code": [0, ih // 2, ih], "scale": [3 * ih // 2, 3 * ih // 2 + ih // 32,
                                             3 * ih // 2 + 2 * (ih // 32)]}
    o["end"] = 3 * ih // 2 + 3 * (ih // 32)
    o["total"] = (o["end"] + 15) // 16 * 16
    return o


def q4_banks(hidden: int, inter: int) -> dict:
    """Byte offsets of a Q4_0 blob (banked): the code banks as NVFP4 (4-bit
    unsigned codes q, weight = d * (q - 8)), then gate/up scales [I, H/32]
    and down scales [H, I/32] as fp16 d, one per 32 consecutive row elements."""
    ih = inter * hidden
    o = {"code": [0, ih // 2, ih], "scale": [3 * ih // 2, 3 * ih // 2 + ih // 16,
                                             3 * ih // 2 + 2 * (ih // 16)]}
    o["end"] = 3 * ih // 2 + 3 * (ih // 16)
    o["total"] = (o["end"] + 15) // 16 * 16
    return o


def blob_bytes(fmt: int, hidden: int, inter: int) -> int:
    if fmt == FMT_BF16:
        return 6 * hidden * inter
    if fmt == FMT_MXFP4:
        return mxfp4_banks(hidden, inter)["total"]
    if fmt == FMT_Q4_0:
        return q4_banks(hidden, inter)["total"]
    return nvfp4_banks(hidden, inter)["total"]


def fill_blob(out: np.ndarray, fmt: int, hidden: int, inter: int, rng: Rng) -> None:
    """Write one expert blob into the uint8 array ``out``."""
    if fmt == FMT_BF16:
        w = rng.normal(3 * hidden * inter) * 0.02
        out[:] = to_bf16_bits(w).view(np.uint8)
        return
    if fmt == FMT_Q4_0:  # random codes; fp16 block scales in [0.001, 0.005)
        o = q4_banks(hidden, inter)
        n_codes = o["scale"][0]
        out[:n_codes] = rng.bytes(n_codes)
        n_sc = (o["end"] - n_codes) // 2
        d = (0.001 + 0.004 * rng.uniform(n_sc)).astype(np.float16)
        out[n_codes:o["end"]] = d.view(np.uint8)
        out[o["end"]:o["total"]] = 0
        return
    if fmt == FMT_MXFP4:  # random codes; block scales 2^-9 .. 2^-6 (E8M0 118..121)
        o = mxfp4_banks(hidden, inter)
        n_codes = o["scale"][0]
        out[:n_codes] = rng.bytes(n_codes)
        out[n_codes:o["end"]] = np.uint8(118) + (rng.bytes(o["end"] - n_codes) & np.uint8(3))
        out[o["end"]:o["total"]] = 0
        return
    o = nvfp4_banks(hidden, inter)
    n_codes = o["scale"][0]
    out[:n_codes] = rng.bytes(n_codes)
    n_scales = o["glob"] - n_codes
    out[n_codes:o["glob"]] = np.uint8(0x28) + (rng.bytes(n_scales) & np.uint8(0x0F))
    g = (0.008 + 0.006 * rng.uniform(3)).astype(np.float32)
    out[o["glob"]:o["glob"] + 12] = g.view(np.uint8)
    out[o["glob"] + 12:o["total"]] = 0


def alloc_host(nbytes: int, pinned: bool):
    import torch
    return torch.empty(nbytes, dtype=torch.uint8, pin_memory=pinned)


class HostBlobs:
    """Expert blobs in (pinned) host memory, one row per distinct blob.

    ``key_to_blob[layer*E + e]`` gives the row holding that expert's weights
    (the identity unless the workload aliases keys onto fewer blobs).
    """

    def __init__(self, w: Workload, pinned: bool = True, stride_align: int = 256,
                 threads: int | None = None):
        self.w = w
        self.nbytes = w.blob_bytes
        self.stride = (self.nbytes + stride_align - 1) // stride_align * stride_align
        n_keys = w.n_keys
        if w.n_blob_alias:
            self.n_blobs = w.n_blob_alias
            self.key_to_blob = Rng(w.seed, S_ALIAS).below(self.n_blobs, n_keys).astype(np.int64)
        else:
            self.n_blobs = n_keys
            self.key_to_blob = np.arange(n_keys, dtype=np.int64)
        self.buf = alloc_host(self.n_blobs * self.stride, pinned)
        arr = self.buf.numpy()

        def one(i):
            fill_blob(arr[i * self.stride:i * self.stride + self.nbytes], w.fmt, w.hidden,
                      w.inter, Rng(w.seed, S_WEIGHTS, i))

        nt = threads or min(16, os.cpu_count() or 1)
        if self.n_blobs > 1 and nt > 1:
            with _cf.ThreadPoolExecutor(nt) as ex:
                list(ex.map(one, range(self.n_blobs)))
        else:
            for i in range(self.n_blobs):
                one(i)

    def blob(self, key: int) -> np.ndarray:
        i = int(self.key_to_blob[key])
        return self.buf.numpy()[i * self.stride:i * self.stride + self.nbytes]

    def addr(self, key: int) -> int:
        return self.buf.data_ptr() + int(self.key_to_blob[key]) * self.stride

    def addrs(self) -> np.ndarray:
        return (self.buf.data_ptr() + self.key_to_blob * self.stride).astype(np.uint64)

    def layer_blobs(self, layer: int) -> list:
        E = self.w.n_experts
        return [self.blob(layer * E + e) for e in range(E)]


def make_shared(w: Workload, layer: int = 0):
    """Layer's shared expert blob (uint8) and its sigmoid-gate vector (bf16 bits [H])."""
    if not w.shared_inter:
        return None, None
    blob = np.empty(blob_bytes(w.fmt, w.hidden, w.shared_inter), np.uint8)
    fill_blob(blob, w.fmt, w.hidden, w.shared_inter, Rng(w.seed, S_SHARED, layer, 0))
    gate = to_bf16_bits(Rng(w.seed, S_SHARED, layer, 1).normal(w.hidden) * 0.02)
    return blob, gate


# ------------------------------------------------------------------------ routing

def zipf_cdf(n: int, s: float) -> np.ndarray:
    p = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(p)
    return c / c[-1]


def layer_perms(w: Workload) -> np.ndarray:
    r = Rng(w.seed, S_PERM)
    return np.stack([np.argsort(r.uniform(w.n_experts), kind="stable")
                     for _ in range(w.n_layers)]).astype(np.int32)


def make_routing(w: Workload, steps: int | None = None, batch: int | None = None,
                 start: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """ids [steps, L, B, k] int32 and weights [steps, L, B, k] float32."""
    T = w.steps if steps is None else steps
    B = w.batch if batch is None else batch
    L, E, k = w.n_layers, w.n_experts, w.top_k
    ids = np.empty((T, L, B, k), np.int32)
    if w.routing == "uniform":
        for t in range(T):
            r = Rng(w.seed, S_ROUTING, start + t, B)
            for l in range(L):
                for b in range(B):
                    row = []
                    while len(row) < k:
                        e = int(r.below(E, 1)[0])
                        if e not in row:
                            row.append(e)
                    ids[t, l, b] = row
    else:
        cdf = zipf_cdf(E, w.zipf_s)
        perm = layer_perms(w)
        prev = None
        # temporal reuse needs the previous step: always generate from step 0
        for t in range(start + T):
            r = Rng(w.seed, S_ROUTING, t, B)
            cur = np.empty((L, B, k), np.int32)
            for l in range(L):
                for b in range(B):
                    row: list[int] = []
                    for j in range(k):
                        if prev is not None and w.reuse > 0 and r.uniform(1)[0] < w.reuse:
                            e = int(prev[l, b, j])
                            if e not in row:
                                row.append(e)
                                continue
                        while True:
                            rank = int(np.searchsorted(cdf, r.uniform(1)[0], side="right"))
                            e = int(perm[l, min(rank, E - 1)])
                            if e not in row:
                                row.append(e)
                                break
                    cur[l, b] = row
            if t >= start:
                ids[t - start] = cur
            prev = cur
    wts = np.empty((T, L, B, k), np.float32)
    for t in range(T):
        z = Rng(w.seed, S_RWEIGHTS, start + t, B).normal(L * B * k).reshape(L, B, k)
        z = np.exp(z - z.max(axis=-1, keepdims=True))
        wts[t] = (z / z.sum(axis=-1, keepdims=True)).astype(np.float32)
    return ids, wts


def make_hidden(w: Workload, step: int, batch: int | None = None) -> np.ndarray:
    """x [L, B, H] as bf16 bits, independent N(0, 1) per (step, layer, row)."""
    B = w.batch if batch is None else batch
    z = Rng(w.seed, S_HIDDEN, step, B).normal(w.n_layers * B * w.hidden)
    return to_bf16_bits(z).reshape(w.n_layers, B, w.hidden)


def make_router(w: Workload, layer: int) -> np.ndarray:
    """Router weights of a layer, bf16 bits [E][H] (row e: expert e)."""
    z = Rng(w.seed, S_ROUTER, layer).normal(w.n_experts * w.hidden) / math.sqrt(w.hidden)
    return to_bf16_bits(z).reshape(w.n_experts, w.hidden)


def drift_stream(w: Workload, step: int, s: float, batch: int | None = None) -> np.ndarray:
    """x [L, B, H] as bf16 bits: layer 0 N(0, 1), then x_{l+1} = (x_l + s n_l)
    / sqrt(1 + s^2) (unit variance throughout)."""
    B = w.batch if batch is None else batch
    r = Rng(w.seed, S_DRIFT, step, B)
    x = np.empty((w.n_layers, B, w.hidden), np.float32)
    x[0] = r.normal(B * w.hidden).reshape(B, w.hidden)
    for l in range(1, w.n_layers):
        n = r.normal(B * w.hidden).reshape(B, w.hidden)
        x[l] = (x[l - 1] + s * n) / math.sqrt(1.0 + s * s)
    return to_bf16_bits(x)


def make_predictions(w: Workload, ids_next_layer: np.ndarray, step: int, layer: int) -> np.ndarray:
    """Look-ahead predictions for layer+1: each true id kept with p=pred_keep,
    else uniform; ``n_pred`` entries (true ids first, padded uniform)."""
    r = Rng(w.seed, S_PRED, step, layer)
    true = list(np.asarray(ids_next_layer).ravel())[: w.n_pred]
    out = []
    for e in true:
        if r.uniform(1)[0] < w.pred_keep:
            out.append(int(e))
        else:
            out.append(int(r.below(w.n_experts, 1)[0]))
    while len(out) < w.n_pred:
        out.append(int(r.below(w.n_experts, 1)[0]))
    return np.asarray(out, np.int32)


def prefill_ids(w: Workload, layer: int = 0) -> np.ndarray:
    """Experts placed in the cache before the first step."""
    if w.prefill_all:
        return np.arange(w.n_experts, dtype=np.int32)
    if w.prefill_frac > 0:
        n = int(round(w.prefill_frac * w.n_experts))
        perm = np.argsort(Rng(w.seed, S_PREFILL, layer).uniform(w.n_experts), kind="stable")
        return np.sort(perm[:n]).astype(np.int32)
    return np.zeros(0, np.int32)


def uniform_ids(w: Workload, batch: int, salt: int) -> np.ndarray:
    """[L, batch*k] distinct-per-row uniform ids (admission sweep)."""
    ids, _ = make_routing(scaled(w, routing="uniform", batch=batch), steps=1, batch=batch,
                          start=salt)
    return ids[0].reshape(w.n_layers, batch * w.top_k)
