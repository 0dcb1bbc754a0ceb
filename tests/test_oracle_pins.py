"""Pins of the CPU oracle to things other than itself (no GPU needed).

* the cache: a brute-force history-scan re-derivation on tiny random pools,
  invariants, and the pages' worked examples (tests/golden/worked_examples.json);
* the number formats: the OCP e2m1 table (tests/golden/e2m1_ocp.json) and
  torch's float8_e4m3fn / bfloat16 conversions, exhaustively;
* the layer math: closed forms (zero input, a one-weight expert), numpy fp64
  matrix products, complementary route masks.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.bruteforce import Brute

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------- cache

def _state_pairs(oc: oracle.OracleCache, bf: Brute):
    st = oc.state()
    sk = st["slot_key"].reshape(oc.n_pools, oc.S)
    for p in range(oc.n_pools):
        assert list(sk[p]) == bf.slot_key[p], f"pool {p} slot_key"
    for layer in range(oc.L):
        assert oc.stats(layer) == bf.stats[layer], f"layer {layer} stats"
    assert list(st["decode_freq"]) == bf.decode_freq


def _invariants(oc: oracle.OracleCache, routes_by_layer):
    st = oc.state()
    sk = st["slot_key"].reshape(oc.n_pools, oc.S)
    mp = st["map"]
    # map and slot->key agree, no key twice
    for key in range(oc.L * oc.E):
        layer = key // oc.E
        p = layer if oc.per_layer else 0
        if mp[key] >= 0:
            assert sk[p][mp[key]] == key
    for p in range(oc.n_pools):
        keys = [k for k in sk[p] if k >= 0]
        assert len(keys) == len(set(keys)) <= oc.S
        for s, k in enumerate(sk[p]):
            if k >= 0:
                assert mp[k] == s
    # every route >= 0 maps to a slot that holds its expert
    for layer, (ids, slots) in routes_by_layer.items():
        p = layer if oc.per_layer else 0
        for e, s in zip(ids, slots):
            if s >= 0:
                assert sk[p][s] == layer * oc.E + e
            else:
                assert not (0 <= e < oc.E) or mp[layer * oc.E + e] < 0
    for layer in range(oc.L):
        s = oc.stats(layer)
        assert s["hits"] + s["misses"] == s["lookups"]
        assert s["fetched"] <= s["misses"]


@pytest.mark.parametrize("seed", range(12))
def test_oracle_matches_bruteforce_random(seed):
    rnd = random.Random(seed)
    L = rnd.choice([1, 2, 3])
    E = rnd.randint(3, 16)
    S = rnd.randint(1, 6)
    per_layer = rnd.random() < 0.4
    oc = oracle.OracleCache(L, E, S, per_layer)
    oc_split = oracle.OracleCache(L, E, S, per_layer)
    bf = Brute(L, E, S, per_layer)
    if rnd.random() < 0.5:  # prefill some experts of layer 0
        n = rnd.randint(0, min(S, E))
        ids = rnd.sample(range(E), n)
        oc.prefill(0, ids)
        oc_split.prefill(0, ids)
        bf.prefill(0, ids)
    for step in range(150):
        op = rnd.random()
        layer = rnd.randrange(L)
        if op < 0.08:
            slot = rnd.randrange(S)
            pin = rnd.random() < 0.5
            oc.pin(layer, slot, pin)
            oc_split.pin(layer, slot, pin)
            bf.pin(layer, slot, pin)
        elif op < 0.25:
            pred = [rnd.randint(-1, E) for _ in range(rnd.randint(0, 6))]
            a = oc.prefetch(layer, pred)
            assert oc_split.prefetch(layer, pred) == a
            assert bf.prefetch(layer, pred) == a
        else:
            R = rnd.randint(0, 10)
            ids = [rnd.randint(-1, E) if rnd.random() < 0.1 else rnd.randrange(E) for _ in range(R)]
            cap = rnd.choice([-1, -1, 0, 1, 2, 3])
            a = oc.admit(layer, ids, cap)
            b = bf.admit(layer, ids, cap)
            sw = rnd.randint(1, 4)
            c = oc_split.admit(layer, ids, cap, split_width=sw)
            assert list(a["slots"]) == b["slots"], (step, ids)
            assert a["plan"] == b["plan"]
            assert a["groups"] == b["groups"]
            # a split admission equals the single one
            assert list(c["slots"]) == list(a["slots"])
            assert c["plan"] == a["plan"] and c["groups"] == a["groups"]
            nd = len({e for e in ids if 0 <= e < E})
            assert c["widths"] == [min(sw, nd - i) for i in range(0, nd, sw)]
            _invariants(oc, {layer: (ids, list(a["slots"]))})
            if rnd.random() < 0.1:  # a failed copy rolls its bookings back
                oc.rollback(a["plan"])
                oc_split.rollback(a["plan"])
                bf.rollback(a["plan"])
        _state_pairs(oc, bf)
        _state_pairs(oc_split, bf)


def test_lru_order_is_stamp_then_slot():
    oc = oracle.OracleCache(1, 8, 4)
    assert oc.lru_order() == [0, 1, 2, 3]  # all empty, slot order
    oc.admit(0, [5, 2])          # clock 2: 2 -> slot 0, 5 -> slot 1
    oc.admit(0, [7])             # clock 3: 7 -> slot 2
    assert oc.lru_order() == [3, 0, 1, 2]
    r = oc.admit(0, [5, 6])      # 5 hit (slot 1), 6 -> empty slot 3
    assert list(r["slots"]) == [1, 3]
    assert oc.lru_order() == [0, 2, 1, 3]
    r = oc.admit(0, [1, 0])      # two misses take slots 0 (expert 2) and 2 (expert 7)
    assert r["plan"] == [(0, 0, 0), (2, 0, 1)]
    assert list(r["slots"]) == [2, 0]


def test_all_hit_steps_never_evict():
    rnd = random.Random(7)
    oc = oracle.OracleCache(2, 32, 40, per_layer=True)
    for layer in range(2):
        oc.prefill(layer, list(range(32)))
    for _ in range(100):
        layer = rnd.randrange(2)
        ids = [rnd.randrange(32) for _ in range(rnd.randint(1, 64))]
        r = oc.admit(layer, ids)
        assert r["plan"] == []
        assert all(s >= 0 for s in r["slots"])
    for layer in range(2):
        st = oc.stats(layer)
        assert st["evictions"] == 0 and st["misses"] == 0 and st["fetched"] == 0


def test_capacity_shortfall_is_an_implicit_cap():
    oc = oracle.OracleCache(1, 16, 3)
    oc.pin(0, 1, True)
    r = oc.admit(0, [9, 4, 12, 4])  # 3 distinct misses, 2 evictable slots
    assert r["plan"] == [(0, 0, 4), (2, 0, 9)]
    assert list(r["slots"]) == [2, 0, -1, 0]
    st = oc.stats(0)
    assert st["status_bits"] & oracle.STATUS_CAPACITY
    assert st["misses"] == 3 and st["fetched"] == 2 and st["overflow_routes"] == 1


def test_route_split_example():
    """[11, 42] -> cache [3, -1] with a fetch cap of 0 and expert 11 in slot 3."""
    g = gold("worked_examples.json")["route_split"]
    oc = oracle.OracleCache(1, 64, 8)
    oc.prefill(0, [1, 2, 5, 11])  # 11 lands in slot 3
    r = oc.admit(0, g["ids"], cap=0)
    assert list(r["slots"]) == g["cache_result"]
    assert oc.stats(0)["overflow_routes"] == 1


def test_wide_step_example():
    g = gold("worked_examples.json")["wide_step"]
    rows, k = g["rows"], g["top_k"]
    # 150 rows x top-2 over experts 0..159: row i routes to i and i+10 (mod 160)
    ids = [e for i in range(rows) for e in (i % 160, (i + 10) % 160)]
    assert len(set(ids)) == g["distinct_experts"]
    resident = [3, 17, 42, 64, 99, 120, 155]
    assert len(resident) == g["resident"]
    for split in (0, 128):
        oc = oracle.OracleCache(1, 256, 400)
        oc.prefill(0, resident)
        r = oc.admit(0, ids, split_width=split)
        st = oc.stats(0)
        assert (st["lookups"], st["misses"], st["calls"]) == (g["lookups"], g["misses"], g["calls"])
        assert int(oc.state()["decode_freq"].sum()) == g["decode_freq_sum"]
        if split:
            assert r["widths"] == g["query_widths"]
        # an 8-route step stays one query
        r8 = oc.admit(0, ids[:g["narrow_routes"]], split_width=split)
        assert len(r8["widths"]) == g["narrow_query_widths_count"]


def test_on_demand_chunk_example():
    g = gold("worked_examples.json")["on_demand_chunk"]
    ids = list(range(0, 2 * g["routes"], 2))  # 300 distinct experts of 640
    oc = oracle.OracleCache(1, g["n_experts"], 1000)
    r = oc.admit(0, ids, split_width=128)
    assert r["widths"] == g["query_widths"]


def _guard_case(demands: int):
    """3-slot pool: slot 0 holds a resident demanded `demands` times, the
    other two slots hold experts touched after it; then a never-seen expert is
    predicted."""
    oc = oracle.OracleCache(1, 32, 3)
    for _ in range(demands):
        oc.admit(0, [5])
    oc.admit(0, [6, 7])
    assert oc.lru_order()[0] == oc.state()["map"][5]
    plan = oc.prefetch(0, [20])
    return oc, plan


def test_guard_example():
    g = gold("worked_examples.json")["guard"]
    oc, plan = _guard_case(g["protected_demand_accesses_under_formula"])
    st = oc.stats(0)
    assert plan == [] and st["pf_dropped_guard"] == 1 and st["pf_evictions"] == 0
    assert oc.state()["map"][5] >= 0
    r = oc.admit(0, [5])  # still a demand hit
    assert oc.stats(0)["hits"] == st["hits"] + 1 and r["plan"] == []
    oc, plan = _guard_case(g["cold_demand_accesses"])
    assert len(plan) == 1 and oc.stats(0)["pf_evictions"] == 1
    assert oc.state()["map"][5] < 0
    # the page's 3-access case: not protected under the stated formula
    oc, plan = _guard_case(g["page_warm_demand_accesses"])
    assert len(plan) == 1


def test_guard_threshold_integer_form():
    """score_res > 1.25 * score_pred + 1024 evaluated exactly: with a
    never-seen prediction (score 0) a resident is protected iff its score
    exceeds 1024, i.e. at 4 recent demand accesses but not at 3."""
    for demands, protected in [(2, False), (3, False), (4, True), (6, True)]:
        oc, plan = _guard_case(demands)
        assert (plan == []) == protected, demands


def test_prefetch_fill_protects_against_same_batch():
    oc = oracle.OracleCache(2, 16, 2)
    oc.admit(0, [1])                  # clock 2: expert (0,1) -> slot 0
    oc.admit(1, [2])                  # clock 3: expert (1,2) -> slot 1 (touched now)
    plan = oc.prefetch(1, [3, 4, 5])  # only slot 0 is evictable; a fill takes it once
    assert plan == [(0, 1, 3)]
    st = oc.stats(1)
    assert st["pf_no_victim"] == 2 and st["pf_filled"] == 1 and st["pf_requests"] == 3
    assert st["pf_evictions"] == 1


def test_prefetch_never_touches_current_admission():
    oc = oracle.OracleCache(2, 16, 4)
    oc.admit(0, [1, 2, 3, 4])       # fills the whole pool in one admission
    plan = oc.prefetch(1, [7, 8])   # nothing evictable: all touched at this clock
    assert plan == [] and oc.stats(1)["pf_no_victim"] == 2


def test_prefetch_ignores_invalid_and_resident():
    oc = oracle.OracleCache(1, 8, 4)
    oc.admit(0, [2])
    a = oc.admit(0, [3])
    plan = oc.prefetch(0, [-1, 8, 2, 2, 5])
    st = oc.stats(0)
    assert st["pf_invalid"] == 2 and st["pf_resident"] == 1 and st["pf_requests"] == 2
    assert [p[2] for p in plan] == [5]
    assert a["plan"][0][0] != plan[0][0]


# ---------------------------------------------------------------------- formats

def test_e2m1_table():
    g = gold("e2m1_ocp.json")
    for c, v in zip(g["codes"], g["values"]):
        got = oracle.e2m1(c)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), c


def test_e4m3_exhaustive_against_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for b in range(256):
        got = oracle.e4m3(b)
        want = float(ref[b])
        if math.isnan(want):
            assert math.isnan(got), b
        else:
            assert got == want, b
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x01) == 2.0 ** -9 and oracle.e4m3(0x38) == 1.0


def test_e8m0_exhaustive_against_torch():
    """E8M0, the MXFP4 block scale (OCP Microscaling Formats): every code
    against torch's float8_e8m0fnu, plus the spec's anchors."""
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no float8_e8m0fnu")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    for b in range(256):
        got, want = oracle.e8m0(b), float(ref[b])
        if math.isnan(want):
            assert math.isnan(got), b
        else:
            assert got == want, b
    assert oracle.e8m0(127) == 1.0 and oracle.e8m0(0) == 2.0 ** -127
    assert oracle.e8m0(254) == 2.0 ** 127 and math.isnan(oracle.e8m0(255))


def test_f16_exhaustive_against_numpy():
    """IEEE binary16 (the Q4_0 block scale): every code against numpy's float16."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16(int(b)) for b in bits])
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[~fin]))


def test_bf16_against_torch():
    bits = np.arange(0, 65536, 37, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[np.isnan(ref)]))


def _np_dequant_nvfp4(blob: np.ndarray, H: int, I: int, which: int) -> np.ndarray:
    """Independent numpy decode of one NVFP4 matrix of a blob."""
    table = np.array(gold("e2m1_ocp.json")["values"])
    banks = synth.nvfp4_banks(H, I)
    rows, cols = (H, I) if which == 2 else (I, H)
    codes = blob[banks["code"][which]:banks["code"][which] + rows * cols // 2]
    nib = np.empty(rows * cols, np.int64)
    nib[0::2] = codes & 15
    nib[1::2] = codes >> 4
    sc = blob[banks["scale"][which]:banks["scale"][which] + rows * cols // 16]
    scale = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    g = float(blob[banks["glob"] + 4 * which:banks["glob"] + 4 * which + 4].view(np.float32)[0])
    w = table[nib].reshape(rows, cols) * np.repeat(scale.reshape(rows, cols // 16), 16, axis=1)
    return w * g


def _np_dequant_mxfp4(blob: np.ndarray, H: int, I: int, which: int) -> np.ndarray:
    """Independent numpy decode of one MXFP4 matrix: e2m1 codes from the OCP
    table fixture, one power-of-two scale per 32 row elements."""
    table = np.array(gold("e2m1_ocp.json")["values"])
    banks = synth.mxfp4_banks(H, I)
    rows, cols = (H, I) if which == 2 else (I, H)
    codes = blob[banks["code"][which]:banks["code"][which] + rows * cols // 2]
    nib = np.empty(rows * cols, np.int64)
    nib[0::2] = codes & 15
    nib[1::2] = codes >> 4
    sc = blob[banks["scale"][which]:banks["scale"][which] + rows * cols // 32].astype(np.int64)
    scale = np.ldexp(1.0, sc - 127)
    return table[nib].reshape(rows, cols) * np.repeat(scale.reshape(rows, cols // 32), 32, axis=1)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_mxfp4_dequant_against_numpy(which):
    H, I = 64, 96
    blob = np.empty(synth.blob_bytes(synth.FMT_MXFP4, H, I), np.uint8)
    synth.fill_blob(blob, synth.FMT_MXFP4, H, I, synth.Rng(6, which))
    assert oracle.blob_bytes(oracle.FMT_MXFP4, H, I) == len(blob) == 3 * H * I // 2 + 3 * H * I // 32
    got = oracle.dequant(oracle.FMT_MXFP4, blob, H, I, which)
    assert np.array_equal(got, _np_dequant_mxfp4(blob, H, I, which))
    # a planted change of one scale moves exactly its 32 elements by a power of two
    banks = synth.mxfp4_banks(H, I)
    b2 = blob.copy()
    b2[banks["scale"][which]] += 1
    d = oracle.dequant(oracle.FMT_MXFP4, b2, H, I, which)
    assert np.array_equal(d[0, :32], 2 * got[0, :32]) and np.array_equal(d[0, 32:], got[0, 32:])


def _np_dequant_q4(blob: np.ndarray, H: int, I: int, which: int) -> np.ndarray:
    """Independent numpy decode of one Q4_0 matrix (banked): d * (q - 8)."""
    banks = synth.q4_banks(H, I)
    rows, cols = (H, I) if which == 2 else (I, H)
    codes = blob[banks["code"][which]:banks["code"][which] + rows * cols // 2]
    q = np.empty(rows * cols, np.int64)
    q[0::2] = codes & 15
    q[1::2] = codes >> 4
    sc = blob[banks["scale"][which]:banks["scale"][which] + rows * cols // 16]
    d = sc.view(np.float16).astype(np.float64).reshape(rows, cols // 32)
    return (q - 8).reshape(rows, cols) * np.repeat(d, 32, axis=1)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_q4_0_dequant_against_numpy(which):
    H, I = 64, 96
    blob = np.empty(synth.blob_bytes(synth.FMT_Q4_0, H, I), np.uint8)
    synth.fill_blob(blob, synth.FMT_Q4_0, H, I, synth.Rng(7, which))
    assert oracle.blob_bytes(oracle.FMT_Q4_0, H, I) == len(blob) == 3 * H * I // 2 + 3 * H * I // 16
    got = oracle.dequant(oracle.FMT_Q4_0, blob, H, I, which)
    assert np.array_equal(got, _np_dequant_q4(blob, H, I, which))
    # code 8 is zero whatever the scale; code 0 is -8 d
    banks = synth.q4_banks(H, I)
    b2 = blob.copy()
    b2[banks["code"][which]] = 0x08  # element 0: q = 8, element 1: q = 0
    d = oracle.dequant(oracle.FMT_Q4_0, b2, H, I, which)
    d0 = float(blob[banks["scale"][which]:banks["scale"][which] + 2].view(np.float16)[0])
    assert d[0, 0] == 0.0 and d[0, 1] == -8 * d0


@pytest.mark.parametrize("which", [0, 1, 2])
def test_nvfp4_dequant_against_numpy(which):
    H, I = 64, 96
    blob = np.empty(synth.blob_bytes(synth.FMT_NVFP4, H, I), np.uint8)
    synth.fill_blob(blob, synth.FMT_NVFP4, H, I, synth.Rng(5, which))
    assert oracle.blob_bytes(oracle.FMT_NVFP4, H, I) == len(blob)
    got = oracle.dequant(oracle.FMT_NVFP4, blob, H, I, which)
    assert np.array_equal(got, _np_dequant_nvfp4(blob, H, I, which))


def _np_ffn(Wg, Wu, Wd, x):
    g = Wg @ x
    u = Wu @ x
    return Wd @ (g / (1 + np.exp(-g)) * u)


@pytest.mark.parametrize("fmt", [oracle.FMT_BF16, oracle.FMT_NVFP4, oracle.FMT_MXFP4,
                                 oracle.FMT_Q4_0])
def test_expert_ffn_against_numpy(fmt):
    H, I = 64, 128
    blob = np.empty(synth.blob_bytes(fmt, H, I), np.uint8)
    synth.fill_blob(blob, fmt, H, I, synth.Rng(9, fmt))
    x = synth.to_bf16_bits(synth.Rng(10).normal(H))
    W = [oracle.dequant(fmt, blob, H, I, m) for m in range(3)]
    if fmt == oracle.FMT_BF16:  # independent decode of the bf16 banks
        raw = blob.view(np.uint16)
        ref = torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        assert np.array_equal(W[0].ravel(), ref[:H * I])
        assert np.array_equal(W[1].ravel(), ref[H * I:2 * H * I])
        assert np.array_equal(W[2].ravel(), ref[2 * H * I:])
    xd = np.array([oracle.bf16(int(v)) for v in x])
    y = oracle.expert_ffn(fmt, blob, H, I, x)
    assert np.allclose(y, _np_ffn(W[0], W[1], W[2], xd), rtol=1e-12, atol=1e-14)


def test_one_weight_expert_closed_form():
    """Only Wg[2,5]=a, Wu[2,5]=b, Wd[7,2]=c are nonzero: y[7] = c*silu(a x5)*(b x5)."""
    H, I = 32, 32
    w = np.zeros(3 * H * I, np.float32)
    a, b, c = 0.75, -1.5, 2.0
    w[2 * H + 5] = a
    w[H * I + 2 * H + 5] = b
    w[2 * H * I + 7 * I + 2] = c
    blob = synth.to_bf16_bits(w).view(np.uint8)
    x = np.zeros(H, np.float32)
    x[5] = 1.25
    y = oracle.expert_ffn(oracle.FMT_BF16, blob, H, I, synth.to_bf16_bits(x))
    g = a * 1.25
    want = c * (g / (1 + math.exp(-g))) * (b * 1.25)
    assert y[7] == pytest.approx(want, rel=1e-15)
    assert np.count_nonzero(y) == 1


def _set_code(blob, bank_off, row, k, cols, code):
    """Put a 4-bit code at element (row, k) of a code bank (even element in the low nibble)."""
    i = bank_off + row * (cols // 2) + k // 2
    blob[i] = (blob[i] & 0xF0) | code if k % 2 == 0 else (blob[i] & 0x0F) | (code << 4)


@pytest.mark.parametrize("fmt", [synth.FMT_MXFP4, synth.FMT_Q4_0])
def test_one_weight_expert_closed_form_4bit_formats(fmt):
    """Only Wg[2,5] = 0.75, Wu[2,5] = -1.5 and Wd[7,2] = 2 are nonzero, spelled
    in the format's own codes and block scales: y[7] = 2 silu(0.75 x5) (-1.5 x5)."""
    H, I = 64, 64
    blob = np.zeros(synth.blob_bytes(fmt, H, I), np.uint8)
    if fmt == synth.FMT_MXFP4:
        o = synth.mxfp4_banks(H, I)  # codes 0 are +0; scales E8M0
        blob[o["scale"][0]:o["end"]] = 127
        _set_code(blob, o["code"][0], 2, 5, H, 0x3)        # e2m1 1.5, block scale 2^-1
        blob[o["scale"][0] + 2 * (H // 32) + 0] = 126
        _set_code(blob, o["code"][1], 2, 5, H, 0x8 | 0x3)  # -1.5, scale 1
        _set_code(blob, o["code"][2], 7, 2, I, 0x4)        # 2.0, scale 1
    else:
        o = synth.q4_banks(H, I)  # code 8 is zero; scales fp16 d
        blob[:o["scale"][0]] = 0x88
        d = np.full((o["end"] - o["scale"][0]) // 2, 0.5, np.float16)
        blob[o["scale"][0]:o["end"]] = d.view(np.uint8)
        _set_code(blob, o["code"][0], 2, 5, H, 8 + 3)      # 0.25 * 3 below
        blob[o["scale"][0] + 2 * (2 * (H // 32)):][:2] = np.array([0.25], np.float16).view(np.uint8)
        _set_code(blob, o["code"][1], 2, 5, H, 8 - 3)      # 0.5 * -3
        _set_code(blob, o["code"][2], 7, 2, I, 8 + 4)      # 0.5 * 4
    W = [oracle.dequant(fmt, blob, H, I, m_) for m_ in range(3)]
    assert W[0][2, 5] == 0.75 and W[1][2, 5] == -1.5 and W[2][7, 2] == 2.0
    assert [np.count_nonzero(w_) for w_ in W] == [1, 1, 1]
    x = np.zeros(H, np.float32)
    x[5] = 1.25
    y = oracle.expert_ffn(fmt, blob, H, I, synth.to_bf16_bits(x))
    g = 0.75 * 1.25
    assert y[7] == pytest.approx(2.0 * (g / (1 + math.exp(-g))) * (-1.5 * 1.25), rel=1e-15)
    assert np.count_nonzero(y) == 1


def test_layer_zero_input_and_masks():
    w = synth.scaled(synth.workloads()["tiny"], shared_inter=64)
    blobs = synth.HostBlobs(w, pinned=False)
    sblob, sgate = synth.make_shared(w)
    ids, wts = synth.make_routing(w, steps=1)
    x = synth.make_hidden(w, 0)[0]
    zero = np.zeros_like(x)
    out0 = oracle.layer(w.fmt, blobs.layer_blobs(0), w.n_experts, w.hidden, w.inter, zero,
                        ids[0, 0], wts[0, 0], shared_blob=sblob, shared_inter=64,
                        shared_gate_w=sgate)
    assert np.all(out0 == 0.0)
    full = oracle.layer(w.fmt, blobs.layer_blobs(0), w.n_experts, w.hidden, w.inter, x,
                        ids[0, 0], wts[0, 0])
    m = np.array([[1, 0]], np.uint8)
    part = [oracle.layer(w.fmt, blobs.layer_blobs(0), w.n_experts, w.hidden, w.inter, x,
                         ids[0, 0], wts[0, 0], mask=mm) for mm in (m, 1 - m)]
    assert np.allclose(part[0] + part[1], full, rtol=0, atol=1e-15)
    # routed part = sum of weighted single-expert FFNs
    want = sum(float(wts[0, 0, 0, j]) * oracle.expert_ffn(
        w.fmt, blobs.blob(int(ids[0, 0, 0, j])), w.hidden, w.inter, x[0]) for j in range(2))
    assert np.allclose(full[0], want, rtol=1e-13, atol=1e-15)
    # sigmoid gate: a zero gate vector gives exactly half of the shared FFN
    zg = np.zeros_like(sgate)
    s_only = oracle.layer(w.fmt, blobs.layer_blobs(0), w.n_experts, w.hidden, w.inter, x,
                          ids[0, 0], np.zeros_like(wts[0, 0]), shared_blob=sblob,
                          shared_inter=64, shared_gate_w=zg)
    ffn_s = oracle.expert_ffn(w.fmt, sblob, w.hidden, 64, x[0])
    assert np.allclose(s_only[0], 0.5 * ffn_s, rtol=1e-14, atol=1e-16)


def _one_weight_bf16_blob(H, I, a, b, c):
    """bf16 expert whose only nonzero weights are Wg[2,5] = a, Wu[2,5] = b, Wd[7,2] = c."""
    w = np.zeros(3 * H * I, np.float32)
    w[2 * H + 5] = a
    w[H * I + 2 * H + 5] = b
    w[2 * H * I + 7 * I + 2] = c
    return synth.to_bf16_bits(w).view(np.uint8)


@pytest.mark.parametrize("wg", [0.75, -0.75])
def test_shared_gate_one_hot_closed_form(wg):
    """The shared expert's gate sigmoid(x . w_g) with a one-hot w_g (only
    w_g[9] = wg) and x nonzero at 5 and 9: z = x9 * wg exactly, and the layer
    output is the routed sum plus sigmoid(z) times the shared FFN's closed form,
    at both signs of z.  A sigma(-z), a z taken over the wrong vector or element,
    or the gate applied to the routed part fails here."""
    H, I, E = 32, 32, 4
    x = np.zeros(H, np.float32)
    x[5], x[9] = 1.25, 2.0
    xb = synth.to_bf16_bits(x)
    sblob = _one_weight_bf16_blob(H, I, 0.75, -1.5, 2.0)      # shared: y[7] only
    rblob = _one_weight_bf16_blob(H, I, 0.5, 1.0, -1.0)       # routed expert 1: y[7] only
    gate = np.zeros(H, np.float32)
    gate[9] = wg
    gw = synth.to_bf16_bits(gate)
    z = 2.0 * wg
    sig = 1.0 / (1.0 + math.exp(-z))
    g_s = 0.75 * 1.25
    ffn_s = 2.0 * (g_s / (1 + math.exp(-g_s))) * (-1.5 * 1.25)
    g_r = 0.5 * 1.25
    ffn_r = -1.0 * (g_r / (1 + math.exp(-g_r))) * (1.0 * 1.25)
    blobs = [None, rblob, None, None]
    ids = np.array([[1, 1]], np.int32)             # expert 1 twice: weights 0.25 + 0.5
    wts = np.array([[0.25, 0.5]], np.float32)
    out = oracle.layer(oracle.FMT_BF16, blobs, E, H, I, xb[None, :], ids, wts,
                       shared_blob=sblob, shared_inter=I, shared_gate_w=gw)
    assert out[0, 7] == pytest.approx(0.75 * ffn_r + sig * ffn_s, rel=1e-14)
    assert np.count_nonzero(out[0]) == 1
    # the shared term alone (zero routing weights): exactly the gated closed form
    s_only = oracle.layer(oracle.FMT_BF16, blobs, E, H, I, xb[None, :], ids, np.zeros_like(wts),
                          shared_blob=sblob, shared_inter=I, shared_gate_w=gw)
    assert s_only[0, 7] == pytest.approx(sig * ffn_s, rel=1e-14)
    assert (s_only[0, 7] / ffn_s > 0.5) == (wg > 0)


@pytest.mark.parametrize("age,protected", [(1, True), (254, True), (255, False), (300, False)])
def test_guard_recency_byte_boundary(age, protected):
    """Score (4 << 8) | rec against a never-seen prediction: protected iff
    4 * (1024 + rec) > 4096, i.e. rec >= 1, i.e. the last demand is fewer
    than 255 admissions old (the recency byte saturates at 0 from age 255)."""
    oc = oracle.OracleCache(1, 32, 3)
    for _ in range(4):
        oc.admit(0, [5])
    oc.admit(0, [6, 7])
    for i in range(age - 1):   # hits only; expert 5's slot stays the LRU head
        oc.admit(0, [6 + i % 2])
    assert oc.lru_order()[0] == oc.state()["map"][5]
    assert oc.state()["clock"][0] - oc.state()["last_demand"][5] == age
    plan = oc.prefetch(0, [20])
    assert (plan == []) == protected


# ----------------------------------------------------------------------------
# The look-ahead producer (llama.cpp fork PR #126 "cuda : MoE look-ahead
# expert prefetch (PR-A consumer) + LFRU eviction guard", sections What and
# "Open for PR-P1 (producer)").  The pages leave the predictor open; the
# reading: layer L+1's router applied to layer L's hidden state, each row's k
# largest logits, ties to the lower id.

def _bf16_bits(vals) -> np.ndarray:
    """bf16 bits of values that bf16 holds exactly."""
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _one_hot_router() -> np.ndarray:
    """Row e holds e + 1 in column e mod 4 and zeros elsewhere, so that
    z[b][e] = (e + 1) * x_b[e mod 4] exactly."""
    r = np.zeros((8, 4), np.float32)
    for e in range(8):
        r[e, e % 4] = e + 1
    return r


def test_lookahead_predict_closed_form():
    """x_0 = (1, 2, 3, 4): z = 1, 4, 9, 16, 5, 12, 21, 32, so the top 3 are
    experts 7, 6, 3.  x_1 = (4, 3, 2, 1): z = 4, 6, 6, 4, 20, 18, 14, 8, so
    the top 3 are 4, 5, 6.  A transposed product, the first row's x used for
    every row, or an ascending order each fails."""
    x = np.array([[1, 2, 3, 4], [4, 3, 2, 1]], np.float32)
    pred, z = oracle.lookahead_predict(_bf16_bits(x), _bf16_bits(_one_hot_router()), 3)
    assert pred.tolist() == [[7, 6, 3], [4, 5, 6]]
    assert z.tolist() == [[1, 4, 9, 16, 5, 12, 21, 32], [4, 6, 6, 4, 20, 18, 14, 8]]


def test_lookahead_predict_ties_negative_and_nan():
    """The full order of x_1's logits has two ties (6 at experts 1 and 2, 4 at
    0 and 3), each going to the lower id; negated x reverses the order of the
    distinct values; a NaN router weight makes that expert's logit NaN, which
    ranks after every number."""
    router = _one_hot_router()
    x1 = np.array([[4, 3, 2, 1]], np.float32)
    pred, _ = oracle.lookahead_predict(_bf16_bits(x1), _bf16_bits(router), 8)
    assert pred[0].tolist() == [4, 5, 6, 7, 1, 2, 0, 3]
    pred, _ = oracle.lookahead_predict(_bf16_bits(-x1), _bf16_bits(router), 8)
    assert pred[0].tolist() == [0, 3, 1, 2, 7, 6, 5, 4]  # -4,-4,-6,-6,-8,-14,-18,-20
    router[7, 3] = np.nan
    x0 = np.array([[1, 2, 3, 4]], np.float32)
    pred, z = oracle.lookahead_predict(_bf16_bits(x0), _bf16_bits(router), 8)
    assert math.isnan(z[0, 7])
    assert pred[0].tolist() == [6, 3, 5, 2, 4, 1, 0, 7]
    with pytest.raises(ValueError):
        oracle.lookahead_predict(_bf16_bits(x0), _bf16_bits(router), 9)  # k > n_experts
