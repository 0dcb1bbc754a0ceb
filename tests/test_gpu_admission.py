"""GPU admission, prefetch, gather and rollback against the oracle, bit-exact.

Every call goes through the C ABI; after each step the whole device state
(expert->slot map, slot keys, stamps, clocks, frequencies), the miss plan, the
rewritten slot ids and the per-layer statistics must equal the oracle's.
"""
import random

import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import Rig, assert_state_equal, gpu_plan

pytestmark = pytest.mark.gpu


def _admit(rig, layer, ids, cap=-1, inplace=False):
    m = rig.m
    ids = np.asarray(ids, np.int32).ravel()
    d_ids = torch.from_numpy(ids.copy()).cuda()
    d_out = d_ids if inplace else torch.full_like(d_ids, -7)
    m.moe_admit(rig.sc.handle, layer, d_ids, d_out, len(ids), cap)
    ref = rig.oc.admit(layer, ids, cap)
    got = d_out.cpu().numpy()
    assert np.array_equal(got, ref["slots"]), f"slots gpu {got.tolist()} oracle {ref['slots'].tolist()}"
    assert gpu_plan(rig.sc, 0) == ref["plan"]
    return ref


def _prefetch(rig, layer, pred):
    m = rig.m
    pred = np.asarray(pred, np.int32).ravel()
    d = torch.from_numpy(pred.copy()).cuda()
    m.moe_prefetch(rig.sc.handle, layer, d, len(pred))
    ref = rig.oc.prefetch(layer, pred)
    assert gpu_plan(rig.sc, 1) == ref
    return ref


@pytest.mark.parametrize("seed", range(8))
def test_random_tiny_pools(seed):
    """Random op sequences on tiny pools: admissions with caps, invalid and
    duplicate ids, pins, prefetches and rollbacks."""
    rnd = random.Random(100 + seed)
    L = rnd.choice([1, 2, 3])
    E = rnd.randint(3, 40)
    S = rnd.randint(1, 12)
    per_layer = rnd.random() < 0.4
    w = synth.Workload("t", L, E, 2, 0, 0, 0, S, per_layer, 1, 1, 1)
    rig = Rig(w, storage=False, max_routes=64, max_pred=8)
    m = rig.m
    for step in range(120):
        op = rnd.random()
        layer = rnd.randrange(L)
        if op < 0.06:
            slot, pin = rnd.randrange(S), rnd.random() < 0.5
            m.moe_cache_pin(rig.sc.handle, layer, slot, int(pin))
            rig.oc.pin(layer, slot, pin)
        elif op < 0.22:
            _prefetch(rig, layer, [rnd.randint(-2, E + 1) for _ in range(rnd.randint(0, 8))])
        else:
            R = rnd.randint(0, 64)
            ids = [rnd.randint(-3, E + 2) if rnd.random() < 0.08 else rnd.randrange(E)
                   for _ in range(R)]
            ref = _admit(rig, layer, ids, rnd.choice([-1, -1, 0, 1, 2, 5]),
                         inplace=rnd.random() < 0.5)
            if ref["plan"] and rnd.random() < 0.1:
                m.moe_rollback_plan(rig.sc.handle, m.MOE_PLAN_DEMAND)
                rig.oc.rollback(ref["plan"])
        assert_state_equal(rig.sc, rig.oc, what=f"seed {seed} step {step}")


def test_edge_cases():
    w = synth.Workload("e", 2, 5, 2, 0, 0, 0, 3, False, 1, 1, 1)
    rig = Rig(w, storage=False, max_routes=32, max_pred=4)
    _admit(rig, 0, [])                       # empty step still counts a call
    _admit(rig, 0, [-1, 5, 7, -100])          # all invalid
    _admit(rig, 1, [4, 4, 4, 4])              # duplicates of one expert
    _admit(rig, 0, [0, 1, 2, 3, 4], cap=0)    # cap 0: everything overflows
    _admit(rig, 0, [0, 1, 2, 3, 4])           # more misses than slots: capacity shortfall
    for s in range(3):
        rig.m.moe_cache_pin(rig.sc.handle, 0, s, 1)
        rig.oc.pin(0, s, True)
    _admit(rig, 1, [0, 1, 2])                 # every slot pinned: nothing admitted
    _prefetch(rig, 1, [3, 3, -1])             # no victim
    assert_state_equal(rig.sc, rig.oc)
    st = rig.sc.stats(0)
    assert st["status_bits"] == 3 and st["invalid_routes"] == 4


def test_max_experts_and_slots():
    """Wide pools: 16,384 experts, 20,000 slots, 16,384-route steps."""
    w = synth.Workload("big", 1, 16384, 8, 0, 0, 0, 20000, False, 1, 1, 1)
    rig = Rig(w, storage=False, max_routes=16384, max_pred=4096)
    rnd = np.random.default_rng(5)
    for step in range(6):
        ids = rnd.integers(0, 16384, 16384 if step % 2 else 1000).astype(np.int32)
        _admit(rig, 0, ids, cap=-1 if step != 4 else 3000)
        _prefetch(rig, 0, rnd.integers(-5, 16390, 4096).astype(np.int32))
        assert_state_equal(rig.sc, rig.oc, what=f"step {step}")


def test_a_smaller_cache_leaves_a_larger_caches_limits():
    """Shared-memory limits belong to the kernels, not to a cache: a 512-expert,
    4,000-slot pool keeps its admission state in 54 KB of shared memory, and
    creating a 16-expert, 8-slot cache afterwards must not lower the limit the
    larger cache's admissions need.  Both keep admitting with the state exact."""
    big = synth.Workload("big", 1, 512, 8, 0, 0, 0, 4000, False, 1, 1, 7)
    small = synth.Workload("small", 1, 16, 2, 0, 0, 0, 8, False, 1, 1, 8)
    rnd = np.random.default_rng(11)
    rb = Rig(big, storage=False, max_routes=512)
    _admit(rb, 0, rnd.integers(0, 512, 400).astype(np.int32))
    rs = Rig(small, storage=False, max_routes=8)
    for step in range(3):
        _admit(rs, 0, rnd.integers(0, 16, 6).astype(np.int32))
        _admit(rb, 0, rnd.integers(0, 512, 400).astype(np.int32))
    assert_state_equal(rb.sc, rb.oc, what="the larger cache")
    assert_state_equal(rs.sc, rs.oc, what="the smaller cache")


def test_qwen3moe_admission_sequence():
    """The 40-layer, 3,164-slot routing of the decode benchmark, admission
    only: state exact after every token (radix select over old stamps)."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], steps=160)
    rig = Rig(w, storage=False)
    ids, _ = synth.make_routing(w)
    for t in range(w.steps):
        for layer in range(w.n_layers):
            _admit(rig, layer, ids[t, layer].ravel())
        if t % 8 == 0 or t == w.steps - 1:
            assert_state_equal(rig.sc, rig.oc, what=f"token {t}")


def test_wide_decode_admission():
    """600 rows x top-2 over 1,024 experts, 1,100 slots, 307 pre-resident."""
    w = synth.workloads()["wide_decode"]
    rig = Rig(w, storage=False)
    rig.prefill(0, synth.prefill_ids(w))
    ids, _ = synth.make_routing(w, steps=2)
    for t in range(2):
        ref = _admit(rig, 0, ids[t, 0].ravel())
        assert len(ref["plan"]) > 0
    assert_state_equal(rig.sc, rig.oc)


def test_hybrid_prefetch_sequence():
    """Capped fetch (4) and look-ahead prefetch (8 predictions) over 48 layers
    with one 1,024-slot pool: state and all prefetch counters exact."""
    w = synth.scaled(synth.workloads()["hybrid_prefetch"], steps=24)
    rig = Rig(w, storage=False)
    ids, _ = synth.make_routing(w)
    for t in range(w.steps):
        for layer in range(w.n_layers):
            _admit(rig, layer, ids[t, layer].ravel(), cap=w.fetch_cap)
            if layer + 1 < w.n_layers:
                _prefetch(rig, layer + 1, synth.make_predictions(w, ids[t, layer + 1], t, layer))
        assert_state_equal(rig.sc, rig.oc, what=f"token {t}")
    st = [rig.sc.stats(l) for l in range(w.n_layers)]
    assert sum(s["pf_filled"] for s in st) > 0 and sum(s["overflow_routes"] for s in st) > 0
    assert sum(s["pf_dropped_guard"] for s in st) > 0


@pytest.mark.parametrize("batch", [1, 4, 8, 12, 13, 16, 24, 32, 48, 128])
def test_wide_admission_sweep_graph(batch):
    """48 per-layer 2,100-slot pools holding all 512 experts; 48 admissions
    captured in one CUDA graph and replayed; slot ids and stats exact."""
    w = synth.workloads()["wide_admission"]
    rig = Rig(w, storage=False, max_routes=batch * w.top_k)
    for layer in range(w.n_layers):
        rig.prefill(layer, synth.prefill_ids(w))
    ids = synth.uniform_ids(w, batch, salt=batch)
    d_ids = torch.from_numpy(ids).cuda()
    d_out = torch.empty_like(d_ids)
    m = rig.m
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for layer in range(w.n_layers):  # warm-up (eager)
            m.moe_admit(rig.sc.handle, layer, d_ids[layer], d_out[layer], ids.shape[1], -1, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for layer in range(w.n_layers):
            m.moe_admit(rig.sc.handle, layer, d_ids[layer], d_out[layer], ids.shape[1], -1, s)
    replays = 5
    for _ in range(replays):
        g.replay()
    torch.cuda.synchronize()
    for _ in range(1 + replays):
        for layer in range(w.n_layers):
            ref = rig.oc.admit(layer, ids[layer])
    assert np.array_equal(d_out.cpu().numpy()[-1], ref["slots"])
    assert_state_equal(rig.sc, rig.oc)


def test_gather_copies_plan_bytes():
    """After admission + gather every resident slot holds its expert's blob,
    byte for byte; prefetch fills too; a rolled-back plan leaves no booking."""
    w = synth.scaled(synth.workloads()["tiny"], n_layers=3, n_slots=6, n_pred=4)
    rig = Rig(w, max_pred=4, max_routes=8)
    m = rig.m
    rnd = random.Random(3)
    for step in range(40):
        layer = rnd.randrange(3)
        _admit(rig, layer, [rnd.randrange(16) for _ in range(4)])
        m.moe_gather_missing(rig.sc.handle, m.MOE_PLAN_DEMAND)
        if layer + 1 < 3:
            _prefetch(rig, layer + 1, [rnd.randrange(16) for _ in range(4)])
            m.moe_gather_missing(rig.sc.handle, m.MOE_PLAN_PREFETCH)
        torch.cuda.synchronize()
        st = rig.oc.state()
        for s, key in enumerate(st["slot_key"]):
            if key >= 0:
                assert np.array_equal(rig.slot_bytes(0, s), rig.blobs.blob(int(key))), (step, s)
    # injected gather failure: nothing enqueued, bookings rolled back
    ref = _admit(rig, 0, [13, 14, 15])
    m.moe_cache_fail_next_gather(rig.sc.handle, 1)
    with pytest.raises(m.MoeError):
        m.moe_gather_missing(rig.sc.handle, m.MOE_PLAN_DEMAND)
    m.moe_rollback_plan(rig.sc.handle, m.MOE_PLAN_DEMAND)
    rig.oc.rollback(ref["plan"])
    assert_state_equal(rig.sc, rig.oc)
    assert gpu_plan(rig.sc, 0) == []
