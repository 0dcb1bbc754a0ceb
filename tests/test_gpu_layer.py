"""Whole offloaded decode layers on the GPU against the fp64 oracle.

Outputs must agree elementwise within |gpu - ref| <= atol + rtol*|ref|
(NVFP4: atol 2e-2, rtol 1e-2; bf16: atol 5e-3, rtol 1e-2); slot ids, plans,
statistics and the whole cache state must be bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import Rig, assert_close, assert_state_equal

pytestmark = pytest.mark.gpu


def _dev(a, dtype=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


class Stepper:
    """Feeds one workload's steps through moe_decode_layer, mirroring every
    admission/prefetch on the oracle."""

    def __init__(self, rig: Rig, overlap: bool = True, n_pred: int = 0, fused: bool = False,
                 hybrid: bool = False):
        self.rig = rig
        self.hybrid = hybrid
        self.overlap = overlap
        self.fused = fused
        self.n_pred = n_pred
        self.side = torch.cuda.Stream()
        w = rig.w
        self.out = torch.empty(w.n_layers, w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
        self.slots = torch.empty(w.n_layers, w.batch * w.top_k, dtype=torch.int32, device="cuda")

    def step(self, t: int, ids: np.ndarray, wts: np.ndarray, x: np.ndarray, check_state=True,
             layers=None):
        rig, w, m = self.rig, self.rig.w, self.rig.m
        cs = torch.cuda.current_stream()
        d_x = _dev(x)
        d_ids = _dev(ids.reshape(w.n_layers, -1))
        d_w = _dev(wts.reshape(w.n_layers, -1))
        flags = ((m.MOE_OVERLAP if self.overlap else 0) | (m.MOE_FUSED if self.fused else 0) |
                 (m.MOE_HYBRID if self.hybrid else 0))
        refs = []
        for layer in range(w.n_layers):
            pred = None
            if self.n_pred and layer + 1 < w.n_layers:
                pred = synth.make_predictions(w, ids[layer + 1], t, layer)
            m.moe_decode_layer(rig.sc.handle, layer, d_x[layer], d_ids[layer], d_w[layer],
                               self.slots[layer], w.batch, w.top_k, w.fetch_cap,
                               None if pred is None else _dev(pred), 0 if pred is None else len(pred),
                               *rig.d_shared[layer], self.out[layer], cs, self.side,
                               flags)
            refs.append(rig.oc.admit(layer, ids[layer].ravel(), w.fetch_cap))
            if pred is not None:
                rig.oc.prefetch(layer + 1, pred)
        torch.cuda.synchronize()
        got = self.slots.cpu().numpy()
        for layer in range(w.n_layers):
            assert np.array_equal(got[layer], refs[layer]["slots"]), f"step {t} layer {layer}"
        if check_state:
            assert_state_equal(rig.sc, rig.oc, what=f"step {t}")
        return refs


@pytest.mark.parametrize("overlap", [True, False])
def test_tiny_all_steps(overlap):
    w = synth.workloads()["tiny"]
    rig = Rig(w)
    st = Stepper(rig, overlap)
    ids, wts = synth.make_routing(w)
    worst = 0.0
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        st.step(t, ids[t], wts[t], x)
        ref = rig.oracle_layer(0, x[0], ids[t, 0], wts[t, 0])
        worst = max(worst, assert_close(st.out[0], ref, w.fmt, f"step {t}")["max_abs"])
    s = rig.sc.stats(0)
    assert s["misses"] > 0 and s["evictions"] > 0 and s["hits"] > 0


def test_tiny_with_shared_expert_and_batch():
    w = synth.scaled(synth.workloads()["tiny"], shared_inter=96, batch=5, steps=12, n_slots=9)
    rig = Rig(w)
    st = Stepper(rig)
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        st.step(t, ids[t], wts[t], x)
        assert_close(st.out[0], rig.oracle_layer(0, x[0], ids[t, 0], wts[t, 0]), w.fmt, f"step {t}")


def test_overlap_bytes_equal_serial():
    """[FreeToken issue #753, Correctness]: only where the gather runs differs,
    so overlapped outputs are byte-equal to serial ones."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=6, steps=12)
    blobs = synth.HostBlobs(w, pinned=True)
    a, b = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    sa, sb = Stepper(a, True), Stepper(b, False)
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        sa.step(t, ids[t], wts[t], x)
        sb.step(t, ids[t], wts[t], x)
        assert torch.equal(sa.out.view(torch.int16), sb.out.view(torch.int16)), f"step {t}"


def test_fused_layer_equals_two_launch_path():
    """MOE_FUSED runs the whole layer in one launch (admission, gather, shared
    expert, routed experts); the overlap of [FreeToken issue #753, What we
    changed] moves inside it.  Slot ids, state and statistics stay exact
    against the oracle, the output bytes equal the two-launch path's, and every
    resident slot holds its expert's bytes (the misses went through staging)."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=6, steps=12, n_slots=80)
    blobs = synth.HostBlobs(w, pinned=True)
    a, b = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    sa, sb = Stepper(a, True, fused=True), Stepper(b, True)
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        sa.step(t, ids[t], wts[t], x)
        sb.step(t, ids[t], wts[t], x)
        assert torch.equal(sa.out.view(torch.int16), sb.out.view(torch.int16)), f"step {t}"
        if t in (0, w.steps - 1):
            for layer in (0, w.n_layers - 1):
                ref = a.oracle_layer(layer, x[layer], ids[t, layer], wts[t, layer])
                assert_close(sa.out[layer], ref, w.fmt, f"step {t} layer {layer}")
    assert sum(a.sc.stats(l)["fetched"] for l in range(w.n_layers)) > 50
    assert a.sc.stats(0)["status_bits"] == 0
    state = a.oc.state()
    for s, key in enumerate(state["slot_key"]):
        if key >= 0:
            assert np.array_equal(a.slot_bytes(0, s), a.blobs.blob(int(key))), s


def test_fused_layer_uncapped_staging_and_fallback_bf16():
    """Uncapped hybrid shapes with prefetch: 25 MB blobs leave room for two
    staging entries (64 MB), so a step with at most two misses copies them
    through staging and one with more waits for the admission's slots.  Both
    give the two-launch path's output bytes, exact state, and slots holding
    their experts."""
    w = synth.scaled(synth.workloads()["hybrid_prefetch"], n_layers=6, steps=6, fetch_cap=-1)
    blobs = synth.HostBlobs(w, pinned=True)
    a, b = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    sa, sb = Stepper(a, True, n_pred=w.n_pred, fused=True), Stepper(b, True, n_pred=w.n_pred)
    ids, wts = synth.make_routing(w)
    misses = []
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        before = [a.sc.stats(l)["misses"] for l in range(w.n_layers)]
        sa.step(t, ids[t], wts[t], x)
        sb.step(t, ids[t], wts[t], x)
        misses += [a.sc.stats(l)["misses"] - before[l] for l in range(w.n_layers)]
        assert torch.equal(sa.out.view(torch.int16), sb.out.view(torch.int16)), f"step {t}"
    assert any(0 < m <= 2 for m in misses) and any(m > 2 for m in misses), misses
    state = a.oc.state()
    for s, key in enumerate(state["slot_key"]):
        if key >= 0:
            assert np.array_equal(a.slot_bytes(0, s), a.blobs.blob(int(key))), s


def test_fused_layer_capped_prefetch_bf16():
    """The hybrid shapes (bf16, H 4096, I 1024, fetch cap 4, look-ahead
    prefetch of 8 ids under the LFRU guard) through MOE_FUSED: the prefetch
    plan is copied inside the launch; state and prefetch counters exact, output
    bytes equal to the two-launch path's."""
    w = synth.scaled(synth.workloads()["hybrid_prefetch"], n_layers=6, steps=5)
    blobs = synth.HostBlobs(w, pinned=True)
    a, b = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    sa, sb = Stepper(a, True, n_pred=w.n_pred, fused=True), Stepper(b, True, n_pred=w.n_pred)
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        sa.step(t, ids[t], wts[t], x)
        sb.step(t, ids[t], wts[t], x)
        assert torch.equal(sa.out.view(torch.int16), sb.out.view(torch.int16)), f"step {t}"
    st = [a.sc.stats(l) for l in range(w.n_layers)]
    assert sum(s["pf_filled"] for s in st) > 0 and sum(s["overflow_routes"] for s in st) > 0
    # the prefetched experts' bytes arrived: every resident slot holds its expert
    state = a.oc.state()
    for s, key in enumerate(state["slot_key"]):
        if key >= 0:
            assert np.array_equal(a.slot_bytes(0, s), a.blobs.blob(int(key))), s


def test_slot_placement_does_not_change_bits():
    """[FreeToken PR #680, Tests]: the GEMV over the slots equals the GEMV over
    the streamed layer exactly.  Here: the same experts placed in different
    slots (a cold cache vs. one pre-filled in another order) give identical
    output bytes."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=2, steps=4, n_slots=64)
    blobs = synth.HostBlobs(w, pinned=True)
    a, b = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    b.prefill(0, np.arange(255, 215, -1, dtype=np.int32))
    sa, sb = Stepper(a), Stepper(b)
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        sa.step(t, ids[t], wts[t], x)
        sb.step(t, ids[t], wts[t], x)
        assert torch.equal(sa.out.view(torch.int16), sb.out.view(torch.int16))
    assert not np.array_equal(sa.slots.cpu().numpy(), sb.slots.cpu().numpy())


@pytest.mark.slow
@pytest.mark.parametrize("fused", [False, True])
def test_qwen3moe_full_size(fused):
    """The decode benchmark's workload at full size (40 layers x 256 NVFP4
    experts, 3,164 slots, shared expert), eagerly, on the four-launch
    overlapped path and on the one-launch layer (MOE_FUSED) the benchmark
    captures: state exact every token, the outputs of every 16th token and of
    the last on every layer vs fp64."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], steps=20)
    rig = Rig(w)
    st = Stepper(rig, fused=fused)
    if fused:
        plan = rig.m.moe_decode_layer_plan(rig.sc.handle, w.batch, w.top_k, shared=True,
                                           flags=rig.m.MOE_FUSED | rig.m.MOE_OVERLAP)
        assert plan == ["c:layer_admit"], plan
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        st.step(t, ids[t], wts[t], x)
        if t % 16 == 0 or t == w.steps - 1:
            for layer in range(w.n_layers):
                ref = rig.oracle_layer(layer, x[layer], ids[t, layer], wts[t, layer])
                assert_close(st.out[layer], ref, w.fmt, f"token {t} layer {layer}")
    misses = sum(rig.sc.stats(l)["misses"] for l in range(w.n_layers))
    assert misses > 300


@pytest.mark.slow
def test_qwen3moe_benchmark_graph_full_size():
    """The path bench.py times, as it times it: bench.Decode (40 layers x 256
    NVFP4 experts, 3,164 slots, shared expert, MOE_FUSED: one launch per
    layer with the admission inside) captured as one CUDA graph per token and
    replayed for 14 tokens with each token's inputs written into the graph's
    fixed buffers [FreeToken issue #753, What we changed: fixed addresses,
    device-side miss counts, no host sync].  After every token the slot ids,
    the whole cache state and every layer's statistics equal the oracle's;
    at two tokens all 40 layers' outputs are within the NVFP4 tolerance of
    fp64; at the end every resident slot holds its expert's bytes."""
    import oracle

    import bench
    from tests.gpu_util import assert_close, assert_state_equal
    dec = bench.Decode(0, warm_tokens=2, total_tokens=16)
    w, m = dec.w, dec.m
    plan = m.moe_decode_layer_plan(dec.cache.handle, w.batch, w.top_k, shared=True,
                                   flags=m.MOE_FUSED | m.MOE_OVERLAP)
    assert plan == ["c:layer_admit"], plan  # the one-launch layer at the full size
    ids = dec.d_ids.cpu().numpy()           # [T, L, R], as the graph's inputs
    wts = dec.d_w.cpu().numpy()
    oc = oracle.OracleCache(w.n_layers, w.n_experts, w.n_slots)
    for t in range(2):                      # the eager warm-up tokens
        for layer in range(w.n_layers):
            oc.admit(layer, ids[t, layer])
    assert_state_equal(dec.cache, oc, what="after the eager tokens")
    shared = [synth.make_shared(w, l) for l in range(w.n_layers)]
    misses = 0
    for t in range(2, dec.T):
        before = sum(dec.cache.stats(l)["misses"] for l in range(w.n_layers))
        assert dec.t == t
        dec.step()
        torch.cuda.synchronize()
        got = dec.b_slots.cpu().numpy()
        for layer in range(w.n_layers):
            ref = oc.admit(layer, ids[t, layer])
            assert np.array_equal(got[layer], ref["slots"]), f"token {t} layer {layer}"
        assert_state_equal(dec.cache, oc, what=f"token {t}")
        misses += sum(dec.cache.stats(l)["misses"] for l in range(w.n_layers)) - before
        if t in (2, dec.T - 1):
            x = dec.d_x[t].cpu().numpy().view(np.uint16)
            for layer in range(w.n_layers):
                ref = oracle.layer(w.fmt, [dec.blobs.addr(layer * w.n_experts + e)
                                           for e in range(w.n_experts)],
                                   w.n_experts, w.hidden, w.inter, x[layer],
                                   ids[t, layer].reshape(w.batch, w.top_k),
                                   wts[t, layer].reshape(w.batch, w.top_k),
                                   shared_blob=shared[layer][0], shared_inter=w.shared_inter,
                                   shared_gate_w=shared[layer][1])
                assert_close(dec.b_out[layer], ref, w.fmt, f"token {t} layer {layer}")
    assert misses > 100  # the replayed tokens really gather (about 28 per token at steady state)
    for l in range(w.n_layers):
        assert dec.cache.stats(l)["status_bits"] == 0
    # every resident slot holds its expert's bytes, compared on the device in chunks
    state = oc.state()
    keys = state["slot_key"]
    res = np.nonzero(keys >= 0)[0]
    host = dec.blobs.buf.view(-1, dec.blobs.stride)
    dev = dec.storage.view(w.n_slots, dec.blobs.stride)
    nb = dec.blobs.nbytes
    for c0 in range(0, len(res), 128):
        sl = res[c0:c0 + 128]
        rows = torch.from_numpy(dec.blobs.key_to_blob[keys[sl]])
        want = host.index_select(0, rows)[:, :nb].cuda()
        assert torch.equal(dev[torch.from_numpy(sl).cuda()][:, :nb], want), f"slots {sl[:4]}"


@pytest.mark.slow
def test_qwen3moe_graph_replay_equals_eager():
    """One token (40 layers) captured as a CUDA graph and replayed with new
    routes written into its input buffers equals the eager pipeline, byte for
    byte, with identical cache state [FreeToken issue #753, What we changed:
    fixed addresses, device-side miss counts, no host sync]."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=8, steps=10)
    blobs = synth.HostBlobs(w, pinned=True)
    eager, graphed = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    se = Stepper(eager)
    m = graphed.m
    ids, wts = synth.make_routing(w)
    L, R = w.n_layers, w.routes
    b_x = torch.empty(L, w.batch, w.hidden, dtype=torch.int16, device="cuda")
    b_ids = torch.empty(L, R, dtype=torch.int32, device="cuda")
    b_w = torch.empty(L, R, dtype=torch.float32, device="cuda")
    b_slots = torch.empty(L, R, dtype=torch.int32, device="cuda")
    b_out = torch.empty(L, w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
    cs, side = torch.cuda.Stream(), torch.cuda.Stream()

    def enqueue():
        for layer in range(L):
            m.moe_decode_layer(graphed.sc.handle, layer, b_x[layer], b_ids[layer], b_w[layer],
                               b_slots[layer], w.batch, w.top_k, -1, None, 0,
                               *graphed.d_shared[layer], b_out[layer], cs, side,
                               m.MOE_OVERLAP)

    def load(t):
        b_x.copy_(_dev(synth.make_hidden(w, t)))
        b_ids.copy_(_dev(ids[t].reshape(L, -1)))
        b_w.copy_(_dev(wts[t].reshape(L, -1)))

    load(0)
    with torch.cuda.stream(cs):
        enqueue()  # token 0 eagerly (also warms up)
    torch.cuda.synchronize()
    se.step(0, ids[0], wts[0], synth.make_hidden(w, 0))
    assert torch.equal(b_out.view(torch.int16), se.out.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        enqueue()
    for t in range(1, w.steps):
        load(t)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        se.step(t, ids[t], wts[t], synth.make_hidden(w, t))
        assert torch.equal(b_out.view(torch.int16), se.out.view(torch.int16)), f"token {t}"
        assert torch.equal(b_slots, se.slots)
    for layer in range(L):
        assert graphed.sc.stats(layer) == eager.sc.stats(layer)


def _gpu_groups(sc, max_routes: int) -> list[tuple[int, list[int]]]:
    """The route groups moe_routed_experts wrote on the grouped path:
    [G, slot[max_routes], start[max_routes + 1], route[max_routes]]."""
    from tests.gpu_util import dev_copy
    n = 1 + max_routes + (max_routes + 1) + max_routes
    a = dev_copy(sc.views().groups, n, np.int32)
    G = int(a[0])
    slot = a[1:1 + G]
    start = a[1 + max_routes:1 + max_routes + G + 1]
    route = a[2 + 2 * max_routes:]
    return [(int(slot[g]), [int(r) for r in route[start[g]:start[g + 1]]]) for g in range(G)]


def wide_layer_oracle(rig, x, ids, wts, experts_per_call: int = 64, layer: int = 0) -> np.ndarray:
    """The fp64 layer over every row, computed as a sum of partial layers over
    disjoint sets of experts (ascending id, `experts_per_call` at a time), so
    that one oracle call dequantises at most that many experts; the gated
    shared expert (when the workload has one) is added once."""
    w = rig.w
    blobs = [rig.blobs.addr(layer * w.n_experts + e) for e in range(w.n_experts)]
    used = np.unique(ids[(ids >= 0) & (ids < w.n_experts)])
    full = np.zeros((x.shape[0], w.hidden), np.float64)
    for c0 in range(0, len(used), experts_per_call):
        part = used[c0:c0 + experts_per_call]
        mask = np.isin(ids, part).astype(np.uint8)
        full += oracle.layer(w.fmt, blobs, w.n_experts, w.hidden, w.inter, x, ids, wts, mask=mask)
    if w.shared_inter:  # every route masked off: the shared expert alone
        none = np.zeros(np.shape(ids), np.uint8)
        full += rig.oracle_layer(layer, x, ids, wts, mask=none)
    return full


@pytest.mark.slow
@pytest.mark.parametrize("routing,min_misses", [("uniform", 400), ("zipf", 200)])
def test_wide_decode_step(routing, min_misses):
    """[FreeToken PR #680, Tests]: 600 rows x top-2 = 1,200 routes over 1,024
    NVFP4 experts with 1,100 slots, 30% pre-resident: admission + gather +
    grouped routed FFNs.  Every slot id exact; the route groups the GPU built
    equal the oracle's; every one of the 600 rows' outputs within the NVFP4
    tolerance of the fp64 layer.  Uniform routing gives every expert one to a
    few routes (37 groups of four or more go to the tensor cores in the
    automatic mode, the rest to the CUDA cores); Zipf routing gives some
    experts dozens (47 groups of four or more)."""
    w = synth.scaled(synth.workloads()["wide_decode"], routing=routing)
    rig = Rig(w)
    rig.prefill(0, synth.prefill_ids(w))
    st = Stepper(rig)
    ids, wts = synth.make_routing(w, steps=1)
    x = synth.make_hidden(w, 0)
    refs = st.step(0, ids[0], wts[0], x)
    assert _gpu_groups(rig.sc, rig.sc.desc.max_routes) == refs[0]["groups"]
    ref = wide_layer_oracle(rig, x[0], ids[0, 0], wts[0, 0])
    info = assert_close(st.out[0], ref, w.fmt, "wide step, all rows")
    assert info["max_abs"] > 0
    s = rig.sc.stats(0)
    assert s["fetched"] == s["misses"] > min_misses and s["evictions"] == 0
    if routing == "zipf":
        assert max(len(r) for _, r in refs[0]["groups"]) >= 4  # tensor-core groups


@pytest.mark.parametrize("routing,batch", [("zipf", 200), ("uniform", 40)])
def test_wide_step_tensor_cores_and_cuda_cores(routing, batch):
    """A wide step small enough to check whole on every grouped path: 64 NVFP4
    experts (H 256, I 128), top-4.  Zipf routing over 200 rows gives hot
    experts more than 32 routes (several route chunks per tile, MMA N of 16 and
    32) and cold ones a single route, so the automatic mode splits the groups
    between the two kernel families; uniform routing over 40 rows gives groups
    of one to a few routes.  The tensor-core mode (tcgen05 for every group),
    the CUDA-core mode and the automatic mode each match the fp64 layer on
    every row; slot ids, route groups and state are identical."""
    import expert_slot_cache_lru_gb300 as m
    w = synth.scaled(synth.workloads()["wide_decode"], n_experts=64, top_k=4, hidden=256,
                     inter=128, n_slots=64, batch=batch, routing=routing, prefill_frac=0.0)
    blobs = synth.HostBlobs(w, pinned=True)
    modes = [m.MOE_WIDE_TENSOR_CORES, m.MOE_WIDE_CUDA_CORES, m.MOE_WIDE_AUTO]
    rigs = [Rig(w, blobs=blobs) for _ in modes]
    ids, wts = synth.make_routing(w, steps=2)
    for rig, mode in zip(rigs, modes):
        m.moe_cache_set_wide_path(rig.sc.handle, mode)
        st = Stepper(rig)
        for t in range(2):
            x = synth.make_hidden(w, t)
            refs = st.step(t, ids[t], wts[t], x)
            assert _gpu_groups(rig.sc, rig.sc.desc.max_routes) == refs[0]["groups"]
            ref = rig.oracle_layer(0, x[0], ids[t, 0], wts[t, 0])
            assert_close(st.out[0], ref, w.fmt, f"step {t}, mode {mode}")
        if routing == "zipf":
            sizes = [len(r) for _, r in refs[0]["groups"]]
            assert max(sizes) > 32 and min(sizes) < 4, sizes
    assert_state_equal(rigs[0].sc, rigs[1].oc)
    with pytest.raises(m.MoeError):
        m.moe_cache_set_wide_path(rigs[0].sc.handle, 3)


@pytest.mark.parametrize("hidden,inter", [(1024, 64), (2048, 96), (3072, 64), (4096, 32),
                                          (1024, 1024), (2048, 768), (3072, 512), (4096, 256)])
def test_wide_step_warp_row_kernels_every_width(hidden, inter):
    """The gate/up and down kernels that keep x and h in registers: gate/up for
    H a multiple of 1,024 up to 4,096 (two routes per pass up to 2,048, one
    above), down for I of 256, 512, 768 and 1,024 (lanes holding one or two
    block scales).  32 NVFP4 experts, top-4 over 24 rows, uniform routing, so
    groups of one to several routes take full and partial passes.  The first
    four shapes leave the down projection to the other CUDA-core kernels (I of
    96 and 32 to the unstaged one).  Every row against the fp64 layer, in the
    CUDA-core and the automatic mode."""
    import expert_slot_cache_lru_gb300 as m
    w = synth.scaled(synth.workloads()["wide_decode"], n_experts=32, top_k=4, hidden=hidden,
                     inter=inter, n_slots=32, batch=24, routing="uniform", prefill_frac=0.0)
    blobs = synth.HostBlobs(w, pinned=True)
    for mode in (m.MOE_WIDE_CUDA_CORES, m.MOE_WIDE_AUTO):
        rig = Rig(w, blobs=blobs)
        m.moe_cache_set_wide_path(rig.sc.handle, mode)
        st = Stepper(rig)
        ids, wts = synth.make_routing(w, steps=2)
        for t in range(2):
            x = synth.make_hidden(w, t)
            refs = st.step(t, ids[t], wts[t], x)
            sizes = [len(r) for _, r in refs[0]["groups"]]
            assert max(sizes) >= 3 and min(sizes) == 1, sizes
            ref = rig.oracle_layer(0, x[0], ids[t, 0], wts[t, 0])
            assert_close(st.out[0], ref, w.fmt, f"H {hidden}, step {t}, mode {mode}")


@pytest.mark.slow
@pytest.mark.parametrize("tokens", [16, 64])
def test_prefill_chunk_through_the_layer(tokens):
    """A prefill chunk at the decode workload's layer shape (256 NVFP4 experts,
    H 2048, I 512, top-8, gated shared expert) goes through moe_decode_layer
    as one wide step [FreeToken PR #680, Problem: DeepSeek-V4's on-demand
    prefill chunks, taken while T * top_k < num_experts, and Tests: a chunk
    admitted whole]: 16 tokens (128 routes, fewer than the experts) and 64
    tokens (512 routes) over two layers from a cold cache.  One admission per
    layer whatever the width; slot ids and state exact; every token's output
    within the NVFP4 tolerance of the fp64 layer."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=2, steps=1, batch=tokens,
                     n_slots=600)
    rig = Rig(w)
    st = Stepper(rig)
    ids, wts = synth.make_routing(w)
    x = synth.make_hidden(w, 0)
    st.step(0, ids[0], wts[0], x)
    for layer in range(w.n_layers):
        ref = wide_layer_oracle(rig, x[layer], ids[0, layer], wts[0, layer], layer=layer)
        assert_close(st.out[layer], ref, w.fmt, f"{tokens} tokens, layer {layer}")
        s = rig.sc.stats(layer)
        assert s["calls"] == 1 and s["misses"] == s["lookups"] > 0


@pytest.mark.parametrize("mode", ["auto", "cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("hidden,inter", [(256, 128), (1024, 256)])
def test_wide_step_with_a_fetch_cap_skips_the_overflow_routes(mode, hidden, inter):
    """A wide step under a fetch cap [FreeToken PR #491, sections 4 and 5: the
    misses beyond the cap come back as -1 and contribute nothing on the GPU]:
    200 Zipf rows x top-4 over 64 NVFP4 experts from a cold cache, cap 5, so
    many routes are -1 and the grouped kernels of every family must skip them
    (H 256: the thread-per-row CUDA-core kernels; H 1,024, I 256: the warp-row
    ones).  Slot ids and state exact; every row equals the fp64 layer over the
    routes that got a slot."""
    import expert_slot_cache_lru_gb300 as m
    w = synth.scaled(synth.workloads()["wide_decode"], n_experts=64, top_k=4, hidden=hidden,
                     inter=inter, n_slots=64, batch=200, routing="zipf", prefill_frac=0.0,
                     fetch_cap=5)
    rig = Rig(w)
    m.moe_cache_set_wide_path(rig.sc.handle, {"auto": m.MOE_WIDE_AUTO,
                                              "cuda_cores": m.MOE_WIDE_CUDA_CORES,
                                              "tensor_cores": m.MOE_WIDE_TENSOR_CORES}[mode])
    st = Stepper(rig)
    ids, wts = synth.make_routing(w, steps=2)
    for t in range(2):
        x = synth.make_hidden(w, t)
        refs = st.step(t, ids[t], wts[t], x)
        slots = refs[0]["slots"].reshape(w.batch, w.top_k)
        assert (slots < 0).any() and (slots >= 0).any()
        ref = rig.oracle_layer(0, x[0], ids[t, 0], wts[t, 0], mask=(slots >= 0).astype(np.uint8))
        assert_close(st.out[0], ref, w.fmt, f"step {t}")


@pytest.mark.parametrize("fmt", [synth.FMT_MXFP4, synth.FMT_Q4_0])
def test_4bit_formats_wide_step_equals_oracle(fmt):
    """Wide steps of MXFP4 and Q4_0 experts (formats listed in FreeToken PR
    #491, section 7, "What did not change"): 40 rows x top-4 over 64 experts
    (H 256, I 128) with a gated shared expert of the same format (I 128).
    The routed experts take the grouped kernels on the CUDA cores, the shared
    expert the per-row kernels (more rows than the streaming kernels take).
    Two steps with misses: route groups and state exact, every row within the
    fp4 tolerance of the fp64 layer."""
    w = synth.scaled(synth.workloads()["wide_decode"], fmt=fmt, n_experts=64, top_k=4,
                     hidden=256, inter=128, n_slots=64, batch=40, routing="uniform",
                     prefill_frac=0.0, shared_inter=128)
    rig = Rig(w)
    st = Stepper(rig)
    ids, wts = synth.make_routing(w, steps=2)
    for t in range(2):
        x = synth.make_hidden(w, t)
        refs = st.step(t, ids[t], wts[t], x)
        assert _gpu_groups(rig.sc, rig.sc.desc.max_routes) == refs[0]["groups"]
        ref = rig.oracle_layer(0, x[0], ids[t, 0], wts[t, 0])
        assert_close(st.out[0], ref, w.fmt, f"step {t}")
    s = rig.sc.stats(0)
    assert s["misses"] > 0 and s["status_bits"] == 0


@pytest.mark.slow
def test_hybrid_capped_prefetch_partial_plus_cpu():
    """Capped fetch (4 per layer) + look-ahead prefetch over 48 bf16 layers:
    the GPU computes the routes that got a slot, the oracle computes the -1
    routes (the CPU side of [FreeToken PR #491, sections 4-5]); GPU partial +
    CPU partial equals the full layer within the bf16 tolerance."""
    w = synth.scaled(synth.workloads()["hybrid_prefetch"], steps=6)
    rig = Rig(w)
    st = Stepper(rig, n_pred=w.n_pred)
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        refs = st.step(t, ids[t], wts[t], x)
        if t in (0, w.steps - 1):
            for layer in (0, 1, 23, 47):
                slots = refs[layer]["slots"].reshape(w.batch, w.top_k)
                cpu_mask = (slots < 0).astype(np.uint8)
                full = rig.oracle_layer(layer, x[layer], ids[t, layer], wts[t, layer])
                cpu = rig.oracle_layer(layer, x[layer], ids[t, layer], wts[t, layer], mask=cpu_mask)
                got = st.out[layer].float().cpu().numpy().astype(np.float64) + cpu
                atol, rtol = 5e-3, 1e-2
                assert np.all(np.abs(got - full) <= atol + rtol * np.abs(full)), (t, layer)
    tot = [rig.sc.stats(l) for l in range(w.n_layers)]
    assert sum(s["overflow_routes"] for s in tot) > 0 and sum(s["pf_filled"] for s in tot) > 0


@pytest.mark.parametrize("fused", [False, True])
def test_hybrid_executor_adds_the_cpu_partial(fused):
    """MOE_HYBRID [FreeToken PR #491, sections 4-5]: the routes the capped
    admission leaves at -1 run on the host's cores and are added to the GPU's
    output; the whole layer must match the fp64 oracle's full layer (all
    routes) within the bf16 tolerance, every step posts one job (also steps
    with no -1 route), and the executor counts exactly the -1 routes."""
    w = synth.scaled(synth.workloads()["hybrid_prefetch"], n_layers=6, steps=4)
    rig = Rig(w)
    rig.m.moe_hybrid_start(rig.sc.handle, 8)
    st = Stepper(rig, n_pred=w.n_pred, fused=fused, hybrid=True)
    ids, wts = synth.make_routing(w)
    n_cpu = 0
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        refs = st.step(t, ids[t], wts[t], x)
        for layer in range(w.n_layers):
            n_cpu += int((refs[layer]["slots"] < 0).sum())
            full = rig.oracle_layer(layer, x[layer], ids[t, layer], wts[t, layer])
            assert_close(st.out[layer], full, w.fmt, what=f"step {t} layer {layer}")
    c = rig.m.moe_hybrid_counters(rig.sc.handle)
    assert c["jobs"] == w.steps * w.n_layers
    assert c["cpu_routes"] == n_cpu > 0
    for layer in range(w.n_layers):
        assert not rig.sc.stats(layer)["status_bits"] & 4  # no timed-out wait
    rig.m.moe_hybrid_stop(rig.sc.handle)


def test_hybrid_graph_replay_equals_eager():
    """The hybrid layers captured once as a CUDA graph and replayed with new
    routes equal the eager calls byte for byte, cache state included: the
    host side is driven by the job numbers the graph's kernels post."""
    w = synth.scaled(synth.workloads()["hybrid_prefetch"], n_layers=6, steps=4)
    blobs = synth.HostBlobs(w, pinned=True)
    eager, graphed = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    m = graphed.m
    for r in (eager, graphed):
        m.moe_hybrid_start(r.sc.handle, 8)
    se = Stepper(eager, n_pred=w.n_pred, fused=True, hybrid=True)
    ids, wts = synth.make_routing(w)
    L, R = w.n_layers, w.routes
    b_x = torch.empty(L, w.batch, w.hidden, dtype=torch.int16, device="cuda")
    b_ids = torch.empty(L, R, dtype=torch.int32, device="cuda")
    b_w = torch.empty(L, R, dtype=torch.float32, device="cuda")
    b_pred = torch.empty(L, w.n_pred, dtype=torch.int32, device="cuda")
    b_slots = torch.empty(L, R, dtype=torch.int32, device="cuda")
    b_out = torch.empty(L, w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
    cs = torch.cuda.Stream()
    flags = m.MOE_FUSED | m.MOE_HYBRID

    def enqueue():
        for layer in range(L):
            has_pred = layer + 1 < L
            m.moe_decode_layer(graphed.sc.handle, layer, b_x[layer], b_ids[layer], b_w[layer],
                               b_slots[layer], w.batch, w.top_k, w.fetch_cap,
                               b_pred[layer] if has_pred else None, w.n_pred if has_pred else 0,
                               None, None, b_out[layer], cs, None, flags)

    def load(t):
        b_x.copy_(_dev(synth.make_hidden(w, t)))
        b_ids.copy_(_dev(ids[t].reshape(L, -1)))
        b_w.copy_(_dev(wts[t].reshape(L, -1)))
        for layer in range(L - 1):
            b_pred[layer].copy_(_dev(synth.make_predictions(w, ids[t, layer + 1], t, layer)))

    load(0)
    with torch.cuda.stream(cs):
        enqueue()
    torch.cuda.synchronize()
    se.step(0, ids[0], wts[0], synth.make_hidden(w, 0))
    assert torch.equal(b_out.view(torch.int16), se.out.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        enqueue()
    for t in range(1, w.steps):
        load(t)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        se.step(t, ids[t], wts[t], synth.make_hidden(w, t))
        assert torch.equal(b_out.view(torch.int16), se.out.view(torch.int16)), f"token {t}"
        assert torch.equal(b_slots, se.slots)
    for layer in range(L):
        assert graphed.sc.stats(layer) == eager.sc.stats(layer)
    ce, cg = (m.moe_hybrid_counters(r.sc.handle) for r in (eager, graphed))
    assert ce["jobs"] == cg["jobs"] == w.steps * L and ce["cpu_routes"] == cg["cpu_routes"]


@pytest.mark.parametrize("fmt", [synth.FMT_MXFP4, synth.FMT_Q4_0])
def test_4bit_formats_layer_fused_equals_four_launch_path_and_oracle(fmt):
    """MXFP4 (e2m1 codes, one E8M0 scale per 32 row elements) and Q4_0 (fp16
    d * (q - 8) per 32 row elements) experts -- formats listed in FreeToken PR
    #491, section 7, "What did not change": the one-launch layer equals the
    four-launch path byte for byte, both match the fp64 oracle within the fp4
    tolerance, and every resident slot holds its expert's bytes.  The shared
    expert has the routed experts' format."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], fmt=fmt, n_layers=4, steps=8,
                     n_slots=60)
    blobs = synth.HostBlobs(w, pinned=True)
    a, b = Rig(w, blobs=blobs), Rig(w, blobs=blobs)
    sa, sb = Stepper(a, True, fused=True), Stepper(b, True)
    ids, wts = synth.make_routing(w)
    for t in range(w.steps):
        x = synth.make_hidden(w, t)
        sa.step(t, ids[t], wts[t], x)
        sb.step(t, ids[t], wts[t], x)
        assert torch.equal(sa.out.view(torch.int16), sb.out.view(torch.int16)), f"step {t}"
        if t in (0, w.steps - 1):
            for layer in range(w.n_layers):
                ref = a.oracle_layer(layer, x[layer], ids[t, layer], wts[t, layer])
                assert_close(sa.out[layer], ref, w.fmt, f"step {t} layer {layer}")
    assert sum(a.sc.stats(l)["fetched"] for l in range(w.n_layers)) > 20
    assert a.sc.stats(0)["status_bits"] == 0
    state = a.oc.state()
    for s, key in enumerate(state["slot_key"]):
        if key >= 0:
            assert np.array_equal(a.slot_bytes(0, s), a.blobs.blob(int(key))), s


def test_hybrid_wait_runs_out_and_reports_timeout():
    """Failure detection without a fault: while the executor is paused nothing
    answers the step's job, so the add kernel's bounded wait (1 s of
    %globaltimer) runs out, sets MOE_STATUS_TIMEOUT and leaves the GPU
    partial as the output; the context stays usable, and after resuming the
    next step is whole again."""
    w = synth.scaled(synth.workloads()["tiny"], steps=3, fetch_cap=1, batch=2)
    rig = Rig(w)
    m = rig.m
    m.moe_hybrid_start(rig.sc.handle, 2)
    st = Stepper(rig, hybrid=True)
    ids, wts = synth.make_routing(w)

    def run(t, whole):
        x = synth.make_hidden(w, t)
        refs = st.step(t, ids[t], wts[t], x, check_state=False)
        gs, os_ = rig.sc.stats(0), rig.oc.stats(0)  # exact, but for the timeout bit
        assert {**gs, "status_bits": 0} == {**os_, "status_bits": 0}, t
        slots = refs[0]["slots"].reshape(w.batch, w.top_k)
        mask = None if whole else (slots >= 0).astype(np.uint8)
        ref = rig.oracle_layer(0, x[0], ids[t, 0], wts[t, 0], mask=mask)
        assert_close(st.out[0], ref, w.fmt, f"step {t}")
        return slots

    run(0, whole=True)
    assert not rig.sc.stats(0)["status_bits"] & m.MOE_STATUS_TIMEOUT
    m.moe_hybrid_pause(rig.sc.handle, True)
    slots = run(1, whole=False)
    assert (slots < 0).any()  # the step had CPU routes, which the output now lacks
    assert rig.sc.stats(0)["status_bits"] & m.MOE_STATUS_TIMEOUT
    m.moe_hybrid_pause(rig.sc.handle, False)
    run(2, whole=True)
    m.moe_hybrid_stop(rig.sc.handle)
