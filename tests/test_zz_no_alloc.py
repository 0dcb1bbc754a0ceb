"""moe_routed_experts_noalloc through the C ABI.

The allocation-free entry point must give, bit for bit, what
moe_routed_experts gives for the same slots, inputs and weights (both run
the same streaming kernel, so the sums are taken in the same order), on two
calls in a row with nothing between them. It must also allocate no device
memory once its per-device set-up is done. The file name puts it last in
collection, so it runs both alone and after every other test in one process.
"""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import Rig, assert_close


def _workload():
    # Qwen3-MoE-like expert shapes (hidden 2048, inter 512, NVFP4), one layer of
    # 48 experts in 48 slots, 4 rows x top-8: 32 routes per call.
    return synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=1, n_experts=48,
                        n_slots=48, shared_inter=0, batch=4, steps=2)


def _resident_step(rig, t, ids):
    """Admit step t's routes and copy their misses in; device slot ids."""
    m = rig.m
    flat = np.ascontiguousarray(ids[t, 0].ravel(), np.int32)
    d_ids = torch.from_numpy(flat).cuda()
    d_slots = torch.empty_like(d_ids)
    m.moe_admit(rig.sc.handle, 0, d_ids, d_slots, len(flat), -1)
    m.moe_gather_missing(rig.sc.handle, m.MOE_PLAN_DEMAND)
    ref = rig.oc.admit(0, flat)
    return d_slots, ref


@pytest.mark.gpu
def test_noalloc_matches_routed_experts_on_two_calls_in_a_row():
    w = _workload()
    rig = Rig(w, max_rows=w.batch)
    m = rig.m
    ids, wts = synth.make_routing(w)
    d_x, d_s, d_w = [], [], []
    for t in range(2):
        d_slots, ref = _resident_step(rig, t, ids)
        assert (ref["slots"] >= 0).all()
        d_s.append(d_slots)
        d_x.append(torch.from_numpy(synth.make_hidden(w, t)[0].view(np.int16)).cuda())
        d_w.append(torch.from_numpy(np.ascontiguousarray(wts[t, 0], np.float32)).cuda())
    torch.cuda.synchronize()

    # the existing entry point, with the cache's own scratch
    want = []
    for t in range(2):
        o = torch.empty(w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
        m.moe_routed_experts(rig.sc.handle, 0, d_x[t], d_s[t], d_w[t], w.batch, w.top_k,
                             None, None, o)
        want.append(o)
    torch.cuda.synchronize()

    # the allocation-free entry point: two calls in a row on one stream
    status = torch.zeros(1, dtype=torch.int64, device="cuda")
    got = [torch.full((w.batch, w.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
           for _ in range(2)]
    for t in range(2):
        m.moe_routed_experts_noalloc(w.fmt, w.hidden, w.inter, rig.storage, rig.blobs.stride,
                                     w.n_slots, d_x[t], d_s[t], d_w[t], w.batch, w.top_k,
                                     got[t], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for t in range(2):
        a = got[t].view(torch.int16).cpu().numpy()
        b = want[t].view(torch.int16).cpu().numpy()
        assert np.array_equal(a, b), f"call {t}: {int((a != b).sum())} of {a.size} bf16 values differ"
        ref = rig.oracle_layer(0, synth.make_hidden(w, t)[0], ids[t, 0], wts[t, 0])
        assert_close(got[t], ref, w.fmt, f"call {t} against the oracle")

    # once set up, further calls allocate nothing: neither torch's allocator nor
    # the device's free memory moves
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    for t in (1, 0, 1):
        m.moe_routed_experts_noalloc(w.fmt, w.hidden, w.inter, rig.storage, rig.blobs.stride,
                                     w.n_slots, d_x[t], d_s[t], d_w[t], w.batch, w.top_k,
                                     got[t], status)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_before
    assert torch.cuda.mem_get_info()[0] == free_before
    assert np.array_equal(got[1].view(torch.int16).cpu().numpy(),
                          want[1].view(torch.int16).cpu().numpy())


@pytest.mark.gpu
def test_noalloc_skips_slot_ids_outside_the_pool():
    """Routes whose slot id lies outside [0, n_slots) (-1, n_slots, a large id)
    contribute nothing: the output equals moe_routed_experts' for the same slot
    ids byte for byte, and the oracle's layer with those routes masked out."""
    w = _workload()
    rig = Rig(w, max_rows=w.batch)
    m = rig.m
    ids, wts = synth.make_routing(w)
    d_slots, ref = _resident_step(rig, 0, ids)
    s = d_slots.cpu().numpy().reshape(w.batch, w.top_k).copy()
    bad = np.zeros_like(s, dtype=bool)
    for (b, j), v in zip([(0, 1), (1, 7), (2, 0), (3, 3), (3, 4)],
                         [-1, w.n_slots, 1 << 20, -7, w.n_slots + 1]):
        s[b, j] = v
        bad[b, j] = True
    d_s = torch.from_numpy(s.ravel().copy()).cuda()
    x = synth.make_hidden(w, 0)[0]
    d_x = torch.from_numpy(x.view(np.int16)).cuda()
    d_w = torch.from_numpy(np.ascontiguousarray(wts[0, 0], np.float32)).cuda()
    want = torch.empty(w.batch, w.hidden, dtype=torch.bfloat16, device="cuda")
    m.moe_routed_experts(rig.sc.handle, 0, d_x, d_s, d_w, w.batch, w.top_k, None, None, want)
    status = torch.zeros(1, dtype=torch.int64, device="cuda")
    got = [torch.full((w.batch, w.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
           for _ in range(2)]
    for t in range(2):
        m.moe_routed_experts_noalloc(w.fmt, w.hidden, w.inter, rig.storage, rig.blobs.stride,
                                     w.n_slots, d_x, d_s, d_w, w.batch, w.top_k, got[t], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    b = want.view(torch.int16).cpu().numpy()
    for t in range(2):
        assert np.array_equal(got[t].view(torch.int16).cpu().numpy(), b), f"call {t}"
    masked = rig.oracle_layer(0, x, ids[0, 0], wts[0, 0], mask=(~bad).astype(np.uint8))
    assert_close(got[1], masked, w.fmt, "skipped routes against the masked oracle layer")


@pytest.mark.gpu
def test_noalloc_rejects_unsupported_shape():
    import expert_slot_cache_lru_gb300 as m
    w = _workload()
    slots = torch.empty(256 * 1024 * 1024 // 64, dtype=torch.uint8, device="cuda")
    x = torch.zeros(17, w.hidden, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    ids = torch.zeros(17, dtype=torch.int32, device="cuda")
    wt = torch.ones(17, dtype=torch.float32, device="cuda")
    stride = (synth.blob_bytes(w.fmt, w.hidden, w.inter) + 255) // 256 * 256
    with pytest.raises(m.MoeError) as e:  # 17 rows: more than the streaming kernel takes
        m.moe_routed_experts_noalloc(w.fmt, w.hidden, w.inter, slots, stride, 1, x, ids, wt, 17,
                                     1, out)
    assert e.value.code == m.MOE_ERR_UNSUPPORTED


def test_noalloc_host_checks_without_a_device():
    """Size and argument checks happen on the host before any CUDA call."""
    import expert_slot_cache_lru_gb300 as m
    H, I, fmt = 2048, 512, synth.FMT_NVFP4
    stride = (synth.blob_bytes(fmt, H, I) + 255) // 256 * 256
    base, x, ids, wt, out = 1 << 20, 2 << 20, 3 << 20, 4 << 20, 5 << 20  # never dereferenced

    def call(**kw):
        a = dict(wfmt=fmt, hidden=H, inter=I, d_slots=base, slot_stride=stride, n_slots=8,
                 d_x=x, d_slot_ids=ids, d_w=wt, n_rows=1, k=8, d_out=out, stream=0)
        a.update(kw)
        with pytest.raises(m.MoeError) as e:
            m.moe_routed_experts_noalloc(**a)
        return e.value.code

    # 16 rows x 64 routes x 512 x 4 bytes = 2 MiB > 1 MiB of scratch
    assert call(n_rows=16, k=64) == m.MOE_ERR_SCRATCH
    limit = (m.MOE_NOALLOC_SCRATCH_BYTES - 256) // 4
    assert call(n_rows=1, k=1, inter=(limit // 32 + 1) * 32,
                slot_stride=1 << 30) == m.MOE_ERR_SCRATCH
    assert "1 MiB" in m.moe_strerror(m.MOE_ERR_SCRATCH)
    assert call(slot_stride=stride - 256) == m.MOE_ERR_INVALID_ARG
    assert call(slot_stride=stride + 16) == m.MOE_ERR_INVALID_ARG
    assert call(d_slots=base + 16) == m.MOE_ERR_INVALID_ARG
    assert call(d_x=x + 8) == m.MOE_ERR_INVALID_ARG
    assert call(d_out=x) == m.MOE_ERR_INVALID_ARG
    assert call(d_w=None) == m.MOE_ERR_INVALID_ARG
    assert call(wfmt=7) == m.MOE_ERR_INVALID_ARG
    assert call(n_slots=0) == m.MOE_ERR_INVALID_ARG
