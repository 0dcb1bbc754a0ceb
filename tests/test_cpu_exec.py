"""The hybrid CPU executor's host math (moe_cpu_experts) against the fp64 oracle.

The CPU partial of a step is the sum, over the routes the admission left at -1
(FreeToken PR #491 "refactor(moe): extract hybrid decode orchestration",
section 5 "How routes are split"), of w * FFN_e(x_b), computed in fp32 on the
host.  It must match the oracle's masked layer within fp32 rounding, ignore
routes with a slot or an invalid id, and give the same bits for any thread
count.  No GPU is needed.
"""
import numpy as np
import pytest

import expert_slot_cache_lru_gb300 as m
import oracle
import synth

FMT = {synth.FMT_BF16: m.MOE_W_BF16, synth.FMT_NVFP4: m.MOE_W_NVFP4,
       synth.FMT_MXFP4: m.MOE_W_MXFP4, synth.FMT_Q4_0: m.MOE_W_Q4_0}


def _case(w, batch, seed, frac_cpu=0.5):
    """Blobs of one layer, x, ids, slot ids (-1 = CPU route) and weights."""
    blobs = synth.HostBlobs(w, pinned=False)
    ptrs = [blobs.addr(e) for e in range(w.n_experts)]
    rng = np.random.default_rng(seed)
    x = synth.make_hidden(synth.scaled(w, n_layers=1), seed, batch=batch)[0]
    ids = np.stack([rng.choice(w.n_experts, w.top_k, replace=False) for _ in range(batch)])
    ids = ids.astype(np.int32)
    slots = np.where(rng.random(ids.shape) < frac_cpu, -1, 7).astype(np.int32)
    wts = rng.random(ids.shape).astype(np.float32)
    return blobs, ptrs, x, ids, slots, wts


def _reference(w, blobs, x, ids, slots, wts):
    mask = ((slots < 0) & (ids >= 0) & (ids < w.n_experts)).astype(np.uint8)
    return oracle.layer(w.fmt, [blobs.blob(e) for e in range(w.n_experts)], w.n_experts,
                        w.hidden, w.inter, x, np.clip(ids, 0, w.n_experts - 1), wts, mask=mask)


def _close(got, ref):
    atol = 1e-5 * float(np.max(np.abs(ref))) + 1e-12
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= atol + 1e-4 * np.abs(ref)), float(np.max(err))


SHAPES = {
    "bf16_tiny": synth.scaled(synth.workloads()["tiny"], n_experts=16, top_k=2),
    "nvfp4_small": synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=1, n_experts=8,
                                hidden=256, inter=128, top_k=4),
    "mxfp4_small": synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=1, n_experts=8,
                                hidden=256, inter=128, top_k=4, fmt=synth.FMT_MXFP4),
    "q4_0_small": synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=1, n_experts=8,
                               hidden=256, inter=128, top_k=4, fmt=synth.FMT_Q4_0),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_cpu_partial_matches_masked_oracle(name):
    w = SHAPES[name]
    blobs, ptrs, x, ids, slots, wts = _case(w, batch=3, seed=11)
    got = m.moe_cpu_experts(FMT[w.fmt], w.hidden, w.inter, ptrs, x, ids, slots, wts, n_threads=3)
    _close(got, _reference(w, blobs, x, ids, slots, wts))


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_thread_count_does_not_change_bits(name):
    w = SHAPES[name]
    _, ptrs, x, ids, slots, wts = _case(w, batch=4, seed=12, frac_cpu=0.7)
    outs = [m.moe_cpu_experts(FMT[w.fmt], w.hidden, w.inter, ptrs, x, ids, slots, wts, n_threads=t)
            for t in (1, 2, 5, 16)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_routes_with_a_slot_or_an_invalid_id_contribute_nothing():
    w = SHAPES["bf16_tiny"]
    blobs, ptrs, x, ids, slots, wts = _case(w, batch=3, seed=13)
    # every route has a slot: exact zeros
    got = m.moe_cpu_experts(FMT[w.fmt], w.hidden, w.inter, ptrs, x, ids, np.zeros_like(slots), wts)
    assert not np.any(got)
    # one CPU route in row 1 only; an out-of-range id at -1 in row 2 is ignored
    slots = np.zeros_like(slots)
    slots[1, 0] = -1
    ids = ids.copy()
    ids[2, 1], slots[2, 1] = w.n_experts + 5, -1
    got = m.moe_cpu_experts(FMT[w.fmt], w.hidden, w.inter, ptrs, x, ids, slots, wts)
    assert not np.any(got[0]) and not np.any(got[2])
    one = wts[1, 0] * oracle.expert_ffn(w.fmt, blobs.blob(int(ids[1, 0])), w.hidden, w.inter, x[1])
    _close(got[1:2], one[None, :])


def test_full_size_hybrid_expert_rows():
    """Two CPU routes of the hybrid decode's expert shape (bf16, H 4096, I 1024)."""
    w = synth.scaled(synth.workloads()["hybrid_prefetch"], n_layers=1, n_experts=3,
                     n_blob_alias=0, top_k=3)
    blobs, ptrs, x, ids, slots, wts = _case(w, batch=1, seed=14)
    slots[:] = [[-1, 3, -1]]
    got = m.moe_cpu_experts(FMT[w.fmt], w.hidden, w.inter, ptrs, x, ids, slots, wts, n_threads=8)
    _close(got, _reference(w, blobs, x, ids, slots, wts))


def test_argument_checks():
    w = SHAPES["bf16_tiny"]
    _, ptrs, x, ids, slots, wts = _case(w, batch=1, seed=15)
    with pytest.raises(m.MoeError):
        m.moe_cpu_experts(7, w.hidden, w.inter, ptrs, x, ids, slots, wts)
    with pytest.raises(m.MoeError):
        m.moe_cpu_experts(FMT[w.fmt], w.hidden + 1, w.inter, ptrs, x, ids, slots, wts)
    with pytest.raises(m.MoeError):
        m.moe_cpu_experts(FMT[w.fmt], w.hidden, w.inter, ptrs, x, ids, slots, wts, n_threads=0)


@pytest.mark.parametrize("name,threads,jobs", [("bf16_tiny", 4, 3000), ("bf16_tiny", 1, 300),
                                               ("nvfp4_small", 8, 400), ("q4_0_small", 3, 200)])
def test_job_protocol_over_host_mailbox(name, threads, jobs):
    """The executor's coordinator and workers over a mailbox in plain host
    memory, fed thousands of random steps the way the GPU posts them (a pause
    every 97th job, which must stay unanswered while paused): every answer
    equals the direct host math bit for bit and no job is lost."""
    w = SHAPES[name]
    blobs = synth.HostBlobs(w, pinned=False)
    ptrs = [blobs.addr(e) for e in range(w.n_experts)]
    assert m.moe_hybrid_selftest(FMT[w.fmt], w.hidden, w.inter, ptrs, max_rows=3, k=w.top_k,
                                 n_threads=threads, n_jobs=jobs, seed=jobs) == 0
