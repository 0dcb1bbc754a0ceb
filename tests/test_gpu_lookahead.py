"""The look-ahead producer on the GPU against the oracle.

llama.cpp fork PR #126 "cuda : MoE look-ahead expert prefetch (PR-A consumer)
+ LFRU eviction guard", sections What and "Open for PR-P1 (producer)": the
predicted ids of layer L+1, produced while layer L runs.  The reading (the
pages leave the predictor open): layer L+1's router on layer L's hidden
state, each row's k largest logits, ties to the lower id.

The GPU sums in fp32 and the oracle in fp64, so where two logits are closer
than the fp32 rounding bound either order is correct: each GPU pick is
checked to be a valid largest remaining logit within that bound, and rows
whose order is unambiguous must equal the oracle's exactly.  Logits that are
bit-identical on both sides (duplicated router rows) must follow the tie rule.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import Rig

pytestmark = pytest.mark.gpu


def _bf16_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _rig(E: int, H: int, rows: int, n_pred: int = 0, n_layers: int = 1) -> Rig:
    """A cache of E experts of width H (NVFP4, the smallest intermediate, so
    that the host blobs stay small); the producer uses only its shape."""
    w = synth.scaled(synth.workloads()["qwen3moe_decode"], n_layers=n_layers, n_experts=E,
                     hidden=H, inter=32, shared_inter=0, n_slots=min(E, 64), batch=rows, steps=1,
                     n_pred=n_pred)
    return Rig(w, max_rows=rows)


def _predict(rig: Rig, x: np.ndarray, router: np.ndarray, k: int, stream=None) -> np.ndarray:
    m = rig.m
    d_x = torch.from_numpy(x.view(np.int16)).cuda()
    d_r = torch.from_numpy(router.view(np.int16)).cuda()
    d_p = torch.full((x.shape[0] * k,), -7, dtype=torch.int32, device="cuda")
    m.moe_lookahead_predict(rig.sc.handle, d_x, d_r, x.shape[0], k, d_p, stream)
    torch.cuda.synchronize()
    return d_p.cpu().numpy().reshape(x.shape[0], k)


def _check(got: np.ndarray, x: np.ndarray, router: np.ndarray, k: int) -> int:
    """Every row valid within the fp32 bound; returns the rows equal to the oracle."""
    want, z = oracle.lookahead_predict(x, router, k)
    H = x.shape[1]
    # |fp32 sum - exact| <= (H / 32 + 5) * 2^-24 * sum |w x|: a lane's H / 32
    # sequential fma, then a 5-level tree; (H / 32 + 7) and doubled for margin
    mag = np.abs(_bf16_f32(x)).astype(np.float64) @ np.abs(_bf16_f32(router)).astype(np.float64).T
    eps = 2.0 * (H / 32 + 7) * 2.0 ** -24 * mag
    equal = 0
    for b in range(x.shape[0]):
        g = got[b]
        assert len(set(g.tolist())) == k and g.min() >= 0 and g.max() < router.shape[0], (b, g)
        left = np.ones(router.shape[0], bool)
        for r in range(k):
            e = int(g[r])
            assert left[e], (b, r, e)
            o = np.flatnonzero(left)
            # no expert still available beats the pick by more than both bounds
            assert np.all(z[b, e] + eps[b, e] + eps[b, o] >= z[b, o]), (b, r, e)
            left[e] = False
        equal += int(np.array_equal(g, want[b]))
        zs = np.sort(z[b])[::-1]
        n = min(k, len(zs) - 1)  # the gaps inside the top k and, if any, to the next
        gaps = zs[:n] - zs[1:n + 1]
        if np.all(gaps > 2 * eps[b].max()):  # unambiguous: the oracle's answer exactly
            assert np.array_equal(g, want[b]), (b, g, want[b])
    return equal


@pytest.mark.parametrize("rows,k", [(1, 8), (20, 8), (16, 32)])
def test_lookahead_matches_oracle(rows, k):
    """256 experts, H 2048 (the decode benchmark's layer shape): one row (the
    decode step), 20 rows (x staged in chunks of 8) and 16 rows at k = 32."""
    rig = _rig(256, 2048, rows)
    w = rig.w
    router = synth.make_router(w, 1)
    x = synth.make_hidden(w, 0)[0]
    got = _predict(rig, x, router, k)
    assert _check(got, x, router, k) >= rows - 1  # near-ties at the fp32 bound are rare


@pytest.mark.parametrize("E,H,k", [(250, 1024, 1), (20, 1024, 20), (64, 4096, 5),
                                   (1000, 3072, 32)])
def test_lookahead_shapes(E, H, k):
    """Expert counts that are not a multiple of the CTA's 4 warps, k = 1,
    k = n_experts, and the other supported widths."""
    rig = _rig(E, H, 3)
    router = synth.make_router(rig.w, 0)
    x = synth.make_hidden(rig.w, 1)[0]
    got = _predict(rig, x, router, k)
    _check(got, x, router, k)


def test_lookahead_ties_go_to_the_lower_id():
    """Router rows 3, 9 and 40 are set to the row with the highest logits over
    the batch, and row 5 to row 2: copies give the same logit bits on the GPU
    (the same operations in the same order), so within each group of copies
    the lower id comes first, as in the oracle."""
    rig = _rig(64, 1024, 4)
    router = synth.make_router(rig.w, 0)
    x = synth.make_hidden(rig.w, 2)[0]
    _, z = oracle.lookahead_predict(x, router, 1)
    top = int(np.argmax(z.sum(axis=0)))  # copies of a row that is high in every row of x
    for e in (3, 9, 40):
        router[e] = router[top]
    router[5] = router[2]
    got = _predict(rig, x, router, 16)
    groups = [sorted({3, 9, 40, top}), [2, 5]]
    seen = 0
    for b in range(x.shape[0]):
        g = got[b].tolist()
        for grp in groups:
            idx = [g.index(e) for e in grp if e in g]
            assert idx == sorted(idx), (b, grp, g)
            seen += len(idx) > 1
    assert seen > 0  # some tie was inside a top 16
    _check(got, x, router, 16)


def test_lookahead_nan_logit_ranks_last():
    """A NaN router weight makes expert 7's logit NaN in every row: the GPU
    never picks it while any number remains, and ranks it last at k = n_experts."""
    rig = _rig(20, 1024, 3)
    router = synth.make_router(rig.w, 0)
    router[7, 5] = 0x7fc0  # bf16 NaN
    x = synth.make_hidden(rig.w, 3)[0]
    got = _predict(rig, x, router, 19)
    assert not (got == 7).any()
    got = _predict(rig, x, router, 20)
    assert (got[:, -1] == 7).all()
    want, _ = oracle.lookahead_predict(x, router, 20)
    assert (want[:, -1] == 7).all()


def test_lookahead_graph_replay_and_repeat():
    """The launch resets its own counter: three launches on different inputs
    captured in one graph and replayed twice give the eager answers."""
    rig = _rig(256, 2048, 2)
    m, w = rig.m, rig.w
    xs = [synth.make_hidden(w, t)[0] for t in range(3)]
    routers = [synth.make_router(w, l) for l in range(3)]
    eager = [_predict(rig, xs[i], routers[i], 8) for i in range(3)]
    d_x = [torch.from_numpy(x.view(np.int16)).cuda() for x in xs]
    d_r = [torch.from_numpy(r.view(np.int16)).cuda() for r in routers]
    d_p = [torch.zeros(2 * 8, dtype=torch.int32, device="cuda") for _ in range(3)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        for i in range(3):
            m.moe_lookahead_predict(rig.sc.handle, d_x[i], d_r[i], 2, 8, d_p[i], s)
    for _ in range(2):
        for p in d_p:
            p.zero_()
        g.replay()
        torch.cuda.synchronize()
        for i in range(3):
            assert np.array_equal(d_p[i].cpu().numpy().reshape(2, 8), eager[i])


def test_lookahead_feeds_the_prefetch():
    """The consumer takes the producer's output as it is: the predictions for
    layer 1 go straight from the producer's buffer into moe_prefetch, and the
    cache state equals the oracle's after prefetching the same ids."""
    rig = _rig(256, 2048, 4, n_pred=32, n_layers=2)
    m, w = rig.m, rig.w
    router = synth.make_router(w, 1)
    x = synth.make_hidden(w, 0)[0]
    d_x = torch.from_numpy(x.view(np.int16)).cuda()
    d_r = torch.from_numpy(router.view(np.int16)).cuda()
    d_p = torch.zeros(4 * 8, dtype=torch.int32, device="cuda")
    m.moe_lookahead_predict(rig.sc.handle, d_x, d_r, 4, 8, d_p, None)
    m.moe_prefetch(rig.sc.handle, 1, d_p, 32, None)
    torch.cuda.synchronize()
    pred = d_p.cpu().numpy()
    rig.oc.prefetch(1, pred)
    from tests.gpu_util import assert_state_equal
    assert_state_equal(rig.sc, rig.oc, what="after the producer's prefetch")
    assert rig.sc.stats(1) == rig.oc.stats(1)
    assert rig.sc.stats(1)["pf_filled"] > 0


def test_lookahead_argument_checks():
    rig = _rig(64, 1024, 2)
    m = rig.m
    x = torch.zeros(2, 1024, dtype=torch.int16, device="cuda")
    r = torch.zeros(64, 1024, dtype=torch.int16, device="cuda")
    p = torch.zeros(64, dtype=torch.int32, device="cuda")
    bad = [
        dict(n_rows=3, k_pred=2, code=m.MOE_ERR_CAPACITY),      # more rows than max_rows
        dict(n_rows=2, k_pred=33, code=m.MOE_ERR_UNSUPPORTED),  # k above 32
        dict(n_rows=2, k_pred=0, code=m.MOE_ERR_INVALID_ARG),
        dict(n_rows=-1, k_pred=2, code=m.MOE_ERR_INVALID_ARG),
    ]
    for c in bad:
        with pytest.raises(m.MoeError) as e:
            m.moe_lookahead_predict(rig.sc.handle, x, r, c["n_rows"], c["k_pred"], p, None)
        assert e.value.code == c["code"], c
    with pytest.raises(m.MoeError) as e:
        m.moe_lookahead_predict(rig.sc.handle, None, r, 2, 2, p, None)
    assert e.value.code == m.MOE_ERR_INVALID_ARG
    with pytest.raises(m.MoeError) as e:  # x not 16-byte aligned
        m.moe_lookahead_predict(rig.sc.handle, x.view(-1)[4:].data_ptr(), r, 1, 2, p, None)
    assert e.value.code == m.MOE_ERR_INVALID_ARG
    m.moe_lookahead_predict(rig.sc.handle, x, r, 0, 2, p, None)  # no rows: nothing to do
