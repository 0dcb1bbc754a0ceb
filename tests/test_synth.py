"""The synthetic workloads have the shapes and statistics they claim."""
import numpy as np

import oracle
import synth


def test_qwen3moe_routing_misses_about_28_per_token():
    """Zipf(1.1) routing with temporal reuse on a 3,164-slot LRU pool misses
    about 28 experts per token in steady state (steps 64..511), the miss rate
    of the 16K-context decode in FreeToken issue #753 (section Setup)."""
    w = synth.workloads()["qwen3moe_decode"]
    ids, wts = synth.make_routing(w)
    assert ids.shape == (512, 40, 1, 8)
    assert np.allclose(wts.sum(-1), 1.0, atol=1e-6)
    for t in range(0, 512, 97):  # top-k distinct per row
        assert all(len(set(ids[t, l, 0])) == 8 for l in range(40))
    oc = oracle.OracleCache(w.n_layers, w.n_experts, w.n_slots)
    per_token = []
    for t in range(w.steps):
        before = sum(oc.stats(l)["misses"] for l in range(w.n_layers))
        for l in range(w.n_layers):
            oc.admit(l, ids[t, l].ravel())
        per_token.append(sum(oc.stats(l)["misses"] for l in range(w.n_layers)) - before)
    assert abs(np.mean(per_token[64:]) - 28.0) < 1.0


def test_wide_decode_shapes():
    w = synth.workloads()["wide_decode"]
    ids, _ = synth.make_routing(w, steps=1)
    assert ids.shape == (1, 1, 600, 2)
    assert len(synth.prefill_ids(w)) == 307
    d = len(np.unique(ids))
    assert 650 < d < 760  # about 1024 * (1 - (1 - 2/1024)^600) = 707 distinct


def test_blob_sizes():
    assert synth.blob_bytes(synth.FMT_BF16, 64, 128) == 49152
    assert synth.blob_bytes(synth.FMT_NVFP4, 2048, 512) == 1769472 + 16
    assert synth.blob_bytes(synth.FMT_NVFP4, 2048, 768) == 2654208 + 16
    assert synth.blob_bytes(synth.FMT_BF16, 4096, 1024) == 25165824
    for fmt, H, I in [(0, 64, 128), (1, 2048, 512), (1, 2048, 768), (0, 4096, 1024)]:
        assert oracle.blob_bytes(fmt, H, I) == synth.blob_bytes(fmt, H, I)


def test_4bit_format_blobs_are_deterministic_and_in_range():
    """MXFP4 and Q4_0 blobs: sizes agree with the oracle, the same key gives the
    same bytes, and the scales stay in the recipe's ranges (E8M0 118..121;
    fp16 d in [0.001, 0.005))."""
    H, I = 2048, 512
    assert synth.blob_bytes(synth.FMT_MXFP4, H, I) == 3 * H * I // 2 + 3 * H * I // 32
    assert synth.blob_bytes(synth.FMT_Q4_0, H, I) == 3 * H * I // 2 + 3 * H * I // 16
    for fmt, banks in ((synth.FMT_MXFP4, synth.mxfp4_banks), (synth.FMT_Q4_0, synth.q4_banks)):
        assert oracle.blob_bytes(fmt, H, I) == synth.blob_bytes(fmt, H, I)
        a = np.empty(synth.blob_bytes(fmt, H, I), np.uint8)
        b = np.empty_like(a)
        synth.fill_blob(a, fmt, H, I, synth.Rng(3, 7))
        synth.fill_blob(b, fmt, H, I, synth.Rng(3, 7))
        assert np.array_equal(a, b)
        o = banks(H, I)
        sc = a[o["scale"][0]:o["end"]]
        if fmt == synth.FMT_MXFP4:
            assert sc.min() >= 118 and sc.max() <= 121
        else:
            d = sc.view(np.float16).astype(np.float64)
            assert d.min() >= 0.001 * (1 - 2 ** -10) and d.max() < 0.005 * (1 + 2 ** -10)
