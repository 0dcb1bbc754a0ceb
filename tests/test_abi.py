"""The C-ABI library without a GPU: it builds, loads, exports every entry
point include/moe_cache.h declares, lays its structs out as the binding does,
and rejects bad descriptors on the host before touching CUDA."""
import ctypes as C
import json
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "moe_cache.h")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import expert_slot_cache_lru_gb300 as mod
    return mod


def declared() -> list[str]:
    src = open(HDR).read()
    return re.findall(r"^MOE_API\s+(?:const\s+)?\w+\*?\s+(moe_\w+)\(", src, flags=re.M)


def test_exports_every_declared_symbol(m):
    names = declared()
    assert len(names) >= 16
    out = subprocess.run(["nm", "-D", "--defined-only", m.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (moe_\w+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = C.CDLL(m.LIB_PATH)
    for n in names:
        getattr(lib, n)


def test_struct_layout_matches_header(m, tmp_path):
    prog = tmp_path / "layout.c"
    fields = {
        "moe_cache_desc": [f for f, _ in m.moe_cache_desc._fields_],
        "moe_stats": [f for f, _ in m.moe_stats._fields_],
        "moe_views": [f for f, _ in m.moe_views._fields_],
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HDR}"', "int main(void){"]
    for s, fs in fields.items():
        lines.append(f'printf("{s} %zu\\n", sizeof({s}));')
        for f in fs:
            lines.append(f'printf("{s}.{f} %zu\\n", offsetof({s}, {f}));')
    lines.append("return 0;}")
    prog.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-o", str(exe), str(prog)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                  check=True).stdout.splitlines())
    for s, fs in fields.items():
        cls = getattr(m, s)
        assert int(got[s]) == C.sizeof(cls), s
        for f in fs:
            assert int(got[f"{s}.{f}"]) == getattr(cls, f).offset, (s, f)


def test_host_side_validation(m):
    assert m.abi_version() == 1
    assert m.moe_strerror(m.MOE_ERR_CONFIG) == "invalid cache descriptor"

    def desc(**kw):
        d = m.moe_cache_desc()
        base = dict(n_layers=2, n_experts=8, n_slots=4, pool_mode=0, max_routes=16, max_rows=1)
        base.update(kw)
        for k, v in base.items():
            setattr(d, k, v)
        return d

    bad = [
        dict(n_layers=0), dict(n_experts=0), dict(n_experts=16385), dict(n_slots=-1),
        dict(pool_mode=7), dict(max_routes=0), dict(max_rows=17), dict(max_pred=-1),
        dict(max_pred=4, n_slots=0),                      # prefetch needs a cache
        dict(hidden=48, inter=64, slot_bytes=6 * 48 * 64),  # H not a multiple of 32
        dict(hidden=64, inter=64, slot_bytes=123),         # slot_bytes != blob size
        dict(hidden=64, inter=64, wfmt=7, slot_bytes=6 * 64 * 64),  # no such format
        dict(slot_bytes=64),                               # storage without pointers
    ]
    for kw in bad:
        with pytest.raises(m.MoeError) as ei:
            m.moe_cache_create(desc(**kw))
        assert ei.value.code == m.MOE_ERR_CONFIG, kw
    if not torch.cuda.is_available():
        with pytest.raises(m.MoeError) as ei:
            m.moe_cache_create(desc())
        assert ei.value.code == m.MOE_ERR_CUDA
    # the hybrid executor's entry points check their arguments on the host
    for call in (lambda: m.moe_hybrid_start(0, 4), lambda: m.moe_hybrid_stop(0),
                 lambda: m.moe_hybrid_counters(0)):
        with pytest.raises(m.MoeError) as ei:
            call()
        assert ei.value.code == m.MOE_ERR_INVALID_ARG


def test_blob_bytes_agree_with_header_layout(m):
    import synth
    for fmt, H, I in [(0, 64, 128), (1, 2048, 512), (1, 2048, 768), (0, 4096, 1024),
                      (2, 2048, 512), (2, 64, 96), (3, 2048, 512), (3, 64, 96)]:
        assert m.blob_bytes(fmt, H, I) == synth.blob_bytes(fmt, H, I)


def test_route_split_example(m):
    with open(os.path.join(ROOT, "tests", "golden", "worked_examples.json")) as f:
        g = json.load(f)["route_split"]
    cpu_ids, gpu_slots, gpu_w = m.split_routes(torch.tensor(g["ids"]),
                                               torch.tensor(g["cache_result"]),
                                               torch.tensor(g["weights"]))
    assert cpu_ids.tolist() == g["cpu_ids"]
    assert gpu_slots.tolist() == g["gpu_slot_ids"]
    assert gpu_w.tolist() == pytest.approx(g["gpu_weights"])
    # complementary masks: each route on exactly one side
    assert all((c >= 0) != (w != 0) for c, w in zip(cpu_ids.tolist(), gpu_w.tolist()))


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "expert_slot_cache_lru_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", src), f
    out = subprocess.run(["nm", "-D", os.path.join(pkg, "libmoecache.so")], capture_output=True,
                         text=True).stdout
    names = [ln.split()[-1] for ln in out.splitlines() if ln.strip()]
    assert not [n for n in names if n.startswith(("oc_", "om_"))]
