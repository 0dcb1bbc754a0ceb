"""Host-only schedule test of one decode layer, with fake streams.

The operations moe_decode_layer enqueues (moe_schedule_trace records them in
order, per stream) are replayed on fake FIFO streams: an operation follows the
one before it on its stream, and a wait follows the record of its event.  The
order inside a layer is FreeToken issue #753's ("[Perf] Offloaded decode:
overlap the expert-miss gather with the same layer's shared expert, event-
ordered inside the CUDA graph", What we changed):
  compute: admit -> record(ready) -> shared expert -> wait(done) -> routed
  side:    wait(ready) -> gather -> record(done)
The checks are that the gather follows the admission, the routed FFN follows
the gather, and the shared expert does not wait for the gather.  Like the
page's CPU test, they catch the removal of either the producer's or the
consumer's wait.  Every failure after the fork must still join.
"""
import itertools

import pytest

import expert_slot_cache_lru_gb300 as m


def happens_before(trace):
    """{(i, j): op i completes before op j starts} over the fake streams."""
    n = len(trace)
    edges = {i: set() for i in range(n)}
    last = {}
    recorded = {}
    for i, tok in enumerate(trace):
        stream, op = tok.split(":")
        if stream in last:
            edges[last[stream]].add(i)
        last[stream] = i
        if op.startswith("record_"):
            recorded[op[len("record_"):]] = i
        if op.startswith("wait_"):
            ev = op[len("wait_"):]
            assert ev in recorded, f"wait on {ev} before its record"
            edges[recorded[ev]].add(i)
    hb = set()
    for i in range(n):  # reachability
        stack, seen = [i], set()
        while stack:
            for j in edges[stack.pop()]:
                if j not in seen:
                    seen.add(j)
                    stack.append(j)
        hb |= {(i, j) for j in seen}
    return hb


def index(trace, op):
    hits = [i for i, tok in enumerate(trace) if tok.split(":")[1] == op]
    assert len(hits) <= 1, (op, trace)
    return hits[0] if hits else None


def violations(trace, overlap):
    """The ordering rules of one layer that the trace breaks."""
    hb = happens_before(trace)
    at = {op: index(trace, op) for op in (
        "admit", "post", "prefetch", "gather_demand", "gather_prefetch", "shared", "routed",
        "add_cpu", "layer_stream")}
    bad = []

    def before(a, b):
        ia, ib = at[a], at[b]
        if ia is not None and ib is not None and (ia, ib) not in hb:
            bad.append(f"{a} !< {b}")

    before("admit", "gather_demand")       # the gather reads the admission's plan
    before("gather_demand", "routed")      # the routed FFN reads the gathered slots
    before("admit", "layer_stream")
    before("prefetch", "gather_prefetch")
    before("admit", "post")                # the host gets the rewritten slot ids
    before("post", "add_cpu")
    before("routed", "add_cpu")
    before("layer_stream", "add_cpu")
    if overlap and at["shared"] is not None and (at["gather_demand"], at["shared"]) in hb:
        bad.append("shared waits for the gather")  # the overlap of the page
    return bad


PLANS = [dict(one_launch=o, fused=f, overlap=v, pf=p, shared=s, hybrid=h)
         for o, f, v, p, s, h in itertools.product([False, True], repeat=6)
         if not (o and (not f or h))]  # one launch is a fused plan without the hybrid post


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: "-".join(k for k, v in p.items() if v) or "serial")
def test_every_plan_keeps_the_layer_order(plan):
    rc, trace = m.moe_schedule_trace(**plan)
    assert rc == m.MOE_OK and trace
    assert violations(trace, plan["overlap"] and not plan["fused"]) == []
    if plan["overlap"] and not plan["fused"]:  # the fork is joined within the layer
        assert "s:wait_ready" in trace and "c:wait_done" in trace


@pytest.mark.parametrize("pf,shared", [(False, False), (True, True), (True, False)])
def test_removing_either_wait_is_detected(pf, shared):
    rc, trace = m.moe_schedule_trace(overlap=True, pf=pf, shared=shared)
    assert rc == m.MOE_OK and violations(trace, True) == []
    producer = [t for t in trace if t != "s:wait_ready"]
    consumer = [t for t in trace if t != "c:wait_done"]
    assert "admit !< gather_demand" in violations(producer, True)
    assert "gather_demand !< routed" in violations(consumer, True)
    # the serial order, moved onto one stream, is valid without any event
    rc, serial = m.moe_schedule_trace(overlap=False, pf=pf, shared=shared)
    assert violations(serial, False) == []


def test_every_failure_after_the_fork_still_joins():
    rc, full = m.moe_schedule_trace(overlap=True, pf=True, shared=True)
    fork = full.index("s:wait_ready")
    for i in range(len(full)):
        rc, trace = m.moe_schedule_trace(overlap=True, pf=True, shared=True, fail_at=i)
        assert rc == m.MOE_ERR_CUDA, (i, trace)
        forked = len(trace) > fork and trace[fork] == "s:wait_ready" and i > fork
        if forked:  # a side stream was forked: it is joined before the call returns
            assert "c:wait_done" in trace[fork:] or trace[i] == "s:record_done", (i, trace)
        if trace[i] != "c:wait_done" and i > fork:
            assert "c:routed" not in trace[i + 1:], (i, trace)  # nothing computes after a failure
