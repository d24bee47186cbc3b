"""Pins for the admission oracle (oracle/admission.py): hand-worked budgets
from the pages' rule, the pages' stated behaviours as small scenarios, a
brute-force page count, and invariants over random traces.

Each pin takes the scheduler class and the budget function so that the
mutation test can run the same pins against planted mistakes.
"""

import json
import math
import os
import random

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    with open(os.path.join(HERE, "golden", "admission_budgets.json")) as f:
        return json.load(f)


def pin_golden_budgets(cls, budget_fn):
    g = _golden()
    geo = g["geometry"]
    for c in g["cases"]:
        got = budget_fn(c["prompt"], c["max_new"], geo["num_layers"], geo["page_size"],
                        geo["max_seq_len"])
        assert got == c["budget"], (c, got)
        # the fixture is internally consistent
        assert c["prefix"] == c["prompt"] + c["allowed_new"] - 1
        assert c["pages_per_layer"] == -(-c["prefix"] // geo["page_size"])
        assert c["budget"] == c["pages_per_layer"] * geo["num_layers"]


def pin_budget_counts_touched_pages(cls, budget_fn):
    """Brute force: walk every processed position and count the distinct
    (layer, page index) pairs it touches."""
    rng = random.Random(7)
    for _ in range(300):
        prompt = rng.randint(1, 2047)
        max_new = rng.randint(1, 2500)
        allowed = min(max_new, 2048 - prompt)
        touched = set()
        for pos in range(prompt + allowed - 1):
            for layer in range(16):
                touched.add((layer, pos // 16))
        assert budget_fn(prompt, max_new, 16, 16, 2048) == len(touched)


def pin_pool_facts(cls, budget_fn):
    g = _golden()
    for pool in g["pools"]:
        assert pool["pages"] == pool["mib"] * 1024 * 1024 // 32768
        s = cls(pool["pages"])
        ids = []
        for _ in range(3):
            st, rid = s.submit(1000, 5000)      # the largest budget
            if pool.get("rejects_largest"):
                assert st == "rejected" and rid is None
            else:
                assert st == "ok"
                ids.append(rid)
        if not pool.get("rejects_largest"):
            assert s.admit() == ids[:pool["full_requests_at_once"]]
            assert s.snapshot()["waiting"] == 3 - pool["full_requests_at_once"]


def pin_budget_equal_to_pool_is_accepted(cls, budget_fn):
    s = cls(2048)
    st, rid = s.submit(1000, 5000)
    assert st == "ok" and s.admit() == [rid]
    s2 = cls(2047)
    assert s2.submit(1000, 5000)[0] == "rejected"
    snap = s2.snapshot()
    assert snap["rejected"] == 1 and snap["waiting"] == 0


def pin_fifo_without_overtaking(cls, budget_fn):
    """A small request behind a large one that does not fit waits too."""
    s = cls(3000)
    _, a = s.submit(1000, 5000)        # 2048, leaves 952 credits
    _, c = s.submit(1000, 5000)        # 2048: does not fit now
    _, d = s.submit(1, 16)             # 16: would fit, must not overtake
    assert s.admit() == [a]
    assert s.snapshot()["waiting"] == 2
    assert s.admit() == []
    assert s.finish(a) == "ok"
    assert s.admit() == [c, d]
    snap = s.snapshot()
    assert snap["admission_waits"] == 2 and snap["free_credits"] == 3000 - 2048 - 16


def pin_static_waits_for_the_group(cls, budget_fn):
    s = cls(4096, static_batching=True)
    _, a = s.submit(1, 16)
    _, b = s.submit(1, 16)
    assert s.admit() == [a, b]
    _, c = s.submit(1, 16)
    assert s.admit() == []            # the group is still running
    s.finish(a)
    assert s.admit() == []
    s.finish(b)
    assert s.admit() == [c]
    cont = cls(4096)
    _, a = cont.submit(1, 16)
    assert cont.admit() == [a]
    _, c = cont.submit(1, 16)
    assert cont.admit() == [c]        # continuous: admitted at once


def pin_pages_assigned_lazily(cls, budget_fn):
    s = cls(4096)
    _, a = s.submit(20, 100)           # prefix 119: 8 pages per layer
    s.admit()
    snap = s.snapshot()
    assert snap["free_pages"] == 4096 and snap["free_credits"] == 4096 - 128
    for length, per_layer in ((1, 1), (16, 1), (17, 2), (20, 2), (33, 3), (119, 8)):
        assert s.extend(a, length) == "ok"
        assert s.snapshot()["free_pages"] == 4096 - 16 * per_layer, length
    assert s.extend(a, 120) == "invalid"   # past the reserved prefix
    tables = s.block_tables([a], 128)
    assert len(tables) == 16
    flat = [p for layer in tables for p in layer[0] if p >= 0]
    assert len(flat) == len(set(flat)) == 128
    assert all(layer[0][8:] == [-1] * 120 for layer in tables)


def pin_finish_returns_pages_and_credits(cls, budget_fn):
    s = cls(4096)
    _, a = s.submit(20, 100)
    _, b = s.submit(1, 2047)
    s.admit()
    s.extend(a, 50)
    s.extend(b, 300)
    assert s.finish(a) == "ok"         # early completion
    snap = s.snapshot()
    assert snap["free_credits"] == 4096 - 2048
    assert snap["free_pages"] == 4096 - 16 * 19
    s.finish(b)
    snap = s.snapshot()
    assert snap["free_pages"] == snap["free_credits"] == 4096
    assert snap["peak_assigned_pages"] == 16 * 4 + 16 * 19
    assert s.finish(b) == "invalid"


def pin_invalid_submissions(cls, budget_fn):
    s = cls(4096)
    for prompt, max_new in ((0, 10), (2048, 1), (5000, 1), (10, 0), (-1, 5)):
        assert s.submit(prompt, max_new) == ("invalid", None)
    assert s.snapshot()["submitted"] == 0


def pin_random_trace_invariants(cls, budget_fn):
    """Random continuous and static traces: credits never overcommitted,
    assigned pages within budgets, FIFO admission, every admitted request can
    grow to its full prefix, and all pages come back."""
    for static in (False, True):
        rng = random.Random(11 + static)
        pool = 1024
        s = cls(pool, static_batching=static)
        order, admitted_order, live = [], [], {}
        largest = 0
        for step in range(400):
            if rng.random() < 0.3:
                st, rid = s.submit(rng.randint(1, 600), rng.randint(1, 700))
                if st == "ok":
                    order.append(rid)
            was_idle = not live
            new = s.admit()
            if static and new:
                assert was_idle          # a static group starts only when the last one ended
            admitted_order += new
            for rid in new:
                req = s.requests[rid]
                live[rid] = [req.prompt_tokens, req.prefix, req.budget]
            batch = s.decode_batch()
            largest = max(largest, len(batch))
            assert batch == [r for r in admitted_order if r in live]
            for rid in list(live):
                cur, prefix, budget = live[rid]
                assert s.extend(rid, cur) == "ok"
                per_layer = math.ceil(cur / 16)
                tab = s.block_tables([rid], 128)
                assert all(sum(p >= 0 for p in layer[0]) == per_layer for layer in tab)
                assert per_layer * 16 <= budget
                if cur >= prefix or rng.random() < 0.02:
                    assert s.finish(rid) == "ok"
                    del live[rid]
                else:
                    live[rid][0] = min(prefix, cur + rng.randint(1, 40))
            snap = s.snapshot()
            held = sum(v[2] for v in live.values())
            assert snap["free_credits"] == pool - held >= 0
            assigned = pool - snap["free_pages"]
            assert assigned <= held
        assert admitted_order == order[:len(admitted_order)]
        assert s.snapshot()["largest_decode_batch"] == largest
        for rid in list(live):
            s.finish(rid)
        while s.queue:
            for rid in s.admit():
                req = s.requests[rid]
                assert s.extend(rid, req.prefix) == "ok"
                s.finish(rid)
        snap = s.snapshot()
        assert snap["free_pages"] == snap["free_credits"] == pool


ALL_PINS = [pin_golden_budgets, pin_budget_counts_touched_pages, pin_pool_facts,
            pin_budget_equal_to_pool_is_accepted, pin_fifo_without_overtaking,
            pin_static_waits_for_the_group, pin_pages_assigned_lazily,
            pin_finish_returns_pages_and_credits, pin_invalid_submissions,
            pin_random_trace_invariants]
