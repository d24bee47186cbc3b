"""The admission oracle against its pins, and planted mistakes that the pins
must catch (each mutant is a subclass of the oracle with one rule broken)."""

import heapq
import math

import pytest

from oracle import admission as A
import admission_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_meets_pin(pin):
    pin(A.AdmissionScheduler, A.budget_pages)


def _budget_no_minus_one(p, n, layers=16, page=16, ctx=2048):
    return math.ceil((p + min(n, ctx - p)) / page) * layers


def _budget_one_layer(p, n, layers=16, page=16, ctx=2048):
    return math.ceil((p + min(n, ctx - p) - 1) / page)


class NoMinusOne(A.AdmissionScheduler):
    def budget(self, p, n):
        return _budget_no_minus_one(p, n)


class OneLayer(A.AdmissionScheduler):
    def budget(self, p, n):
        return _budget_one_layer(p, n)


class FirstFit(A.AdmissionScheduler):
    """Admits any queued request that fits, overtaking the head."""
    def admit(self):
        admitted = []
        if not (self.static_batching and self.active):
            for req in list(self.queue):
                if req.budget <= self.credits:
                    self.queue.remove(req)
                    self.credits -= req.budget
                    req.pages = [[] for _ in range(self.num_layers)]
                    self.active.append(req)
                    admitted.append(req.rid)
        for req in self.queue:
            if not req.waited:
                req.waited = True
                self.stats["admission_waits"] += 1
        self.stats["admitted"] += len(admitted)
        self.stats["peak_active"] = max(self.stats["peak_active"], len(self.active))
        return admitted


class StaticNeverWaits(A.AdmissionScheduler):
    def admit(self):
        saved = self.static_batching
        self.static_batching = False
        try:
            return super().admit()
        finally:
            self.static_batching = saved


class KeepsCredits(A.AdmissionScheduler):
    def finish(self, rid):
        req = self.requests.get(rid)
        st = super().finish(rid)
        if st == A.OK:
            self.credits -= req.budget
        return st


class RejectsAtPoolSize(A.AdmissionScheduler):
    def submit(self, p, n):
        if 1 <= p < self.max_seq_len and n >= 1 and self.budget(p, n) == self.num_pages:
            self.stats["submitted"] += 1
            self.stats["rejected"] += 1
            return A.REJECTED, None
        return super().submit(p, n)


class EagerPages(A.AdmissionScheduler):
    def admit(self):
        ids = super().admit()
        for rid in ids:
            req = self.requests[rid]
            need = math.ceil(req.prefix / self.page_size)
            for layer in range(self.num_layers):
                while len(req.pages[layer]) < need:
                    req.pages[layer].append(heapq.heappop(self.free))
        return ids


class WaitsPerPass(A.AdmissionScheduler):
    def admit(self):
        ids = super().admit()
        self.stats["admission_waits"] += sum(1 for r in self.queue if r.waited) - \
            sum(1 for r in self.queue if r.waited and not getattr(r, "_seen", False))
        for r in self.queue:
            r._seen = True
        return ids


MUTANTS = [
    ("budget without the unprocessed last token", NoMinusOne, _budget_no_minus_one),
    ("budget for one layer only", OneLayer, _budget_one_layer),
    ("first-fit admission overtakes the queue head", FirstFit, A.budget_pages),
    ("static batching admits while a group runs", StaticNeverWaits, A.budget_pages),
    ("finish keeps the credits", KeepsCredits, A.budget_pages),
    ("a budget equal to the pool is rejected", RejectsAtPoolSize, A.budget_pages),
    ("pages assigned eagerly at admission", EagerPages, A.budget_pages),
    ("admission waits counted per pass", WaitsPerPass, A.budget_pages),
]


@pytest.mark.parametrize("name,cls,budget_fn", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, cls, budget_fn):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(cls, budget_fn)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches: {name}"
