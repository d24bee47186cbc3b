"""Admission control and lazy page assignment for the shared KV page pool,
stated plainly in Python (TEST INFRASTRUCTURE ONLY: only ``tests/`` and the
CPU legs of ``bench.py`` use it; the library never imports it).

Rules, from the samir-vllm pages
[6 Hours of YouTube and 85 handtyped pages of notes on LLM Inference - Start
here, the README paragraphs after the feature list (admission, FIFO waiting,
rejection, --stats); samir-vllm: Build LLM Inference From Scratch in C++ and
CUDA, "Admission control: how the scheduler avoids deadlock"; roxreport
article on the same project, paged key-value cache paragraph]:

* A request with P prompt tokens and an output allowance N reserves credits
  for its largest processed prefix, P + N - 1 tokens (the last predicted
  token is returned, never processed), rounded up to whole 16-token pages in
  each of the 16 layers.
* N is the requested maximum clamped to the context: N = min(max_new,
  max_seq_len - P). (Reading: prompt plus output stays within the context.)
* A request whose budget exceeds the whole pool is rejected at submission.
* Requests are admitted in FIFO order while their budget fits in the credits
  not held by active requests; a request that does not fit waits, and so
  does everything behind it (no overtaking).
* Continuous batching admits whenever credits allow; static batching admits
  a new group only when the current group has finished.
* Credits are separate from physical pages: pages are taken from the free
  list only when a sequence grows into a new page, one per layer.
* Finishing (early or not) returns the assigned pages and all credits.
* Counters as the --stats flag reports them: pool size, peak active
  requests, largest decode batch, peak assigned pages, admission waits, free
  pages.

Readings where the pages are silent: a prompt must satisfy
1 <= P < max_seq_len and max_new >= 1, else the submission is invalid; free
pages are handed out lowest id first; "admission waits" counts requests that
were still queued after at least one admission pass that followed their
submission (each request at most once).
"""

import heapq
import math

OK = "ok"
INVALID = "invalid"
REJECTED = "rejected"


def allowed_new_tokens(prompt_tokens, max_new_tokens, max_seq_len):
    """Output allowance after clamping to the context."""
    return min(max_new_tokens, max_seq_len - prompt_tokens)


def processed_prefix(prompt_tokens, max_new_tokens, max_seq_len):
    """Largest number of tokens the request ever holds in the cache."""
    return prompt_tokens + allowed_new_tokens(prompt_tokens, max_new_tokens, max_seq_len) - 1


def budget_pages(prompt_tokens, max_new_tokens, num_layers=16, page_size=16, max_seq_len=2048):
    """Credits (physical pages over all layers) a request reserves."""
    prefix = processed_prefix(prompt_tokens, max_new_tokens, max_seq_len)
    return math.ceil(prefix / page_size) * num_layers


class Request:
    def __init__(self, rid, prompt_tokens, max_new_tokens, budget, prefix):
        self.rid = rid
        self.prompt_tokens = prompt_tokens
        self.max_new_tokens = max_new_tokens
        self.budget = budget
        self.prefix = prefix          # largest length it may grow to
        self.pages = None             # per layer: list of physical ids, once admitted
        self.length = 0
        self.waited = False


class AdmissionScheduler:
    def __init__(self, num_pages, num_layers=16, page_size=16, max_seq_len=2048,
                 static_batching=False):
        self.num_pages = num_pages
        self.num_layers = num_layers
        self.page_size = page_size
        self.max_seq_len = max_seq_len
        self.static_batching = static_batching
        self.free = list(range(num_pages))      # a heap: lowest id first
        heapq.heapify(self.free)
        self.credits = num_pages                # credits not held by active requests
        self.queue = []                          # waiting requests, FIFO
        self.active = []                         # admitted, in admission order
        self.requests = {}
        self.next_id = 0
        self.stats = {"pool_pages": num_pages, "submitted": 0, "rejected": 0, "admitted": 0,
                      "finished": 0, "peak_active": 0, "largest_decode_batch": 0,
                      "peak_assigned_pages": 0, "admission_waits": 0}

    def budget(self, prompt_tokens, max_new_tokens):
        return budget_pages(prompt_tokens, max_new_tokens, self.num_layers, self.page_size,
                            self.max_seq_len)

    # -- submission
    def submit(self, prompt_tokens, max_new_tokens):
        """Returns (status, request id or None)."""
        if prompt_tokens < 1 or prompt_tokens >= self.max_seq_len or max_new_tokens < 1:
            return INVALID, None
        budget = self.budget(prompt_tokens, max_new_tokens)
        self.stats["submitted"] += 1
        if budget > self.num_pages:
            self.stats["rejected"] += 1
            return REJECTED, None
        rid = self.next_id
        self.next_id += 1
        req = Request(rid, prompt_tokens, max_new_tokens, budget,
                      processed_prefix(prompt_tokens, max_new_tokens, self.max_seq_len))
        self.requests[rid] = req
        self.queue.append(req)
        return OK, rid

    # -- admission
    def admit(self):
        """One admission pass; returns the ids admitted, in order."""
        admitted = []
        if not (self.static_batching and self.active):
            while self.queue and self.queue[0].budget <= self.credits:
                req = self.queue.pop(0)
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

    # -- growth
    def extend(self, rid, length):
        """Makes positions < length addressable: a page per layer for every
        16-token page the sequence reaches. Returns a status."""
        req = self.requests.get(rid)
        if req is None or req.pages is None or length < 0 or length > req.prefix:
            return INVALID
        need = math.ceil(length / self.page_size)
        for layer in range(self.num_layers):
            while len(req.pages[layer]) < need:
                req.pages[layer].append(heapq.heappop(self.free))
        req.length = max(req.length, length)
        self.stats["peak_assigned_pages"] = max(self.stats["peak_assigned_pages"],
                                                self.assigned_pages())
        return OK

    def finish(self, rid):
        req = self.requests.get(rid)
        if req is None or req.pages is None:
            return INVALID
        for layer_pages in req.pages:
            for p in layer_pages:
                heapq.heappush(self.free, p)
        self.credits += req.budget
        self.active.remove(req)
        del self.requests[rid]
        self.stats["finished"] += 1
        return OK

    # -- a decode step's batch
    def decode_batch(self):
        """The active requests in admission order (one decode step's batch)."""
        ids = [r.rid for r in self.active]
        self.stats["largest_decode_batch"] = max(self.stats["largest_decode_batch"], len(ids))
        return ids

    def block_tables(self, ids, max_pages):
        """[layers][len(ids)][max_pages] page ids, -1 where none is assigned."""
        rows = []
        for layer in range(self.num_layers):
            layer_rows = []
            for rid in ids:
                pages = self.requests[rid].pages[layer]
                layer_rows.append(pages + [-1] * (max_pages - len(pages)))
            rows.append(layer_rows)
        return rows

    # -- counters
    def assigned_pages(self):
        return self.num_pages - len(self.free)

    def snapshot(self):
        s = dict(self.stats)
        s["free_pages"] = len(self.free)
        s["free_credits"] = self.credits
        s["active"] = len(self.active)
        s["waiting"] = len(self.queue)
        return s
