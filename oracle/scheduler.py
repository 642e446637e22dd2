"""Plain-Python oracle of the request scheduler -- TEST INFRASTRUCTURE ONLY.

A direct restatement of the admission rules of the Tiny-vLLM README
translation ("Hours of YouTube and 85 handtyped pages of notes on LLM
Inference - Start here", section "現在のスコープ", and the static /
continuous batching item of "これまでの進捗"):

  * a request reserves credits for its largest processed prefix,
    prompt + allowed_new - 1 tokens, rounded up to whole pages, for every
    layer; allowed_new is max_new clamped to the context limit;
  * credits are separate from physical pages, which are taken lazily, the
    lowest free page id first;
  * the queue is FIFO: while the oldest waiting request does not fit, nobody
    behind it is admitted; a request larger than the pool is rejected;
  * static batching admits only when no admitted request is left,
    continuous batching whenever credits are free;
  * finished requests give their pages and credits back at the next
    scheduling point.

Slow and obvious on purpose (lists and linear scans).  The library's C++
scheduler (include/pkv_sched.h) is compared with it decision by decision.
"""
from __future__ import annotations

import math

REJECTED = "rejected"


class Req:
    def __init__(self, rid, prompt, allowed_new, credits):
        self.id = rid
        self.prompt = prompt
        self.allowed_new = allowed_new
        self.credits = credits
        self.state = "waiting"
        self.len = 0
        self.generated = 0
        self.waited = 0
        self.pages = []   # pages[layer] = list of page ids


class OracleScheduler:
    def __init__(self, num_pages, layers, max_context, page_size, static_batching):
        self.num_pages = num_pages
        self.layers = layers
        self.max_context = max_context
        self.page_size = page_size
        self.max_blocks = max_context // page_size
        self.static = bool(static_batching)
        self.free = list(range(num_pages))     # kept sorted
        self.free_credits = num_pages
        self.reqs = {}
        self.queue = []
        self.admitted = []
        self.release_next = []
        self.next_id = 0
        self.stats = dict(peak_active=0, largest_decode_batch=0, peak_allocated_pages=0,
                          admission_wait_total=0, admission_wait_max=0, submitted=0,
                          admitted=0, rejected=0, finished=0)

    def budget(self, prompt, max_new):
        if prompt < 1 or prompt > self.max_context or max_new < 1:
            return None
        allowed = min(max_new, self.max_context + 1 - prompt)
        return math.ceil((prompt + allowed - 1) / self.page_size) * self.layers

    def submit(self, prompt, max_new):
        credits = self.budget(prompt, max_new)
        if credits is None:
            return None
        self.stats["submitted"] += 1
        if credits > self.num_pages:
            self.stats["rejected"] += 1
            return REJECTED
        r = Req(self.next_id, prompt, min(max_new, self.max_context + 1 - prompt), credits)
        self.next_id += 1
        self.reqs[r.id] = r
        self.queue.append(r.id)
        return r.id

    def _take_page(self):
        p = self.free.pop(0)
        held = self.num_pages - len(self.free)
        self.stats["peak_allocated_pages"] = max(self.stats["peak_allocated_pages"], held)
        return p

    def _active(self):
        return [rid for rid in self.admitted if self.reqs[rid].state in ("admitted", "running")]

    def admit(self):
        for rid in self.release_next:
            r = self.reqs[rid]
            for layer in r.pages:
                self.free.extend(layer)
            self.free.sort()
            r.pages = []
            self.free_credits += r.credits
            r.credits = 0
        self.release_next = []
        self.admitted = [rid for rid in self.admitted if self.reqs[rid].state != "finished"]
        n = 0
        if not self.static or not self._active():
            while self.queue:
                head = self.reqs[self.queue[0]]
                if head.credits > self.free_credits:
                    break
                self.free_credits -= head.credits
                head.state = "admitted"
                self.stats["admission_wait_total"] += head.waited
                self.stats["admission_wait_max"] = max(self.stats["admission_wait_max"],
                                                       head.waited)
                self.stats["admitted"] += 1
                self.admitted.append(head.id)
                self.queue.pop(0)
                n += 1
        for rid in self.queue:
            self.reqs[rid].waited += 1
        self.stats["peak_active"] = max(self.stats["peak_active"], len(self._active()))
        return n

    def _finish_by_budget(self, r):
        if r.generated >= r.allowed_new:
            r.state = "finished"
            self.stats["finished"] += 1
            self.release_next.append(r.id)

    def _table(self, r):
        return [[r.pages[l][k] if k < len(r.pages[l]) else -1 for k in range(self.max_blocks)]
                for l in range(self.layers)]

    def next_prefill(self):
        for rid in self.admitted:
            r = self.reqs[rid]
            if r.state != "admitted":
                continue
            blocks = math.ceil(r.prompt / self.page_size)
            r.pages = [[self._take_page() for _ in range(blocks)] for _ in range(self.layers)]
            r.len = r.prompt
            r.generated = 1
            r.state = "running"
            self._finish_by_budget(r)
            return r.id, r.prompt, self._table(r)
        return None

    def decode_batch(self, max_batch):
        out = []
        for rid in self.admitted:
            if len(out) == max_batch:
                break
            r = self.reqs[rid]
            if r.state != "running":
                continue
            if r.len % self.page_size == 0:
                for layer in r.pages:
                    layer.append(self._take_page())
            r.len += 1
            r.generated += 1
            out.append((r.id, r.len, self._table(r)))
            self._finish_by_budget(r)
        self.stats["largest_decode_batch"] = max(self.stats["largest_decode_batch"], len(out))
        return out

    def finish(self, rid):
        r = self.reqs.get(rid)
        if r is None or r.state == "finished":
            return False
        if r.state == "waiting":
            self.queue.remove(rid)
        else:
            self.release_next.append(rid)
        r.state = "finished"
        self.stats["finished"] += 1
        return True
