"""Oracle for KV-load-aware request placement on data-parallel attention ranks.

TEST INFRASTRUCTURE ONLY: used by ``tests/`` alone; the product library never
imports it, and it imports nothing from the product package.

Under DP attention each rank decodes its own requests and the MoE all-to-all
after attention keeps the ranks in lockstep, so the step lasts as long as the
rank with the most cache to read; long-context requests must be spread over
the ranks [dp-attention-expert-parallel-mla-kv-replication
(inferenceinterviews.com), "What it costs" and "What interviewers probe
next"].  The pages name the goal, not a method.  The reading taken here is the
plainest one: a rank's load is the cached tokens of its requests (a decode
reads every one of them), and requests are placed by list scheduling in
decreasing order (Graham 1969): longest first, each onto the least loaded
rank, ties to the lower request index and the lower rank; with a per-rank
capacity a request the least loaded rank cannot hold fits nowhere and is left
out (-1).

``place`` follows those steps with plain loops.  ``optimal_max_load`` is the
exhaustive optimum for tiny inputs, which pins ``place`` through Graham's
bound: its largest load is at most (4/3 - 1/(3m)) of the optimum on m ranks.
"""
from __future__ import annotations

import itertools


def place(kv_tokens, ranks, capacity_tokens=0):
    """Returns (rank_of, rank_load) as Python lists."""
    n = len(kv_tokens)
    order = sorted(range(n), key=lambda i: (-kv_tokens[i], i))
    load = [0] * ranks
    rank_of = [-1] * n
    for i in order:
        least = 0
        for r in range(1, ranks):
            if load[r] < load[least]:
                least = r
        if capacity_tokens and load[least] + kv_tokens[i] > capacity_tokens:
            continue
        rank_of[i] = least
        load[least] += kv_tokens[i]
    return rank_of, load


def place_one(rank_load, kv_tokens, capacity_tokens=0):
    """The rank a new request goes to given the current loads, or -1."""
    least = 0
    for r in range(1, len(rank_load)):
        if rank_load[r] < rank_load[least]:
            least = r
    if capacity_tokens and rank_load[least] + kv_tokens > capacity_tokens:
        return -1
    return least


def optimal_max_load(kv_tokens, ranks):
    """The smallest possible largest load, by trying every assignment
    (ranks ** n of them: tiny inputs only)."""
    best = None
    for assign in itertools.product(range(ranks), repeat=len(kv_tokens)):
        load = [0] * ranks
        for i, r in enumerate(assign):
            load[r] += kv_tokens[i]
        m = max(load)
        if best is None or m < best:
            best = m
    return best if best is not None else 0
