"""Host packing oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module.  Plain, slow restatements of the data step in front of the attention
path, each citing the page it follows:

* ``ffd`` / ``first_fit`` / ``next_fit``: bin packing of sample lengths into windows of
  ``capacity`` tokens.  "Sequence Packing" (llm-compass), section "Methods and formulas /
  binning": naive streaming (open a new window when the sample does not fit) and first-fit
  decreasing (sort by length, longest first, then put each sample into the first window that
  still has room).  "Packing document boundary" (operatorworld), practical checklist: FFD
  with a small per-document reserve for BOS/EOS (``extra`` tokens added to every sample).
  Megatron's dp_balanced scheduler, as "Long-context training: remove padding" (vllbc)
  describes it, is first-fit in the original order (``first_fit``).  A sample longer than
  the window is not truncated (the same page: over-long samples are only reported); it gets
  a window of its own, and such windows are counted.
* ``eta``: the effective-token share sum(L_i) / (B * L_max) ("Sequence Packing", the
  waste metric), which is also the nominal/effective ratio the operatorworld checklist
  asks to monitor (effective document tokens over windows x window length).
* ``lpt``: assignment of packs to ranks by their attention work.  "Sequence packing and
  variable-length attention" (charlestar), section on cross-rank balance: equal token
  counts can hide unequal sum(L_r^2), so balance sum(L_r^2).  The rule written out here is
  the longest-processing-time greedy: packs by cost, largest first, each to the rank with
  the smallest load so far (lowest rank on ties).
* ``brute_min_bins`` / ``brute_min_makespan``: exhaustive optima on tiny inputs, used only
  to pin the heuristics above to something other than themselves.

Ties are broken by the smaller sample (or pack) index everywhere, so every result is unique.
"""
from __future__ import annotations

import itertools

import numpy as np


def _eff(lengths, extra):
    return [int(x) + int(extra) for x in lengths]


def _place(order, sizes, capacity, first_fit=True):
    """Put samples in ``order`` into windows; returns (bin_of, bins as lists in placement order)."""
    bins, room, bin_of = [], [], [None] * len(sizes)
    for i in order:
        s = sizes[i]
        target = None
        if s <= capacity:
            cand = range(len(bins)) if first_fit else ([len(bins) - 1] if bins else [])
            for b in cand:
                if room[b] >= s:
                    target = b
                    break
        if target is None:               # a new window (a sample longer than it fills it alone)
            bins.append([])
            room.append(capacity - s if s <= capacity else 0)
            target = len(bins) - 1
        else:
            room[target] -= s
        bins[target].append(i)
        bin_of[i] = target
    return np.asarray(bin_of, np.int32), bins


def _result(bins, bin_of):
    order = np.asarray([i for b in bins for i in b], np.int64)
    bin_start = np.concatenate([[0], np.cumsum([len(b) for b in bins])]).astype(np.int64)
    return bin_of, order, bin_start


def ffd(lengths, capacity: int, extra: int = 0):
    """First-fit decreasing.  Returns (bin_of [n], order [n], bin_start [nbins+1]): samples
    grouped by window, each window's samples in placement order (longest first)."""
    sizes = _eff(lengths, extra)
    order = sorted(range(len(sizes)), key=lambda i: (-sizes[i], i))
    bin_of, bins = _place(order, sizes, capacity, True)
    return _result(bins, bin_of)


def first_fit(lengths, capacity: int, extra: int = 0):
    """First-fit in the given order (no sort)."""
    sizes = _eff(lengths, extra)
    bin_of, bins = _place(range(len(sizes)), sizes, capacity, True)
    return _result(bins, bin_of)


def next_fit(lengths, capacity: int, extra: int = 0):
    """Naive streaming: append to the current window, open a new one when the sample does not fit."""
    sizes = _eff(lengths, extra)
    bin_of, bins = _place(range(len(sizes)), sizes, capacity, False)
    return _result(bins, bin_of)


def oversize_count(lengths, capacity: int, extra: int = 0) -> int:
    return int(sum(1 for s in _eff(lengths, extra) if s > capacity))


def eta(lengths, nbins: int, capacity: int) -> float:
    """Effective share of the window slots: sum(L_i) / (nbins * capacity)."""
    return float(np.sum(np.asarray(lengths, np.int64))) / float(nbins * capacity)


def pack_costs(lengths, order, bin_start, kind: str = "sumsq"):
    """Per window: its token count (kind='tokens') or the sum of squared lengths ('sumsq')."""
    L = np.asarray(lengths, np.int64)
    out = []
    for b in range(len(bin_start) - 1):
        members = L[order[bin_start[b]:bin_start[b + 1]]]
        out.append(int(members.sum()) if kind == "tokens" else int((members * members).sum()))
    return np.asarray(out, np.int64)


def lpt(costs, ranks: int):
    """Longest-processing-time greedy.  Returns (rank_of [nbins], load [ranks])."""
    costs = [int(c) for c in costs]
    load = [0] * ranks
    rank_of = [0] * len(costs)
    for b in sorted(range(len(costs)), key=lambda i: (-costs[i], i)):
        r = min(range(ranks), key=lambda k: (load[k], k))
        rank_of[b] = r
        load[r] += costs[b]
    return np.asarray(rank_of, np.int32), np.asarray(load, np.int64)


def brute_min_bins(lengths, capacity: int) -> int:
    """Fewest windows that hold all samples (every sample <= capacity), by exhaustive search
    over assignments of samples to window labels (tiny n only)."""
    n = len(lengths)
    best = n
    for labels in itertools.product(range(n), repeat=n):
        if labels[0] != 0:
            continue
        used = max(labels) + 1
        if used >= best:
            continue
        fill = [0] * used
        for s, b in zip(lengths, labels):
            fill[b] += s
        if max(fill) <= capacity:
            best = used
    return best


def brute_min_makespan(costs, ranks: int) -> int:
    """Smallest achievable maximum rank load (tiny inputs only)."""
    best = None
    for labels in itertools.product(range(ranks), repeat=len(costs)):
        load = [0] * ranks
        for c, r in zip(costs, labels):
            load[r] += c
        m = max(load)
        best = m if best is None else min(best, m)
    return int(best)
