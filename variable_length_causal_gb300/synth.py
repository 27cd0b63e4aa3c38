"""Seeded synthetic workloads and slot/pair accounting for isolated sequence packing.

This module holds no attention, RoPE, position or label arithmetic: it draws
segment lengths, packs them, draws bf16 tensors, and counts tokens, slots and
legal causal pairs.  Both the CUDA path's tests and the oracle's tests take
their inputs from here.

Workloads (lengths from ``numpy.random.default_rng(seed)``, seed = workload index;
tensors from ``torch.Generator().manual_seed(1000 + index)``, drawn in the order
q, k, v, dO as fp32 N(0, 1) and rounded to bf16):

  0 tiny  16 segments, lengths uniform in [1, 256], H=4, d=64
  1 sft   lognormal(median 300, sigma 1.0) clipped [16, 4096], first-fit-decreasing
          into 16 bins of 4096, tail pad of each bin as its own ignored segment, H=32, d=128
  2 pt    lognormal(median 400, sigma 0.8) clipped [32, 4096], FFD into 32 x 4096, H=32, d=128
  3 long  one 131072-token buffer: each doc is 128 with probability 0.1, else
          lognormal(median 2048, sigma 1.2) clipped [64, 32768]; docs are appended until one
          does not fit, which is truncated to fill the buffer (a remainder < 64 becomes an
          ignored pad segment), H=32, d=128
  4 pt+bwd  as 2 (seed 4), with dO for the backward pass

The first-fit-decreasing packer follows "Sequence Packing" (llm-compass),
section "Binning: how to pack" / "Implementation notes"; the pages' datasets
(Wikipedia, FLAN, OrcaMath) are not used -- these length laws stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

ROPE_THETA = 10000.0


@dataclasses.dataclass
class Workload:
    name: str
    index: int
    H: int
    d: int
    cu: np.ndarray            # int32 [nseg + 1]
    seg_ignore: np.ndarray    # uint8 [nseg], 1 = padding segment (excluded from metrics)
    theta: float = ROPE_THETA
    backward: bool = False
    description: str = ""

    @property
    def nseg(self) -> int:
        return len(self.cu) - 1

    @property
    def total(self) -> int:
        return int(self.cu[-1])

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.cu.astype(np.int64))

    @property
    def max_seqlen(self) -> int:
        return int(self.lengths.max())

    @property
    def real_lengths(self) -> np.ndarray:
        return self.lengths[self.seg_ignore == 0]


# ----------------------------------------------------------------------------- lengths

def _lognormal_len(rng: np.random.Generator, median: float, sigma: float, lo: int, hi: int) -> int:
    return int(min(hi, max(lo, round(rng.lognormal(math.log(median), sigma)))))


def first_fit_decreasing(lengths: Sequence[int], capacity: int) -> List[List[int]]:
    """Stable sort by length (descending), then put each item in the first bin with room.
    Returns bins as lists of lengths, bins in creation order, items in insertion order."""
    order = sorted(range(len(lengths)), key=lambda i: -int(lengths[i]))
    bins: List[List[int]] = []
    fill: List[int] = []
    for i in order:
        L = int(lengths[i])
        assert L <= capacity
        for b in range(len(bins)):
            if fill[b] + L <= capacity:
                bins[b].append(L)
                fill[b] += L
                break
        else:
            bins.append([L])
            fill.append(L)
    return bins


def _bins_to_cu(bins: List[List[int]], capacity: int):
    lens, ign = [], []
    for b in bins:
        lens.extend(b)
        ign.extend([0] * len(b))
        pad = capacity - sum(b)
        if pad > 0:
            lens.append(pad)
            ign.append(1)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cu, np.asarray(ign, np.uint8)


def _ffd_pack(rng, n_bins: int, capacity: int, median: float, sigma: float, lo: int, hi: int):
    docs: List[int] = []
    while sum(docs) < n_bins * capacity:
        docs.append(_lognormal_len(rng, median, sigma, lo, hi))
    bins = first_fit_decreasing(docs, capacity)[:n_bins]
    return _bins_to_cu(bins, capacity)


def _long_buffer(rng, capacity: int):
    lens, ign = [], []
    used = 0
    while used < capacity:
        if rng.random() < 0.1:
            L = 128
        else:
            L = _lognormal_len(rng, 2048.0, 1.2, 64, 32768)
        room = capacity - used
        if L <= room:
            lens.append(L)
            ign.append(0)
            used += L
            continue
        if room >= 64:
            lens.append(room)
            ign.append(0)
        else:
            lens.append(room)
            ign.append(1)
        used = capacity
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cu, np.asarray(ign, np.uint8)


WORKLOAD_NAMES = ["tiny", "sft", "pt", "long", "pt_bwd"]


def workload(index: int, bins: Optional[int] = None) -> Workload:
    """The five seeded workloads (see module docstring).  ``bins`` shrinks (or grows) a
    workload to that many 4096-token windows with the same length distribution (used for
    small profiling captures); the tiny workload ignores it."""
    rng = np.random.default_rng(index)
    if index == 0:
        lens = rng.integers(1, 257, size=16)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        return Workload("tiny", 0, 4, 64, cu, np.zeros(16, np.uint8),
                        description="16 segments, U[1,256], H=4, d=64, forward")
    if index == 1:
        cu, ign = _ffd_pack(rng, bins or 16, 4096, 300.0, 1.0, 16, 4096)
        return Workload("sft", 1, 32, 128, cu, ign,
                        description="SFT pack: lognormal(300,1.0) FFD into 16x4096, H=32, d=128")
    if index in (2, 4):
        cu, ign = _ffd_pack(rng, bins or 32, 4096, 400.0, 0.8, 32, 4096)
        return Workload("pt" if index == 2 else "pt_bwd", index, 32, 128, cu, ign,
                        backward=(index == 4),
                        description="pretraining windows: lognormal(400,0.8) FFD into 32x4096, "
                                    "H=32, d=128" + (", forward+backward" if index == 4 else ""))
    if index == 3:
        cu, ign = _long_buffer(rng, 4096 * (bins or 32))
        return Workload("long", 3, 32, 128, cu, ign,
                        description="long context: one 131072-token buffer, lognormal(2048,1.2) "
                                    "+10% at 128, H=32, d=128")
    raise ValueError(index)


def custom_workload(lengths: Sequence[int], H: int, d: int, seg_ignore=None, name="custom",
                    theta: float = ROPE_THETA) -> Workload:
    lens = np.asarray(lengths, np.int64)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ign = np.zeros(len(lens), np.uint8) if seg_ignore is None else np.asarray(seg_ignore, np.uint8)
    return Workload(name, -1, H, d, cu, ign, theta=theta)


def random_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n)


# ----------------------------------------------------------------------------- tensors

def make_tensors(w: Workload, device="cpu", seed: Optional[int] = None, with_grad: bool = False):
    """bf16 q, k, v (and dO) of shape [total, H, d], N(0,1) rounded to bf16."""
    import torch

    seed = (1000 + max(w.index, 0)) if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    shape = (w.total, w.H, w.d)
    out = []
    for _ in range(4 if with_grad else 3):
        out.append(torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16))
    return tuple(out)


def make_tokens(w: Workload, seed: Optional[int] = None, vocab: int = 32000) -> np.ndarray:
    rng = np.random.default_rng((2000 + max(w.index, 0)) if seed is None else seed)
    t = rng.integers(1, vocab, size=w.total, dtype=np.int64)
    starts = w.cu[:-1][w.seg_ignore == 1]
    ends = w.cu[1:][w.seg_ignore == 1]
    for a, b in zip(starts, ends):
        t[a:b] = 0   # pad token id 0
    return t


# ----------------------------------------------------------------------------- accounting
# "Fewer empty slots and less attention work are two separate ledgers"
# (charlestar, sequence packing and variable-length attention): token slots
# B*Lmax vs T, dense score slots B*Lmax^2 vs sum L_r^2 vs T^2, legal causal pairs.

def causal_pairs(lengths) -> int:
    """Legal in-segment causal (query, key) pairs, diagonal included: sum L(L+1)/2."""
    L = np.asarray(lengths, np.int64)
    return int(np.sum(L * (L + 1) // 2))


def score_slots_per_segment(lengths) -> int:
    L = np.asarray(lengths, np.int64)
    return int(np.sum(L * L))


def score_slots_padded(lengths) -> int:
    L = np.asarray(lengths, np.int64)
    return int(len(L) * L.max() ** 2)


def score_slots_whole(lengths) -> int:
    return int(np.sum(np.asarray(lengths, np.int64))) ** 2


def token_slots_padded(lengths, L: Optional[int] = None) -> int:
    lens = np.asarray(lengths, np.int64)
    return int(len(lens) * (lens.max() if L is None else L))


def padding_waste(lengths, L: int) -> float:
    """waste = 1 - mean(l) / L (vllbc, "Long-context training: remove padding")."""
    lens = np.asarray(lengths, np.float64)
    return 1.0 - lens.mean() / L


def slot_efficiency(lengths, B: int, Lmax: int) -> float:
    """eta = sum L_i / (B * Lmax) (llm-compass, "Sequence Packing", intuition section)."""
    return float(np.sum(np.asarray(lengths, np.int64))) / (B * Lmax)


def batch_slots(lengths, batch: int) -> int:
    """Token slots when consecutive groups of ``batch`` samples are padded to their group max."""
    lens = list(np.asarray(lengths, np.int64))
    return int(sum(len(lens[i:i + batch]) * max(lens[i:i + batch]) for i in range(0, len(lens), batch)))


def batch_score_slots(lengths, batch: int) -> int:
    lens = list(np.asarray(lengths, np.int64))
    return int(sum(len(lens[i:i + batch]) * max(lens[i:i + batch]) ** 2
                   for i in range(0, len(lens), batch)))


def pack_ledger(lengths, L: int) -> dict:
    """Slot ledger of Table 4-1 (vllbc): fixed-length padding vs ideal packing lower bound."""
    lens = np.asarray(lengths, np.int64)
    T = int(lens.sum())
    fixed = len(lens) * L
    packs = -(-T // L)
    packed = packs * L
    return {
        "T": T, "fixed": fixed, "padding": fixed - T, "waste": (fixed - T) / fixed,
        "packs": packs, "packed": packed, "pack_padding": packed - T,
        "pack_waste": (packed - T) / packed, "saved": fixed - packed,
        "saved_frac": (fixed - packed) / fixed,
        "score_fixed_half": len(lens) * L * L // 2, "score_packed_half": int(np.sum(lens * lens)) // 2,
    }


def fwd_flops(w: Workload) -> float:
    """Effective forward FLOPs: QK^T and PV over legal in-segment pairs of real segments,
    2*d each, per head: 4 * d * H * pairs."""
    return 4.0 * w.d * w.H * causal_pairs(w.real_lengths)


def bwd_flops(w: Workload) -> float:
    """Effective backward FLOPs: S recompute, dP, dV, dK, dQ contractions: 10 * d * H * pairs."""
    return 10.0 * w.d * w.H * causal_pairs(w.real_lengths)


def tile_efficiency(w: Workload, BM: int = 128, BN: int = 128) -> float:
    """Legal pairs over the pairs covered by the issued BM x BN tiles (segment-local tiling)."""
    issued = 0
    for L in w.lengths:
        nq = -(-int(L) // BM)
        for t in range(nq):
            last = min(L, (t + 1) * BM)
            issued += BM * BN * (-(-last // BN))
    return causal_pairs(w.lengths) / issued


def assign_packs(pack_costs: Sequence[float], world: int) -> List[List[int]]:
    """Greedy longest-processing-time assignment of packs to ranks by attention cost
    (sum of L_r^2 per pack, not token count: "two separate ledgers" section, charlestar)."""
    order = sorted(range(len(pack_costs)), key=lambda i: -pack_costs[i])
    load = [0.0] * world
    out: List[List[int]] = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda j: (load[j], j))
        out[r].append(i)
        load[r] += pack_costs[i]
    return [sorted(x) for x in out]
