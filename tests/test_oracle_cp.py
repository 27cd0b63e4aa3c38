"""Pins of the context-parallel oracle (oracle/cp.py) against what the pages and the
mathematics fix, independent of the oracle's own formulas:

* the split needs every segment length to be a multiple of 2 * cp ("Long-context
  training: remove padding", vllbc, failure-modes section) and keeps segment boundaries:
  over the ranks every row of the pack appears exactly once, inside its own segment;
* the zigzag chunks balance the attention work ("Sequence packing and variable-length
  attention", charlestar: balance by sum of L^2, not by tokens): every rank's legal causal
  pairs are the same, counted by brute force over its rows;
* block attention over all keys equals the already pinned oracle's segment-local causal
  forward (oracle.attn_fwd in exact mode) on the same rows, and merging it over any
  partition of the keys reproduces it; two identical partial results merge into the same O
  with LSE + ln 2 (the union of two copies of a key set doubles the sum);
* the block backward over all keys equals the pinned oracle.attn_bwd (exact mode), and its
  blocks over a partition of the keys add up to it.
"""
import numpy as np
import pytest

import oracle
from oracle import cp as ocp


@pytest.mark.parametrize("cp", [1, 2, 3, 4])
def test_partition_covers_every_row_once_inside_its_segment(cp):
    lengths = [2 * cp * m for m in (1, 5, 2, 9)]
    starts = np.concatenate([[0], np.cumsum(lengths)])
    seen = np.zeros(starts[-1], np.int64)
    for rank in range(cp):
        rows, pos, m = ocp.partition(lengths, cp, rank)
        assert len(rows) == starts[-1] // cp
        seen[rows] += 1
        seg = np.searchsorted(starts, rows, side="right") - 1
        assert np.array_equal(pos, rows - starts[seg])
        assert np.array_equal(m, np.array(lengths) // (2 * cp))
        # chunk `rank` of every segment first, then chunk 2 cp - 1 - rank
        half = len(rows) // 2
        assert np.all(pos[:half] // np.repeat(m, m) == rank)
        assert np.all(pos[half:] // np.repeat(m, m) == 2 * cp - 1 - rank)
    assert np.all(seen == 1)


def test_partition_rejects_lengths_not_multiple_of_2cp():
    with pytest.raises(ValueError):
        ocp.partition([8, 6], 2, 0)      # 6 % 4 != 0
    ocp.partition([8, 12], 2, 1)


@pytest.mark.parametrize("cp", [2, 3, 4])
def test_zigzag_balances_causal_pairs(cp):
    lengths = [2 * cp * m for m in (3, 7, 1, 4)]
    per_rank = []
    for rank in range(cp):
        rows, pos, _ = ocp.partition(lengths, cp, rank)
        per_rank.append(int(np.sum(pos + 1)))          # query at position p sees p + 1 keys
    assert len(set(per_rank)) == 1
    assert sum(per_rank) == sum(L * (L + 1) // 2 for L in lengths)


def _rand(n, H, d, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((n, H, d))


def test_block_attention_over_all_keys_is_the_pinned_forward():
    lengths = [24, 8, 40]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, H, d = int(cu[-1]), 2, 16
    q, k, v = _rand(T, H, d, 1), _rand(T, H, d, 2), _rand(T, H, d, 3)
    seg = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.arange(T) - cu[seg]
    o, lse = ocp.block_attention(q, k, v, seg, pos, seg, pos, 1.0 / np.sqrt(d))
    o_ref, lse_ref = oracle.attn_fwd_f64(q, k, v, cu, theta=0.0)
    assert np.abs(o - o_ref).max() < 1e-12
    assert np.abs(lse - lse_ref).max() < 1e-12


def test_merge_over_a_key_partition_reproduces_the_whole():
    lengths = [32, 16]
    cp = 2
    T, H, d = sum(lengths), 2, 8
    q, k, v = _rand(T, H, d, 4), _rand(T, H, d, 5), _rand(T, H, d, 6)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    seg = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.arange(T) - starts[seg]
    scale = 0.3
    rows, rpos, _ = ocp.partition(lengths, cp, 1)
    o_all, lse_all = ocp.block_attention(q[rows], k, v, seg[rows], rpos, seg, pos, scale)
    # keys split by the ranks' chunks (the ring's blocks), plus an empty block
    parts_o, parts_l = [], []
    for rank in range(cp):
        kr, kp, _ = ocp.partition(lengths, cp, rank)
        o_p, l_p = ocp.block_attention(q[rows], k[kr], v[kr], seg[rows], rpos, seg[kr], kp, scale)
        parts_o.append(o_p)
        parts_l.append(l_p)
    empty_o, empty_l = ocp.block_attention(q[rows], k[:0], v[:0], seg[rows], rpos, seg[:0], pos[:0], scale)
    assert np.all(np.isneginf(empty_l))
    o_m, l_m = ocp.lse_merge(parts_o + [empty_o], parts_l + [empty_l])
    assert np.abs(o_m - o_all).max() < 1e-12
    assert np.abs(l_m - lse_all).max() < 1e-12


def test_merge_of_two_copies_adds_ln2():
    o = _rand(5, 3, 4, 7)
    lse = np.random.default_rng(8).standard_normal((3, 5))
    o_m, l_m = ocp.lse_merge([o, o], [lse, lse])
    assert np.abs(o_m - o).max() < 1e-12
    assert np.abs(l_m - (lse + np.log(2.0))).max() < 1e-12


def test_block_backward_over_a_key_partition_adds_up_to_the_pinned_backward():
    lengths = [24, 16, 40]
    cp = 2
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, H, d = int(cu[-1]), 2, 8
    q, k, v, g = (_rand(T, H, d, 10 + i) for i in range(4))
    seg = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.arange(T) - cu[seg]
    scale = 1.0 / np.sqrt(d)
    o, lse = ocp.block_attention(q, k, v, seg, pos, seg, pos, scale)
    delta = np.einsum("nhd,nhd->hn", g, o)
    ref = oracle.attn_bwd_f64(g, q, k, v, cu, theta=0.0)
    whole = ocp.block_attention_backward(q, k, v, g, seg, pos, seg, pos, lse, delta, scale)
    for a, b in zip(whole, ref):
        assert np.abs(a - b).max() < 1e-10
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for rank in range(cp):
        kr, kp, _ = ocp.partition(lengths, cp, rank)
        bq, bk, bv = ocp.block_attention_backward(q, k[kr], v[kr], g, seg, pos, seg[kr], kp, lse, delta, scale)
        dq += bq
        dk[kr] += bk
        dv[kr] += bv
    for a, b in zip((dq, dk, dv), ref):
        assert np.abs(a - b).max() < 1e-10
