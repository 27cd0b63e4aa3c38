"""Context-parallel split oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests may import this module.  Plain, slow restatements (fp64, numpy), sharing
no code with the CUDA path:

* ``partition``: the split of a packed buffer over ``cp`` context-parallel ranks.
  "Long-context training: remove padding" (vllbc), failure-modes section: with context
  parallelism the sequence length must be a multiple of 2 * context_parallel_size,
  because of how CP slices the sequence.  "Sequence packing and variable-length
  attention" (charlestar), section on the two ledgers: shards and communication must
  follow the global segment boundaries, and ranks should be balanced by attention work
  (sum of L_r^2), not by token count.  Reading taken (the pages name the rule, not the
  layout): every segment is cut into 2 * cp chunks of m = L / (2 cp) tokens and rank i
  holds chunks i and 2 cp - 1 - i of every segment, so each rank's causal work inside
  each segment is the same, (2 cp - 1) m^2 + m (m + 1).  The rank's buffer holds first
  chunk i of every segment (segment order), then chunk 2 cp - 1 - i of every segment.
* ``block_attention``: the attention of a set of query rows against a set of key rows of
  the same pack, each row carrying its segment and its position inside the segment; key
  j is visible to query i when both lie in the same segment and pos_j <= pos_i (the
  block-diagonal causal rule of "Sequence packing and variable-length attention",
  section "EOS is content; isolation happens before softmax", written with the global
  positions that survive the split).  Rows that see no key get O = 0, LSE = -inf.
* ``lse_merge``: results over disjoint key sets combined into the result over their
  union: with LSE_k = ln sum_{j in K_k} e^{s_j}, the union has LSE = ln sum_k e^{LSE_k}
  and O = sum_k e^{LSE_k - LSE} O_k (each O_k is a softmax-weighted mean over K_k).
* ``block_attention_backward``: the standard softmax-attention derivatives restricted to
  one block of keys, given the whole attention's LSE and D = rowsum(dO * O):
  P = e^{S - LSE} on the block's visible entries, dV = P^T dO, dP = dO V^T,
  dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.  Every entry of the full
  P, dS lies in exactly one block, so the blocks' dQ add up to the full dQ and each key
  row's dK, dV come whole from the blocks that contain it.
"""
from __future__ import annotations

import numpy as np


def partition(lengths, cp: int, rank: int):
    """Rows of the pack held by ``rank`` (chunk ``rank`` of every segment, then chunk
    2 cp - 1 - rank of every segment), their positions inside their segments, and the
    chunk length m_r of every segment.  Raises ValueError if a segment length is not a
    multiple of 2 cp."""
    lengths = [int(x) for x in lengths]
    if cp < 1 or not 0 <= rank < cp:
        raise ValueError("need cp >= 1 and 0 <= rank < cp")
    for r, L in enumerate(lengths):
        if L % (2 * cp) != 0:
            raise ValueError(f"segment {r} has length {L}, not a multiple of 2 * cp = {2 * cp}")
    rows, pos = [], []
    starts = np.concatenate([[0], np.cumsum(lengths)])
    chunk_len = [L // (2 * cp) for L in lengths]
    for c in (rank, 2 * cp - 1 - rank):
        for r, L in enumerate(lengths):
            m = chunk_len[r]
            for p in range(c * m, (c + 1) * m):
                rows.append(int(starts[r]) + p)
                pos.append(p)
    return np.array(rows, np.int64), np.array(pos, np.int64), np.array(chunk_len, np.int64)


def block_attention(q, k, v, q_seg, q_pos, k_seg, k_pos, scale: float):
    """q [n, H, d], k/v [m, H, d] in fp64 (already rotated); returns O [n, H, d] and
    LSE [H, n] over the visible keys (same segment, key position <= query position)."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    n, H, d = q.shape
    allow = (np.asarray(k_seg)[None, :] == np.asarray(q_seg)[:, None]) & \
            (np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None])
    o = np.zeros((n, H, d))
    lse = np.full((H, n), -np.inf)
    for h in range(H):
        s = q[:, h, :] @ k[:, h, :].T * scale
        s = np.where(allow, s, -np.inf)
        for i in range(n):
            if not allow[i].any():
                continue
            mx = s[i].max()
            e = np.exp(s[i] - mx)
            tot = e.sum()
            o[i, h] = e @ v[:, h, :] / tot
            lse[h, i] = mx + np.log(tot)
    return o, lse


def lse_merge(o_parts, lse_parts):
    """Merge results over disjoint key sets: o_parts [n, H, d] each, lse_parts [H, n] each."""
    lse = np.stack([np.asarray(x, np.float64) for x in lse_parts])          # [k, H, n]
    o = np.stack([np.asarray(x, np.float64) for x in o_parts])              # [k, n, H, d]
    mx = lse.max(axis=0)                                                    # [H, n]
    safe = np.where(np.isfinite(mx), mx, 0.0)
    w = np.where(np.isfinite(lse), np.exp(lse - safe[None]), 0.0)           # [k, H, n]
    tot = w.sum(axis=0)
    out_lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    wn = np.where(tot[None] > 0, w / np.where(tot > 0, tot, 1.0)[None], 0.0)  # [k, H, n]
    out_o = np.einsum("khn,knhd->nhd", wn, o)
    return out_o, out_lse


def block_attention_backward(q, k, v, g, q_seg, q_pos, k_seg, k_pos, lse, delta, scale: float):
    """q, g [n, H, d], k, v [m, H, d] (fp64, rotated), lse / delta [H, n] of the whole attention;
    returns the block's (dq [n, H, d], dk [m, H, d], dv [m, H, d])."""
    q, k, v, g = (np.asarray(x, np.float64) for x in (q, k, v, g))
    n, H, d = q.shape
    allow = (np.asarray(k_seg)[None, :] == np.asarray(q_seg)[:, None]) & \
            (np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None])
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for h in range(H):
        s = q[:, h, :] @ k[:, h, :].T * scale
        fin = np.isfinite(lse[h])[:, None]
        p = np.where(allow & fin, np.exp(np.where(allow, s, 0.0) - np.where(fin, lse[h][:, None], 0.0)), 0.0)
        dp = g[:, h, :] @ v[:, h, :].T
        ds = p * (dp - delta[h][:, None])
        dv[:, h, :] = p.T @ g[:, h, :]
        dq[:, h, :] = scale * ds @ k[:, h, :]
        dk[:, h, :] = scale * ds.T @ q[:, h, :]
    return dq, dk, dv
