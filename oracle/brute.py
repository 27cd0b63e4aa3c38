"""Whole-pack brute force in numpy fp64 -- TEST INFRASTRUCTURE ONLY.

An independent restatement used to pin ``oracle.c`` on tiny inputs.  Where the
C oracle walks one segment at a time with a real-valued rotate-half rotation,
this file builds the full T x T additive mask M (0 where allowed, -inf
elsewhere) and takes

    O = softmax(Q' K'^T / sqrt(d) + M) V

over the whole packed buffer at once ("Sequence packing and variable-length
attention" (charlestar), section "EOS is content; isolation happens before
softmax": allow(i,j) = (s_i == s_j) and (p_j <= p_i), mask added before the
softmax).  Segment ids come from numpy's searchsorted, as the Megatron THD RoPE
path described on "Long-context training: remove padding" (vllbc) does.  RoPE
is written as a complex multiplication (x_j + i x_{j+d/2}) * exp(i p w_j) with
w_j = theta^(-2j/d) ("the pure-RoPE argument" section, RoFormer's rotation).
"""
from __future__ import annotations

import numpy as np


def segment_ids(cu: np.ndarray) -> np.ndarray:
    cu = np.asarray(cu, np.int64)
    t = np.arange(cu[-1])
    return np.searchsorted(cu, t, side="right") - 1


def local_positions(cu: np.ndarray) -> np.ndarray:
    cu = np.asarray(cu, np.int64)
    return np.arange(cu[-1]) - cu[segment_ids(cu)]


def block_causal_allow(cu: np.ndarray) -> np.ndarray:
    """Boolean [T, T] matrix, True where query i may attend to key j."""
    s = segment_ids(cu)
    p = local_positions(cu)
    return (s[:, None] == s[None, :]) & (p[None, :] <= p[:, None])


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 to the nearest bf16 value (ties to even) by integer arithmetic on the
    IEEE-754 binary64 bit pattern: keep 7 fraction bits, round the 45 dropped bits."""
    x = np.ascontiguousarray(x, np.float64)
    b = x.view(np.uint64)
    keep_lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + np.uint64((1 << 44) - 1) + keep_lsb) & ~np.uint64((1 << 45) - 1)
    out = r.view(np.float64)
    return np.where((x == 0) | ~np.isfinite(x), x, out)


def rope_complex(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """x [T, H, d] or [T, d]; rotate pair (j, j + d/2) by angle pos * theta^(-2j/d)."""
    d = x.shape[-1]
    half = d // 2
    w = theta ** (-2.0 * np.arange(half) / d)
    ang = np.asarray(pos, np.float64)[:, None] * w[None, :]
    rot = np.exp(1j * ang)
    if x.ndim == 3:
        rot = rot[:, None, :]
    z = (x[..., :half] + 1j * x[..., half:]) * rot
    return np.concatenate([z.real, z.imag], axis=-1)


def attention(q, k, v, cu, scale=None, theta=10000.0, contract=True, allow=None):
    """q, k, v float64 [T, H, d] (already bf16-valued).  Returns (o [T,H,d], lse [H,T]).
    ``allow`` overrides the block-causal mask (used for the whole-pack comparison)."""
    T, H, d = q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    if theta:
        pos = local_positions(cu)
        q = rope_complex(q, pos, theta)
        k = rope_complex(k, pos, theta)
        if contract:
            q, k = round_bf16(q), round_bf16(k)
    if allow is None:
        allow = block_causal_allow(cu)
    M = np.where(allow, 0.0, -np.inf)
    o = np.zeros((T, H, d))
    lse = np.zeros((H, T))
    for h in range(H):
        S = q[:, h, :] @ k[:, h, :].T * scale + M
        m = S.max(axis=1, keepdims=True)
        e = np.exp(S - m)
        z = e.sum(axis=1, keepdims=True)
        o[:, h, :] = (e / z) @ v[:, h, :]
        lse[h] = (m + np.log(z))[:, 0]
    return o, lse
