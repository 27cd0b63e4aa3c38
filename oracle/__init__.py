"""fp64 CPU oracle for isolated sequence packing -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does; the two
share no code.  ``oracle.c`` holds the segment-by-segment fp64 definitions
(cu_seqlens validation, positions, labels, work lists, RoPE, attention forward
and backward); ``brute.py`` is an independent whole-pack numpy restatement used
to pin it.  Every function cites the page and section it follows in its C
source.

Pins (see tests/test_oracle_pins.py): the pages' nine-token example, the
pre-shifted label example, the 10-versus-3.25 contamination counterexample,
closed forms at Q = 0, packed == per-sample, change-A-keeps-B, brute force
(numpy, full T x T mask), torch CPU fp64 SDPA with a boolean block mask, RoPE
shift invariance and closed-form angles, finite differences for the backward
pass, and for the shifted cross-entropy: uniform-logit closed form, the pages'
token-mean 2.5 versus sample-mean 2 example, torch's fp64 cross_entropy, and
pre-shifted labels == the internal-shift formulation; the interleaved RoPE pairing by its
complex-multiplication form and torch autograd; grouped key/value heads by torch SDPA with
enable_gqa; padded layouts (cu_padded) by a masked attention written directly on the padded
rows.  No oracle function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_CU_FIRST, ERR_CU_ORDER, ERR_CU_TOTAL, ERR_MAXLEN, ERR_ARG = 1, 2, 4, 8, 16


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (-O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.orc_validate_cu.argtypes = [P, i32, i32, i32]
            lib.orc_validate_cu.restype = ctypes.c_int
            lib.orc_positions_labels.argtypes = [P, i32, P, P, P, P]
            lib.orc_positions_labels.restype = None
            for f in (lib.orc_worklist_fwd, lib.orc_worklist_bwd):
                f.argtypes = [P, i32, i32, i32, P, i64]
                f.restype = i64
            lib.orc_rope_rows.argtypes = [P, P, i64, i32, f64, ctypes.c_int, P]
            lib.orc_rope_rows.restype = None
            lib.orc_attn_fwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, f64, ctypes.c_int,
                                         P, P]
            lib.orc_attn_fwd.restype = None
            lib.orc_attn_fwd_rows.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, f64,
                                              ctypes.c_int, P, P, i64, P, P]
            lib.orc_attn_fwd_rows.restype = None
            lib.orc_attn_fwd_seg_heads.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, f64,
                                                   ctypes.c_int, P, P, i64, P, P]
            lib.orc_attn_fwd_seg_heads.restype = None
            lib.orc_attn_bwd.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, f64,
                                         ctypes.c_int, P, P, P]
            lib.orc_attn_bwd.restype = None
            lib.orc_attn_bwd_seg_heads.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, f64,
                                                   ctypes.c_int, P, P, i64, P, P, P]
            lib.orc_attn_bwd_seg_heads.restype = None
            lib.orc_shifted_ce.argtypes = [P, ctypes.c_int, i32, i32, P, P, i32, P, P, P, P]
            lib.orc_shifted_ce.restype = ctypes.c_int
            lib.orc_num_threads.argtypes = []
            lib.orc_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def bf16_bits(x) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 torch tensor (or pass-through for uint16 arrays)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch

    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def validate_cu(cu, total: int, max_seqlen: int) -> int:
    cu = _c(cu, np.int32)
    return int(_load().orc_validate_cu(_ptr(cu), len(cu) - 1, int(total), int(max_seqlen)))


def positions_labels(cu, tokens, seg_ignore=None):
    cu = _c(cu, np.int32)
    tokens = _c(tokens, np.int64)
    nseg = len(cu) - 1
    total = int(cu[-1])
    assert tokens.shape[0] == total
    ign = _c(seg_ignore, np.uint8) if seg_ignore is not None else None
    pos = np.zeros(total, np.int32)
    lab = np.zeros(total, np.int64)
    _load().orc_positions_labels(_ptr(cu), nseg, _ptr(tokens), _ptr(ign), _ptr(pos), _ptr(lab))
    return pos, lab


def _worklist(fn, cu, BM, BN):
    cu = _c(cu, np.int32)
    nseg = len(cu) - 1
    lens = np.diff(cu.astype(np.int64))
    cap = int(np.sum((lens + min(BM, BN) - 1) // min(BM, BN))) + 1
    items = np.zeros((cap, 4), np.int32)
    n = fn(_ptr(cu), nseg, int(BM), int(BN), _ptr(items), cap)
    assert n >= 0
    return items[:n].copy()


def worklist_fwd(cu, BM: int = 128, BN: int = 128) -> np.ndarray:
    """Forward items [n, 4] = {seg, q_tile, kv_lo, kv_hi} (oracle.c: orc_worklist_fwd)."""
    return _worklist(_load().orc_worklist_fwd, cu, BM, BN)


def worklist_bwd(cu, BM: int = 128, BN: int = 128) -> np.ndarray:
    """Backward items [n, 4] = {seg, kv_tile, q_lo, q_hi} (oracle.c: orc_worklist_bwd)."""
    return _worklist(_load().orc_worklist_bwd, cu, BM, BN)


def rope_rows(x, pos, theta: float = 10000.0, interleaved: bool = False) -> np.ndarray:
    x = _c(x, np.float64)
    n, d = x.shape
    pos = _c(pos, np.int64)
    out = np.zeros_like(x)
    _load().orc_rope_rows(_ptr(x), _ptr(pos), n, d, float(theta), int(bool(interleaved)), _ptr(out))
    return out



def real_rows(cu, cu_padded) -> np.ndarray:
    """Row indices of the real tokens of a padded layout: segment r's L_r = cu[r+1] - cu[r]
    tokens sit at rows cu_padded[r] .. cu_padded[r] + L_r - 1 and the rest of its slot
    [cu_padded[r], cu_padded[r+1]) is padding ("Sequence packing and variable-length
    attention", charlestar: Megatron's PackedSeqParams carries padded q/kv offsets next to
    cu_seqlens, and TE's pad_between_seqs leaves padding between the samples).  Padding rows
    are not tokens: no query attends to them and they attend to nothing."""
    cu = np.asarray(cu, np.int64)
    cp = np.asarray(cu_padded, np.int64)
    L = np.diff(cu)
    if len(cp) != len(cu) or cp[0] != 0 or np.any(np.diff(cp) < L):
        raise ValueError("cu_padded must start at 0 and give every segment a slot >= its length")
    return np.concatenate([np.arange(p, p + n) for p, n in zip(cp[:-1], L)]).astype(np.int64)

def _mode(contract: bool, interleaved: bool) -> int:
    return int(bool(contract)) + (4 if interleaved else 0)


def _mode_f64(interleaved: bool) -> int:
    return -5 if interleaved else -1


def _kv_args(cu, cu_kv, total_kv):
    """cu_kv pointer and key/value row count for the C calls (None: self-attention)."""
    if cu_kv is None:
        return None, 0, None
    cu_kv = _c(cu_kv, np.int32)
    if len(cu_kv) != len(cu) or cu_kv[0] != 0 or np.any(np.diff(cu_kv) < np.diff(np.asarray(cu))):
        raise ValueError("cu_kv must start at 0 and give every segment at least as many keys as queries")
    if cu_kv[-1] != total_kv:
        raise ValueError("cu_kv must end at the number of key/value rows")
    return cu_kv, int(total_kv), _ptr(cu_kv)


def attn_fwd(q, k, v, cu, scale: float = 0.0, theta: float = 10000.0, contract: bool = True,
             seg_heads=None, interleaved: bool = False, cu_padded=None, cu_kv=None):
    """Exact per-segment causal attention in fp64.  q/k/v: bf16 tensors or uint16 bit arrays
    [total, H, d] (k and v may have fewer heads Hkv dividing H: query head h reads key/value
    head h // (H // Hkv)).  Returns (o [total, H, d] f64, lse [H, total] f64, natural log).
    With ``seg_heads`` (a list of (segment, head) pairs) only those are computed; the rest
    stay 0.  With ``cu_padded`` the rows follow the padded layout of ``real_rows``: the real
    rows are gathered, attended as a contiguous pack, and scattered back; padding rows get
    O = 0 and LSE = -inf (the log of an empty sum).  With ``cu_kv`` the keys and values
    ([total_kv, Hkv, d]) have segments of their own, at least as long as the query segments;
    queries are bottom-right aligned (query p of a segment with L queries and Lk keys sits at
    position p + Lk - L and sees keys 0 .. p + Lk - L)."""
    if cu_padded is not None:
        idx = real_rows(cu, cu_padded)
        qb, kb, vb = (bf16_bits(x)[idx] for x in (q, k, v))
        o_r, lse_r = attn_fwd(qb, kb, vb, cu, scale, theta, contract, seg_heads, interleaved)
        total, H, d = bf16_bits(q).shape
        o = np.zeros((total, H, d), np.float64)
        lse = np.full((H, total), -np.inf)
        o[idx], lse[:, idx] = o_r, lse_r
        return o, lse
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    total, H, d = qb.shape
    Hkv = kb.shape[1]
    cu = _c(cu, np.int32)
    cu_kv, total_kv, kvp = _kv_args(cu, cu_kv, kb.shape[0])
    o = np.zeros((total, H, d), np.float64)
    lse = np.zeros((H, total), np.float64)
    if seg_heads is None:
        _load().orc_attn_fwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), kvp, len(cu) - 1, total, total_kv, H,
                             Hkv, d, float(scale), float(theta), _mode(contract, interleaved), _ptr(o),
                             _ptr(lse))
    else:
        sh = np.asarray(seg_heads, np.int32).reshape(-1, 2)
        segs, heads = np.ascontiguousarray(sh[:, 0]), np.ascontiguousarray(sh[:, 1])
        _load().orc_attn_fwd_seg_heads(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), kvp, len(cu) - 1, total,
                                       total_kv, H, Hkv, d, float(scale), float(theta),
                                       _mode(contract, interleaved), _ptr(segs), _ptr(heads), sh.shape[0],
                                       _ptr(o), _ptr(lse))
    return o, lse


def attn_fwd_rows(q, k, v, cu, rows, heads, scale: float = 0.0, theta: float = 10000.0,
                  contract: bool = True, interleaved: bool = False, cu_kv=None):
    """Forward for selected (token row, head) pairs: returns (o [n, d], lse [n])."""
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    total, H, d = qb.shape
    Hkv = kb.shape[1]
    cu = _c(cu, np.int32)
    cu_kv, total_kv, kvp = _kv_args(cu, cu_kv, kb.shape[0])
    rows = _c(rows, np.int64)
    heads = _c(heads, np.int32)
    n = rows.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros(n, np.float64)
    _load().orc_attn_fwd_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), kvp, len(cu) - 1, total, total_kv,
                              H, Hkv, d, float(scale), float(theta), _mode(contract, interleaved),
                              _ptr(rows), _ptr(heads), n, _ptr(o), _ptr(lse))
    return o, lse


def attn_fwd_f64(q, k, v, cu, scale: float = 0.0, theta: float = 10000.0, interleaved: bool = False,
                 cu_kv=None):
    """Exact-mode forward on float64 inputs [total, H, d] (finite-difference tests)."""
    q, k, v = (_c(x, np.float64) for x in (q, k, v))
    total, H, d = q.shape
    Hkv = k.shape[1]
    cu = _c(cu, np.int32)
    cu_kv, total_kv, kvp = _kv_args(cu, cu_kv, k.shape[0])
    o = np.zeros((total, H, d), np.float64)
    lse = np.zeros((H, total), np.float64)
    _load().orc_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), kvp, len(cu) - 1, total, total_kv, H, Hkv,
                         d, float(scale), float(theta), _mode_f64(interleaved), _ptr(o), _ptr(lse))
    return o, lse


def attn_bwd_f64(dout, q, k, v, cu, scale: float = 0.0, theta: float = 10000.0, interleaved: bool = False,
                 cu_kv=None):
    """Exact-mode gradients on float64 inputs (finite-difference tests)."""
    g, q, k, v = (_c(x, np.float64) for x in (dout, q, k, v))
    total, H, d = q.shape
    Hkv = k.shape[1]
    cu = _c(cu, np.int32)
    cu_kv, total_kv, kvp = _kv_args(cu, cu_kv, k.shape[0])
    dq = np.zeros((total, H, d), np.float64)
    dk = np.zeros(k.shape, np.float64)
    dv = np.zeros_like(dk)
    _load().orc_attn_bwd(_ptr(g), _ptr(q), _ptr(k), _ptr(v), _ptr(cu), kvp, len(cu) - 1, total, total_kv,
                         H, Hkv, d, float(scale), float(theta), _mode_f64(interleaved), _ptr(dq), _ptr(dk),
                         _ptr(dv))
    return dq, dk, dv


def attn_bwd(dout, q, k, v, cu, scale: float = 0.0, theta: float = 10000.0, contract: bool = True,
             seg_heads=None, interleaved: bool = False, cu_padded=None, cu_kv=None):
    """Gradients (dq [total, H, d], dk and dv shaped like k and v) f64 of sum(O * dO).  With
    ``seg_heads`` (a list of (segment, key/value head) pairs) only those are computed (dq for
    every query head of each pair's group); other entries stay 0.  With ``cu_padded`` the
    padding rows (``real_rows``) take no part and their gradients are 0.  ``cu_kv`` as in
    ``attn_fwd``."""
    if cu_padded is not None:
        idx = real_rows(cu, cu_padded)
        gb, qb, kb, vb = (bf16_bits(x)[idx] for x in (dout, q, k, v))
        r = attn_bwd(gb, qb, kb, vb, cu, scale, theta, contract, seg_heads, interleaved)
        out = []
        for full, part in zip((q, k, v), r):
            z = np.zeros(bf16_bits(full).shape, np.float64)
            z[idx] = part
            out.append(z)
        return tuple(out)
    gb, qb, kb, vb = bf16_bits(dout), bf16_bits(q), bf16_bits(k), bf16_bits(v)
    total, H, d = qb.shape
    Hkv = kb.shape[1]
    cu = _c(cu, np.int32)
    cu_kv, total_kv, kvp = _kv_args(cu, cu_kv, kb.shape[0])
    dq = np.zeros((total, H, d), np.float64)
    dk = np.zeros(kb.shape, np.float64)
    dv = np.zeros_like(dk)
    lib = _load()
    if seg_heads is None:
        lib.orc_attn_bwd(_ptr(gb), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), kvp, len(cu) - 1, total,
                         total_kv, H, Hkv, d, float(scale), float(theta), _mode(contract, interleaved),
                         _ptr(dq), _ptr(dk), _ptr(dv))
    else:
        sh = np.asarray(seg_heads, np.int32).reshape(-1, 2)
        segs = np.ascontiguousarray(sh[:, 0])
        heads = np.ascontiguousarray(sh[:, 1])
        lib.orc_attn_bwd_seg_heads(_ptr(gb), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), kvp, len(cu) - 1,
                                   total, total_kv, H, Hkv, d, float(scale), float(theta),
                                   _mode(contract, interleaved), _ptr(segs), _ptr(heads), sh.shape[0],
                                   _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def shifted_ce(logits, labels, cu=None):
    """Shifted next-token cross-entropy statistics (charlestar: "After isolation one
    cross-boundary prediction pair remains"; "Packing should not decide how much a long
    sample weighs").  logits: [total, vocab] as bf16 bit patterns (uint16) or float64;
    labels: int64 [total], pre-shifted, -100 = ignored.  Returns (status, loss_sum,
    count, seg_loss [nseg], seg_count [nseg]); status 1 flags a label outside [0, vocab)."""
    lib = _load()
    z = np.ascontiguousarray(logits)
    is_f64 = 1 if z.dtype == np.float64 else 0
    if not is_f64 and z.dtype != np.uint16:
        raise TypeError("logits must be uint16 bf16 bits or float64")
    total, vocab = z.shape
    lab = _c(labels, np.int64)
    cuc = None if cu is None else _c(cu, np.int32)
    nseg = 1 if cu is None else len(cuc) - 1
    ls = np.zeros(1, np.float64)
    cnt = np.zeros(1, np.int64)
    sl = np.zeros(nseg, np.float64)
    sc = np.zeros(nseg, np.int64)
    st = lib.orc_shifted_ce(_ptr(z), is_f64, vocab, total, _ptr(lab), None if cuc is None else _ptr(cuc),
                            nseg, _ptr(ls), _ptr(cnt), _ptr(sl), _ptr(sc))
    return int(st), float(ls[0]), int(cnt[0]), sl, sc
