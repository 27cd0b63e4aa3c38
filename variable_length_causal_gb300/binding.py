"""Python binding of libvlc.so: argument marshalling only.

Every step of the path runs in the library's CUDA kernels; PyTorch supplies
device memory (outputs and workspace) and the current stream.  There is no
CPU or PyTorch fallback: if the library is missing or no CUDA device is
present, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import NamedTuple, Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libvlc.so")

VLC_OK, VLC_ERR_ARG, VLC_ERR_CU_SEQLENS, VLC_ERR_UNSUPPORTED = 0, 1, 2, 3
VLC_ERR_WORKSPACE, VLC_ERR_CUDA, VLC_ERR_TIMEOUT, VLC_ERR_LABEL = 4, 5, 6, 7
DEVERR_CU_FIRST, DEVERR_CU_ORDER, DEVERR_CU_TOTAL, DEVERR_MAXLEN = 0x1, 0x2, 0x4, 0x8
DEVERR_TIMEOUT = 0x100
DEVERR_LABEL, DEVERR_CU_PADDED, DEVERR_QKV = 0x10, 0x20, 0x40
WORKLIST_FWD, WORKLIST_BWD = 0, 1
PACK_MODES = {"ffd": 0, "first_fit": 1, "next_fit": 2}
COST_KINDS = {"tokens": 0, "sumsq": 1}
ROPE_INTERLEAVED = 0x1
QK_ROTATED = 0x2
KEYS_ALL_VISIBLE = 0x4
ROPE_TRANSPOSE = 0x8
DEVERR_POS = 0x80
CP_BLOCK_NONE, CP_BLOCK_CAUSAL, CP_BLOCK_ALL = 0, 1, 2
LSE_MERGE_MAX = 16

EXPORTED = [
    "vlc_status_string", "vlc_version", "vlc_workspace_bytes", "vlc_worklist_capacity",
    "vlc_build_positions_labels", "vlc_build_worklist", "vlc_attn_fwd", "vlc_attn_bwd",
    "vlc_get_error", "vlc_attn_fwd_noalloc", "vlc_ce_workspace_bytes", "vlc_shifted_ce",
    "vlc_workspace_bytes_gqa", "vlc_attn_fwd_gqa", "vlc_attn_bwd_gqa", "vlc_attn_fwd_ex",
    "vlc_attn_bwd_ex", "vlc_workspace_bytes_qkv", "vlc_attn_fwd_qkv", "vlc_attn_bwd_qkv", "vlc_pack",
    "vlc_shard_packs", "vlc_rope_qk", "vlc_set_wait_limit_us", "vlc_cp_partition", "vlc_cp_block_mode",
    "vlc_rope_pos_workspace_bytes", "vlc_rope_pos", "vlc_lse_merge", "vlc_sum_parts", "vlc_attn_fwd_rot",
]

_lock = threading.Lock()
_lib = None


class VlcError(RuntimeError):
    def __init__(self, status: int, where: str, bits: int = 0):
        self.status = status
        self.bits = bits
        msg = f"{where}: {load_library().vlc_status_string(status).decode()} (status {status}"
        msg += f", device bits 0x{bits:x})" if bits else ")"
        super().__init__(msg)


def load_library(path: str = LIB_PATH):
    """Load libvlc.so and declare its signatures (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`"
            )
        lib = ctypes.CDLL(path)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        f32, sz, cint = ctypes.c_float, ctypes.c_size_t, ctypes.c_int
        lib.vlc_status_string.argtypes = [cint]
        lib.vlc_status_string.restype = ctypes.c_char_p
        lib.vlc_version.argtypes = []
        lib.vlc_version.restype = cint
        lib.vlc_set_wait_limit_us.argtypes = [ctypes.c_uint32]
        lib.vlc_set_wait_limit_us.restype = None
        lib.vlc_cp_partition.argtypes = [P, i32, i32, i32, P, P, P, P]
        lib.vlc_cp_partition.restype = cint
        lib.vlc_cp_block_mode.argtypes = [i32, i32, i32, i32, i32]
        lib.vlc_cp_block_mode.restype = cint
        lib.vlc_rope_pos_workspace_bytes.argtypes = [i32, i32]
        lib.vlc_rope_pos_workspace_bytes.restype = sz
        lib.vlc_rope_pos.argtypes = [P, P, i32, i32, i32, i32, f32, ctypes.c_uint32, P, P, sz, P]
        lib.vlc_rope_pos.restype = cint
        lib.vlc_lse_merge.argtypes = [P, P, i32, i32, i32, i32, P, P, P]
        lib.vlc_lse_merge.restype = cint
        lib.vlc_sum_parts.argtypes = [P, i32, i64, P, P]
        lib.vlc_sum_parts.restype = cint
        lib.vlc_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, cint]
        lib.vlc_workspace_bytes.restype = sz
        lib.vlc_worklist_capacity.argtypes = [i32, i32, i32]
        lib.vlc_worklist_capacity.restype = i64
        lib.vlc_build_positions_labels.argtypes = [P, i32, P, i32, P, P, P, P, P]
        lib.vlc_build_positions_labels.restype = cint
        lib.vlc_build_worklist.argtypes = [P, i32, i32, i32, i32, i32, cint, P, i64, P, P, P, P]
        lib.vlc_build_worklist.restype = cint
        lib.vlc_attn_fwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f32, f32, P, P, P, sz, P]
        lib.vlc_attn_fwd.restype = cint
        lib.vlc_attn_bwd.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32, f32,
                                     P, P, P, P, sz, P]
        lib.vlc_attn_bwd.restype = cint
        lib.vlc_get_error.argtypes = [P, P, P]
        lib.vlc_get_error.restype = cint
        lib.vlc_attn_fwd_noalloc.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f32, f32, P, P, P, P]
        lib.vlc_attn_fwd_noalloc.restype = cint
        lib.vlc_ce_workspace_bytes.argtypes = [i32, i32]
        lib.vlc_ce_workspace_bytes.restype = sz
        lib.vlc_shifted_ce.argtypes = [P, i32, i32, P, P, i32, P, P, P, P, P, sz, P]
        lib.vlc_shifted_ce.restype = cint
        lib.vlc_workspace_bytes_gqa.argtypes = [i32, i32, i32, i32, i32, i32, cint]
        lib.vlc_workspace_bytes_gqa.restype = sz
        lib.vlc_attn_fwd_gqa.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32, P, P, P, sz, P]
        lib.vlc_attn_fwd_gqa.restype = cint
        lib.vlc_attn_bwd_gqa.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32,
                                         P, P, P, P, sz, P]
        lib.vlc_attn_bwd_gqa.restype = cint
        u32 = ctypes.c_uint32
        lib.vlc_attn_fwd_ex.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32, u32, P, P,
                                        P, sz, P]
        lib.vlc_attn_fwd_ex.restype = cint
        lib.vlc_attn_bwd_ex.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32,
                                        u32, P, P, P, P, sz, P]
        lib.vlc_attn_bwd_ex.restype = cint
        lib.vlc_workspace_bytes_qkv.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, cint]
        lib.vlc_workspace_bytes_qkv.restype = sz
        lib.vlc_attn_fwd_qkv.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, f32,
                                         u32, P, P, P, sz, P]
        lib.vlc_attn_fwd_qkv.restype = cint
        lib.vlc_attn_bwd_qkv.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                         f32, f32, u32, P, P, P, P, sz, P]
        lib.vlc_attn_bwd_qkv.restype = cint
        lib.vlc_rope_qk.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, f32, u32, P, P, P, sz, P]
        lib.vlc_rope_qk.restype = cint
        lib.vlc_attn_fwd_rot.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32, u32, P, P, P, P,
                                         P, sz, P]
        lib.vlc_attn_fwd_rot.restype = cint
        lib.vlc_pack.argtypes = [P, i64, i32, i32, cint, P, P, P, P, P]
        lib.vlc_pack.restype = cint
        lib.vlc_shard_packs.argtypes = [P, P, P, i64, i32, cint, P, P]
        lib.vlc_shard_packs.restype = cint
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status: int, where: str):
    if status != VLC_OK:
        raise VlcError(status, where)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (the library has no CPU path)")


def _cu_info(cu_seqlens: torch.Tensor, cu_padded: Optional[torch.Tensor] = None):
    for c in (cu_seqlens, cu_padded):
        if c is not None and (c.dtype != torch.int32 or c.dim() != 1 or not c.is_contiguous()):
            raise ValueError("cu_seqlens / cu_seqlens_padded must be contiguous 1-D int32 tensors")
    if cu_padded is not None and (cu_padded.numel() != cu_seqlens.numel() or
                                  cu_padded.device != cu_seqlens.device):
        raise ValueError("cu_seqlens_padded must match cu_seqlens in size and device")
    return cu_seqlens.numel() - 1


def workspace_bytes(nseg: int, total: int, H: int, d: int, max_seqlen: int, backward: bool,
                    H_kv: Optional[int] = None, total_kv: Optional[int] = None,
                    max_seqlen_kv: Optional[int] = None) -> int:
    """Workspace bytes for the forward (backward=False) or backward call; H_kv key/value heads
    (default H).  total_kv / max_seqlen_kv: key/value segments of their own (q != kv)."""
    lib = load_library()
    hk = H if H_kv is None else H_kv
    if total_kv is None:
        return int(lib.vlc_workspace_bytes_gqa(nseg, total, H, hk, d, max_seqlen, int(backward)))
    return int(lib.vlc_workspace_bytes_qkv(nseg, total, total_kv, H, hk, d, max_seqlen, max_seqlen_kv,
                                           int(backward)))


def new_workspace(nseg, total, H, d, max_seqlen, backward, device, H_kv=None, total_kv=None,
                  max_seqlen_kv=None) -> torch.Tensor:
    n = workspace_bytes(nseg, total, H, d, max_seqlen, backward, H_kv, total_kv, max_seqlen_kv)
    if n == 0:
        raise VlcError(VLC_ERR_UNSUPPORTED, "workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def set_wait_limit_us(us: int) -> None:
    """Limit of each bounded wait inside the attention kernels launched from now on, in
    microseconds (0: the default of 2 s).  Only for exercising the timeout path."""
    load_library().vlc_set_wait_limit_us(int(us))


def get_error(ws: torch.Tensor) -> Tuple[int, int]:
    """Synchronise the current stream and return (status, device error bits)."""
    bits = ctypes.c_int32(0)
    st = load_library().vlc_get_error(_ptr(ws), ctypes.byref(bits), _stream(ws.device))
    return int(st), int(bits.value)


def _raise_device_error(ws, where):
    st, bits = get_error(ws)
    if st != VLC_OK:
        raise VlcError(st, where, bits)


def build_positions_labels(cu_seqlens: torch.Tensor, tokens: torch.Tensor,
                           seg_ignore: Optional[torch.Tensor] = None,
                           err: Optional[torch.Tensor] = None,
                           out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None):
    """Per-segment positions (int32) and pre-shifted labels (int64, -100 at segment ends).
    ``out`` = (positions, labels) receives the result instead of new tensors."""
    lib = load_library()
    _require_cuda(cu_seqlens, tokens, seg_ignore, err)
    nseg = _cu_info(cu_seqlens)
    if tokens.dtype != torch.int64 or not tokens.is_contiguous():
        raise ValueError("tokens must be contiguous int64")
    total = tokens.numel()
    if seg_ignore is not None and (seg_ignore.dtype != torch.uint8 or seg_ignore.numel() != nseg):
        raise ValueError("seg_ignore must be uint8 with one entry per segment")
    if out is None:
        pos = torch.empty(total, dtype=torch.int32, device=tokens.device)
        lab = torch.empty(total, dtype=torch.int64, device=tokens.device)
    else:
        pos, lab = out
        if (pos.dtype != torch.int32 or lab.dtype != torch.int64 or pos.numel() != total
                or lab.numel() != total or not pos.is_contiguous() or not lab.is_contiguous()):
            raise ValueError("out must be contiguous (int32 positions, int64 labels) of one entry per token")
        _require_cuda(pos, lab)
    st = lib.vlc_build_positions_labels(_ptr(cu_seqlens), nseg, _ptr(tokens), total,
                                        _ptr(seg_ignore), _ptr(pos), _ptr(lab), _ptr(err),
                                        _stream(tokens.device))
    _check(st, "vlc_build_positions_labels")
    return pos, lab


def build_worklist(cu_seqlens: torch.Tensor, total: int, max_seqlen: int, kind: int = WORKLIST_FWD,
                   BM: int = 128, BN: int = 128):
    """Device work list: returns (items [n, 4] int32, seg_order [2*nseg+1] int32, err bits)."""
    lib = load_library()
    _require_cuda(cu_seqlens)
    nseg = _cu_info(cu_seqlens)
    tile = BM if kind == WORKLIST_FWD else BN
    cap = int(lib.vlc_worklist_capacity(nseg, total, tile))
    dev = cu_seqlens.device
    items = torch.zeros((max(cap, 1), 4), dtype=torch.int32, device=dev)
    order = torch.zeros(2 * nseg + 1, dtype=torch.int32, device=dev)
    meta = torch.zeros(2, dtype=torch.int32, device=dev)    # count, err
    st = lib.vlc_build_worklist(_ptr(cu_seqlens), nseg, total, max_seqlen, BM, BN, kind, _ptr(items),
                                cap, _ptr(order), ctypes.c_void_p(meta.data_ptr()),
                                ctypes.c_void_p(meta.data_ptr() + 4), _stream(dev))
    _check(st, "vlc_build_worklist")
    count, bits = (int(x) for x in meta.cpu())
    return items[:count], order, bits


def _scale(softmax_scale, d):
    return float(softmax_scale) if softmax_scale else 1.0 / math.sqrt(d)


def _check_qkv(qs, kvs, separate_kv: bool = False):
    """qs: tensors shaped like q [total, H, d]; kvs: shaped like k [total, H_kv, d] with
    H_kv dividing H (with separate_kv, k has its own row count).  Returns H_kv."""
    ref = qs[0]
    for t in list(qs) + list(kvs):
        if t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
            raise ValueError("q/k/v/o tensors must be contiguous bf16 [total, heads, d]")
        if t.device != ref.device:
            raise ValueError("q/k/v/o tensors must share a device")
    for t in qs:
        if t.shape != ref.shape:
            raise ValueError("q, o and dO must share one shape [total, H, d]")
    kref = kvs[0]
    for t in kvs:
        if t.shape != kref.shape:
            raise ValueError("k and v must share one shape [total, H_kv, d]")
    if ((kref.shape[0] != ref.shape[0] and not separate_kv) or kref.shape[2] != ref.shape[2]
            or ref.shape[1] % kref.shape[1]):
        raise ValueError("k/v must be [total, H_kv, d] with H_kv dividing q's H")
    return kref.shape[1]


def varlen_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                    max_seqlen: int, softmax_scale: Optional[float] = None,
                    rope_theta: float = 10000.0, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    check: bool = True, rope_interleaved: bool = False,
                    cu_seqlens_padded: Optional[torch.Tensor] = None,
                    cu_seqlens_kv: Optional[torch.Tensor] = None, max_seqlen_kv: Optional[int] = None,
                    qk_rotated: bool = False, keys_all_visible: bool = False):
    """Segment-local causal attention with per-segment RoPE reset.  Returns (O, LSE[H, total]).
    k and v may have fewer heads than q (grouped: query head h reads head h // (H // H_kv)).
    rope_interleaved rotates the pairs (x[2j], x[2j+1]) instead of (x[j], x[j + d/2]).
    cu_seqlens_padded gives each segment a slot of rows starting at cu_seqlens_padded[r]
    (padding between segments; padding rows get O = 0, LSE = -inf).
    cu_seqlens_kv / max_seqlen_kv give k and v segments of their own, at least as long as the
    query segments; queries are bottom-right aligned (query p of a segment with L queries and
    Lk keys sits at position p + Lk - L and sees keys up to there).
    qk_rotated: q and k already hold the rotated q', k' of ``rope_qk`` (no rotation here).
    keys_all_visible (with cu_seqlens_kv and qk_rotated): every key of a query's key segment is
    visible, for a key block that precedes the query block (a context-parallel ring step)."""
    lib = load_library()
    _require_cuda(q, k, v, cu_seqlens, cu_seqlens_padded, cu_seqlens_kv)
    qkv = cu_seqlens_kv is not None
    if qkv and (cu_seqlens_padded is not None or max_seqlen_kv is None):
        raise ValueError("cu_seqlens_kv needs max_seqlen_kv and takes no padded layout")
    H_kv = _check_qkv([q] + ([] if out is None else [out]), [k, v], qkv)
    total, H, d = q.shape
    nseg = _cu_info(cu_seqlens, cu_seqlens_padded)
    if qkv:
        _cu_info(cu_seqlens_kv)
        if cu_seqlens_kv.numel() != nseg + 1:
            raise ValueError("cu_seqlens_kv must have one entry per segment boundary, like cu_seqlens")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device) if lse is None else lse
    total_kv = k.shape[0]
    if workspace is None:
        ws = new_workspace(nseg, total, H, d, max_seqlen, False, q.device, H_kv,
                           total_kv if qkv else None, max_seqlen_kv if qkv else None)
    else:
        ws = workspace
    flags = ((ROPE_INTERLEAVED if rope_interleaved else 0) | (QK_ROTATED if qk_rotated else 0)
             | (KEYS_ALL_VISIBLE if keys_all_visible else 0))
    if qkv:
        st = lib.vlc_attn_fwd_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(cu_seqlens_kv), nseg,
                                  total, total_kv, H, H_kv, d, int(max_seqlen), int(max_seqlen_kv),
                                  _scale(softmax_scale, d), float(rope_theta), flags, _ptr(out), _ptr(lse),
                                  _ptr(ws), ws.numel(), _stream(q.device))
    else:
        st = lib.vlc_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(cu_seqlens_padded),
                                 nseg, total, H, H_kv, d, int(max_seqlen), _scale(softmax_scale, d),
                                 float(rope_theta), flags, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                 _stream(q.device))
    _check(st, "vlc_attn_fwd")
    if check:
        _raise_device_error(ws, "vlc_attn_fwd")
    return out, lse


def varlen_attn_bwd(dout: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    o: torch.Tensor, lse: torch.Tensor, cu_seqlens: torch.Tensor, max_seqlen: int,
                    softmax_scale: Optional[float] = None, rope_theta: float = 10000.0,
                    dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                    dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    check: bool = True, rope_interleaved: bool = False,
                    cu_seqlens_padded: Optional[torch.Tensor] = None,
                    cu_seqlens_kv: Optional[torch.Tensor] = None, max_seqlen_kv: Optional[int] = None,
                    qk_rotated: bool = False, keys_all_visible: bool = False):
    """Gradients (dQ, dK, dV) of sum(O * dO) for the forward above (dK, dV shaped like k, v;
    zero at padding rows).  qk_rotated: q and k are the rotated q', k' of ``rope_qk``; the
    gradients returned are still with respect to the unrotated q and k.  keys_all_visible
    (with cu_seqlens_kv and rope_theta=0): the backward of a block whose keys all precede its
    queries, given the merged O and LSE of the whole attention (a context-parallel ring)."""
    lib = load_library()
    _require_cuda(dout, q, k, v, o, lse, cu_seqlens, cu_seqlens_padded, cu_seqlens_kv)
    qkv = cu_seqlens_kv is not None
    if qkv and (cu_seqlens_padded is not None or max_seqlen_kv is None):
        raise ValueError("cu_seqlens_kv needs max_seqlen_kv and takes no padded layout")
    H_kv = _check_qkv([q, dout, o], [k, v], qkv)
    total, H, d = q.shape
    nseg = _cu_info(cu_seqlens, cu_seqlens_padded)
    if qkv:
        _cu_info(cu_seqlens_kv)
        if cu_seqlens_kv.numel() != nseg + 1:
            raise ValueError("cu_seqlens_kv must have one entry per segment boundary, like cu_seqlens")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [H, total]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    total_kv = k.shape[0]
    if workspace is None:
        ws = new_workspace(nseg, total, H, d, max_seqlen, True, q.device, H_kv,
                           total_kv if qkv else None, max_seqlen_kv if qkv else None)
    else:
        ws = workspace
    flags = ((ROPE_INTERLEAVED if rope_interleaved else 0) | (QK_ROTATED if qk_rotated else 0)
             | (KEYS_ALL_VISIBLE if keys_all_visible else 0))
    if qkv:
        st = lib.vlc_attn_bwd_qkv(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                                  _ptr(cu_seqlens_kv), nseg, total, total_kv, H, H_kv, d, int(max_seqlen),
                                  int(max_seqlen_kv), _scale(softmax_scale, d), float(rope_theta), flags,
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(q.device))
    else:
        st = lib.vlc_attn_bwd_ex(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 _ptr(cu_seqlens), _ptr(cu_seqlens_padded), nseg, total, H, H_kv, d,
                                 int(max_seqlen), _scale(softmax_scale, d), float(rope_theta), flags,
                                 _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(q.device))
    _check(st, "vlc_attn_bwd")
    if check:
        _raise_device_error(ws, "vlc_attn_bwd")
    return dq, dk, dv


def shifted_cross_entropy(logits: torch.Tensor, labels: torch.Tensor,
                          cu_seqlens: Optional[torch.Tensor] = None, per_segment: bool = False,
                          workspace: Optional[torch.Tensor] = None, check: bool = True):
    """Next-token cross-entropy statistics over pre-shifted labels (-100 = ignored):
    returns (loss_sum fp32 [1], target_count int64 [1]) and, with per_segment, also
    (seg_loss fp32 [nseg], seg_count int32 [nseg]).  logits: bf16 [total, vocab]."""
    lib = load_library()
    _require_cuda(logits, labels, cu_seqlens, workspace)
    if logits.dtype != torch.bfloat16 or logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous bf16 [total, vocab] tensor")
    total, vocab = logits.shape
    if labels.dtype != torch.int64 or labels.numel() != total or not labels.is_contiguous():
        raise ValueError("labels must be contiguous int64 with one entry per logit row")
    nseg = 1 if cu_seqlens is None else _cu_info(cu_seqlens)
    dev = logits.device
    need = lib.vlc_ce_workspace_bytes(total, nseg)
    ws = workspace if workspace is not None else torch.empty(need, dtype=torch.uint8, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    count = torch.empty(1, dtype=torch.int64, device=dev)
    seg_loss = torch.empty(nseg, dtype=torch.float32, device=dev) if per_segment else None
    seg_count = torch.empty(nseg, dtype=torch.int32, device=dev) if per_segment else None
    st = lib.vlc_shifted_ce(_ptr(logits), vocab, total, _ptr(labels), _ptr(cu_seqlens), nseg, _ptr(loss),
                            _ptr(count), _ptr(seg_loss), _ptr(seg_count), _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "vlc_shifted_ce")
    if check:
        _raise_device_error(ws, "vlc_shifted_ce")
    return (loss, count, seg_loss, seg_count) if per_segment else (loss, count)


def rope_qk(q: torch.Tensor, k: torch.Tensor, cu_seqlens: torch.Tensor, max_seqlen: int,
            rope_theta: float = 10000.0, rope_interleaved: bool = False,
            cu_seqlens_padded: Optional[torch.Tensor] = None, out=None,
            workspace: Optional[torch.Tensor] = None, check: bool = True):
    """(q', k') = (R(p) q, R(p) k) with per-segment positions, for varlen_attn_fwd / _bwd with
    qk_rotated=True (one rotation per training step instead of one per pass)."""
    lib = load_library()
    _require_cuda(q, k, cu_seqlens, cu_seqlens_padded)
    H_kv = _check_qkv([q], [k])
    total, H, d = q.shape
    nseg = _cu_info(cu_seqlens, cu_seqlens_padded)
    qrot, krot = (torch.empty_like(q), torch.empty_like(k)) if out is None else out
    ws = new_workspace(nseg, total, H, d, max_seqlen, False, q.device, H_kv) if workspace is None else workspace
    st = lib.vlc_rope_qk(_ptr(q), _ptr(k), _ptr(cu_seqlens), _ptr(cu_seqlens_padded), nseg, total, H, H_kv, d,
                         int(max_seqlen), float(rope_theta), ROPE_INTERLEAVED if rope_interleaved else 0,
                         _ptr(qrot), _ptr(krot), _ptr(ws), ws.numel(), _stream(q.device))
    _check(st, "vlc_rope_qk")
    if check:
        _raise_device_error(ws, "vlc_rope_qk")
    return qrot, krot


def varlen_attn_fwd_rot(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                        max_seqlen: int, softmax_scale: Optional[float] = None, rope_theta: float = 10000.0,
                        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                        rotated_out=None, workspace: Optional[torch.Tensor] = None, check: bool = True,
                        rope_interleaved: bool = False):
    """The forward with RoPE in the kernel that also returns the rotated operands it attended
    with: (O, LSE, q', k').  A training step runs varlen_attn_bwd(..., qk_rotated=True) on q', k'
    and needs no separate rotation pass.  Self-attention, no padded layout, rope_theta > 0."""
    lib = load_library()
    _require_cuda(q, k, v, cu_seqlens)
    H_kv = _check_qkv([q] + ([] if out is None else [out]), [k, v])
    total, H, d = q.shape
    nseg = _cu_info(cu_seqlens)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device) if lse is None else lse
    qrot, krot = (torch.empty_like(q), torch.empty_like(k)) if rotated_out is None else rotated_out
    for t, ref in ((qrot, q), (krot, k)):
        if t.shape != ref.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("rotated outputs must be contiguous bf16 tensors shaped like q and k")
    ws = new_workspace(nseg, total, H, d, max_seqlen, False, q.device, H_kv) if workspace is None else workspace
    st = lib.vlc_attn_fwd_rot(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), nseg, total, H, H_kv, d, int(max_seqlen),
                              _scale(softmax_scale, d), float(rope_theta), ROPE_INTERLEAVED if rope_interleaved else 0,
                              _ptr(out), _ptr(lse), _ptr(qrot), _ptr(krot), _ptr(ws), ws.numel(), _stream(q.device))
    _check(st, "vlc_attn_fwd_rot")
    if check:
        _raise_device_error(ws, "vlc_attn_fwd_rot")
    return out, lse, qrot, krot


class Packing(NamedTuple):
    """Windows built by ``pack``: ``order[bin_start[w]:bin_start[w+1]]`` are window w's samples."""
    bin_of: np.ndarray      # int32 [n]
    order: np.ndarray       # int64 [n]
    bin_start: np.ndarray   # int64 [nbins + 1]
    nbins: int
    oversize: int
    capacity: int
    eta: float              # sum(lengths) / (nbins * capacity)

    def cu_seqlens(self, lengths, w: int) -> np.ndarray:
        """int32 cu_seqlens of window w (its samples in placement order)."""
        L = np.asarray(lengths, np.int64)[self.order[self.bin_start[w]:self.bin_start[w + 1]]]
        return np.concatenate([[0], np.cumsum(L)]).astype(np.int32)


def _host_i32(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x), dtype=np.int32)
    if a.ndim != 1:
        raise ValueError("lengths must be 1-D")
    return a


def pack(lengths, capacity: int, extra: int = 0, mode: str = "ffd") -> Packing:
    """Pack samples into windows of ``capacity`` tokens (host; see vlc_pack)."""
    lib = load_library()
    L = _host_i32(lengths)
    n = L.shape[0]
    bin_of = np.empty(n, np.int32)
    order = np.empty(n, np.int64)
    bin_start = np.empty(n + 1, np.int64)
    nb, ov = ctypes.c_int64(0), ctypes.c_int64(0)
    st = lib.vlc_pack(L.ctypes.data_as(ctypes.c_void_p), n, int(capacity), int(extra), PACK_MODES[mode],
                      bin_of.ctypes.data_as(ctypes.c_void_p), order.ctypes.data_as(ctypes.c_void_p),
                      bin_start.ctypes.data_as(ctypes.c_void_p), ctypes.byref(nb), ctypes.byref(ov))
    _check(st, "vlc_pack")
    nbins = int(nb.value)
    return Packing(bin_of, order, bin_start[:nbins + 1].copy(), nbins, int(ov.value), int(capacity),
                   float(L.astype(np.int64).sum()) / float(nbins * int(capacity)))


def shard_packs(lengths, packing: Packing, ranks: int, cost: str = "sumsq"):
    """Windows to ranks by attention work (host; see vlc_shard_packs): (rank_of_bin, rank_load)."""
    lib = load_library()
    L = _host_i32(lengths)
    order = np.ascontiguousarray(packing.order, np.int64)
    bs = np.ascontiguousarray(packing.bin_start, np.int64)
    rank_of = np.empty(packing.nbins, np.int32)
    load = np.empty(int(ranks), np.int64)
    st = lib.vlc_shard_packs(L.ctypes.data_as(ctypes.c_void_p), order.ctypes.data_as(ctypes.c_void_p),
                             bs.ctypes.data_as(ctypes.c_void_p), packing.nbins, int(ranks), COST_KINDS[cost],
                             rank_of.ctypes.data_as(ctypes.c_void_p), load.ctypes.data_as(ctypes.c_void_p))
    _check(st, "vlc_shard_packs")
    return rank_of, load


# ----------------------------------------------------------------------------- context-parallel split
def cp_partition(cu_seqlens, cp: int, rank: int):
    """Rows of the pack held by ``rank`` of a ``cp``-rank context-parallel group (host):
    (rows int64 [total / cp], positions int32, cu_chunk int32 [nseg + 1]).  The local buffer
    is the rank's low chunks of every segment, then its high chunks; each half is a packed
    buffer with segment offsets cu_chunk.  Every segment length must be a multiple of 2 cp."""
    lib = load_library()
    cu = _host_i32(cu_seqlens)
    nseg = len(cu) - 1
    total = int(cu[-1])
    if cp < 1 or total % cp != 0:
        raise ValueError("the pack length must be a multiple of cp (every segment a multiple of 2 cp)")
    rows = np.empty(total // cp, np.int64)
    pos = np.empty(total // cp, np.int32)
    cu_chunk = np.empty(nseg + 1, np.int32)
    bad = ctypes.c_int32(-1)
    st = lib.vlc_cp_partition(cu.ctypes.data, nseg, int(cp), int(rank), rows.ctypes.data, pos.ctypes.data,
                              cu_chunk.ctypes.data, ctypes.byref(bad))
    if st != 0 and bad.value >= 0:
        raise ValueError(f"segment {bad.value} has a length that is not a multiple of 2 * cp = {2 * cp}")
    _check(st, "vlc_cp_partition")
    return rows, pos, cu_chunk


def cp_block_mode(cp: int, q_rank: int, q_half: int, kv_rank: int, kv_half: int) -> int:
    """CP_BLOCK_ALL, CP_BLOCK_CAUSAL or CP_BLOCK_NONE for the queries of (q_rank, q_half) against
    the keys of (kv_rank, kv_half) (half 0 = low chunks, 1 = high chunks)."""
    m = load_library().vlc_cp_block_mode(int(cp), int(q_rank), int(q_half), int(kv_rank), int(kv_half))
    if m < 0:
        raise ValueError("invalid cp / rank / half")
    return m


def rope_pos(x: torch.Tensor, pos: torch.Tensor, max_pos: int, rope_theta: float = 10000.0,
             rope_interleaved: bool = False, out: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, check: bool = True, transpose: bool = False) -> torch.Tensor:
    """R(pos[i]) x[i] for every head of every row ([rows, H, d] bf16, pos int32 [rows]);
    transpose applies R(pos[i])^T (gradients back through the rotation)."""
    lib = load_library()
    _require_cuda(x, pos)
    rows, H, d = x.shape
    out = torch.empty_like(x) if out is None else out
    need = lib.vlc_rope_pos_workspace_bytes(int(max_pos), d)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device) if workspace is None else workspace
    st = lib.vlc_rope_pos(_ptr(x), _ptr(pos), rows, H, d, int(max_pos), float(rope_theta),
                          (ROPE_INTERLEAVED if rope_interleaved else 0) | (ROPE_TRANSPOSE if transpose else 0),
                          _ptr(out), _ptr(ws), ws.numel(), _stream(x.device))
    _check(st, "vlc_rope_pos")
    if check:
        _raise_device_error(ws, "vlc_rope_pos")
    return out


def lse_merge(o_parts, lse_parts, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """Merge attention results over disjoint key sets: O parts bf16 [rows, H, d], LSE parts fp32
    [H, rows]; returns (O, LSE) over the union."""
    lib = load_library()
    n = len(o_parts)
    if n != len(lse_parts) or not 1 <= n <= LSE_MERGE_MAX:
        raise ValueError(f"1 to {LSE_MERGE_MAX} parts, as many O as LSE")
    _require_cuda(*o_parts, *lse_parts)
    rows, H, d = o_parts[0].shape
    for a, b in zip(o_parts, lse_parts):
        if tuple(a.shape) != (rows, H, d) or tuple(b.shape) != (H, rows) or not a.is_contiguous() \
                or not b.is_contiguous():
            raise ValueError("parts must be contiguous bf16 [rows, H, d] and fp32 [H, rows]")
    out = torch.empty_like(o_parts[0]) if out is None else out
    lse = torch.empty((H, rows), dtype=torch.float32, device=out.device) if lse is None else lse
    optr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in o_parts])
    lptr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lse_parts])
    st = lib.vlc_lse_merge(optr, lptr, n, rows, H, d, _ptr(out), _ptr(lse), _stream(out.device))
    _check(st, "vlc_lse_merge")
    return out, lse


def sum_parts(parts, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Sum of 1 to 16 bf16 tensors of one shape, accumulated in fp32 and rounded once."""
    lib = load_library()
    n = len(parts)
    if not 1 <= n <= LSE_MERGE_MAX:
        raise ValueError(f"1 to {LSE_MERGE_MAX} parts")
    _require_cuda(*parts)
    for t in parts:
        if t.shape != parts[0].shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("parts must be contiguous bf16 tensors of one shape")
    out = torch.empty_like(parts[0]) if out is None else out
    ptrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in parts])
    st = lib.vlc_sum_parts(ptrs, n, parts[0].numel(), _ptr(out), _stream(out.device))
    _check(st, "vlc_sum_parts")
    return out
