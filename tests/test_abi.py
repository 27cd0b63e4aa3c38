"""The C-ABI library builds, loads, and exports every function include/vlc.h declares (CPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "vlc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vlc_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as vlc

    return vlc.load_library()


def test_header_declares_the_path():
    names = _declared()
    for n in ("vlc_build_positions_labels", "vlc_attn_fwd", "vlc_attn_bwd", "vlc_build_worklist",
              "vlc_get_error", "vlc_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from variable_length_causal_gb300 import binding

    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(binding.EXPORTED) == _declared()


def test_host_side_queries(lib):
    assert lib.vlc_version() >= 100
    assert lib.vlc_status_string(0) == b"ok"
    assert lib.vlc_workspace_bytes(3, 9, 2, 128, 4, 0) > 0
    assert lib.vlc_workspace_bytes(3, 9, 2, 96, 4, 0) == 0        # unsupported head dim
    assert lib.vlc_workspace_bytes(3, 9, 2, 128, 4, 1) > lib.vlc_workspace_bytes(3, 9, 2, 128, 4, 0)
    assert lib.vlc_worklist_capacity(3, 9, 128) == 3 + 0 + 1


def parts_one(ctypes, p):
    arr = (ctypes.c_void_p * 1)()
    arr[0] = p
    return arr


def test_host_argument_checks_need_no_gpu(lib):
    import ctypes

    # null pointers are rejected before anything touches a device
    assert lib.vlc_attn_fwd(None, None, None, None, 3, 9, 2, 128, 4, 0.0, 0.0, None, None, None, 0, None) == 1
    assert lib.vlc_build_positions_labels(None, 3, None, 9, None, None, None, None, None) == 1
    dummy = ctypes.c_void_p(256)
    # unsupported head dim / missing workspace
    assert lib.vlc_attn_fwd(dummy, dummy, dummy, dummy, 3, 9, 2, 96, 4, 0.0, 0.0, dummy, dummy,
                            dummy, 1 << 20, None) == 3
    assert lib.vlc_attn_fwd(dummy, dummy, dummy, dummy, 3, 9, 2, 128, 4, 0.0, 0.0, dummy, dummy,
                            None, 0, None) == 4
    # option words: an unknown bit is refused before the shape checks
    assert lib.vlc_attn_fwd_ex(dummy, dummy, dummy, dummy, None, 3, 9, 2, 2, 128, 4, 0.0, 1e4, 0x8,
                               dummy, dummy, dummy, 1 << 20, None) == 1
    # all keys visible needs separate key segments and operands rotated beforehand
    assert lib.vlc_attn_fwd_ex(dummy, dummy, dummy, dummy, None, 3, 9, 2, 2, 128, 4, 0.0, 1e4, 0x6,
                               dummy, dummy, dummy, 1 << 20, None) == 1
    assert lib.vlc_attn_fwd_qkv(dummy, dummy, dummy, dummy, dummy, 3, 9, 12, 2, 2, 128, 4, 6, 0.0, 1e4, 0x4,
                                dummy, dummy, dummy, 1 << 20, None) == 1
    # the backward takes pre-rotated operands for self-attention only, and all-visible blocks only
    # without RoPE (gradients with respect to the operands as given)
    assert lib.vlc_attn_bwd_qkv(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, 3, 9, 12, 2, 2, 128, 4,
                                6, 0.0, 1e4, 0x2, dummy, dummy, dummy, dummy, 1 << 20, None) == 1
    assert lib.vlc_attn_bwd_qkv(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, 3, 9, 12, 2, 2, 128, 4,
                                6, 0.0, 1e4, 0x4, dummy, dummy, dummy, dummy, 1 << 20, None) == 1
    assert lib.vlc_sum_parts(None, 1, 8, dummy, None) == 1
    assert lib.vlc_sum_parts(parts_one(ctypes, dummy), 1, 12, dummy, None) == 1     # not a multiple of 8
    # context-parallel host calls and argument checks
    assert lib.vlc_cp_block_mode(2, 0, 1, 1, 0) == 2 and lib.vlc_cp_block_mode(2, 0, 2, 0, 0) == -1
    assert lib.vlc_rope_pos(dummy, dummy, 4, 2, 128, 9, 1e4, 0x2, dummy, dummy, 1 << 20, None) == 1
    assert lib.vlc_rope_pos(dummy, dummy, 4, 2, 96, 9, 1e4, 0, dummy, dummy, 1 << 20, None) == 3
    assert lib.vlc_rope_pos(dummy, dummy, 4, 2, 128, 9, 1e4, 0, dummy, None, 0, None) == 4
    assert lib.vlc_rope_pos_workspace_bytes(127, 128) == 256 + 128 * 64 * 8
    assert lib.vlc_lse_merge(None, None, 1, 4, 2, 128, dummy, dummy, None) == 1
    parts = (ctypes.c_void_p * 17)()
    assert lib.vlc_lse_merge(parts, parts, 17, 4, 2, 128, dummy, dummy, None) == 1
    assert lib.vlc_rope_qk(dummy, dummy, dummy, None, 3, 9, 2, 2, 128, 4, 1e4, 0x2, dummy, dummy, dummy,
                           1 << 20, None) == 1
    # the forward that returns q', k': both outputs, RoPE on, only the interleaved bit
    fwd_rot = lambda qr, kr, theta, flags, d=128: lib.vlc_attn_fwd_rot(
        dummy, dummy, dummy, dummy, 3, 9, 2, 2, d, 4, 0.0, theta, flags, dummy, dummy, qr, kr, dummy, 1 << 20, None)
    assert fwd_rot(None, dummy, 1e4, 0) == 1
    assert fwd_rot(dummy, None, 1e4, 0) == 1
    assert fwd_rot(dummy, dummy, 0.0, 0) == 1
    assert fwd_rot(dummy, dummy, 1e4, 0x2) == 1
    assert fwd_rot(dummy, dummy, 1e4, 0x1, d=96) == 3   # the interleaved bit passes; d = 96 is unsupported
    assert lib.vlc_attn_bwd_ex(dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, 3, 9, 2, 2, 128,
                               4, 0.0, 1e4, 0x80000000, dummy, dummy, dummy, dummy, 1 << 20, None) == 1
    # the interleaved bit itself is accepted: the call proceeds to the shape checks
    assert lib.vlc_attn_fwd_ex(dummy, dummy, dummy, dummy, dummy, 3, 9, 2, 2, 96, 4, 0.0, 1e4, 0x1,
                               dummy, dummy, dummy, 1 << 20, None) == 3
