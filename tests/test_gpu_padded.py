"""GPU parity for padded layouts (cu_seqlens_padded: segment r's tokens at rows
cu_padded[r] .. cu_padded[r] + L_r - 1, padding up to cu_padded[r+1]): forward and
backward through the C ABI against the fp64 oracle (O max 2e-2, mean 2e-3, LSE 1e-3,
gradients max 5e-2), padding outputs exactly O = 0, LSE = -inf, zero gradients, and the
real rows bit-identical to the same pack laid out without padding.
"""
import numpy as np
import pytest
import torch

import oracle
from variable_length_causal_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
O_MAX, O_MEAN, LSE_MAX, G_MAX = 2e-2, 2e-3, 1e-3, 5e-2


@pytest.fixture(scope="module")
def vlc():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as m

    m.load_library()
    return m


def _layout(lens, pads):
    lens, pads = np.asarray(lens, np.int64), np.asarray(pads, np.int64)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cp = np.concatenate([[0], np.cumsum(lens + pads)]).astype(np.int32)
    return cu, cp


def _inputs(total, H, Hkv, d, seed, device="cpu"):
    gen = torch.Generator(device=device).manual_seed(seed)
    q, g = (torch.randn((total, H, d), generator=gen, device=device).bfloat16() for _ in range(2))
    k, v = (torch.randn((total, Hkv, d), generator=gen, device=device).bfloat16() for _ in range(2))
    return q, k, v, g


def _cmp(got, want, bound, name):
    got = got.float().cpu().numpy()
    want = np.asarray(want)
    assert np.isfinite(got).all(), name
    e = np.abs(got - want)
    assert e.max() <= bound, f"{name} max err {e.max()}"
    return e


LENS = [1, 130, 7, 257, 64, 129, 300]
PADS = [127, 0, 9, 3, 64, 0, 31]   # the padding rows hold random (finite) values


@pytest.mark.parametrize("H,Hkv,d,theta,il", [(4, 4, 128, 10000.0, False), (8, 2, 64, 10000.0, False),
                                              (6, 3, 128, 0.0, False), (4, 2, 128, 500000.0, True)])
def test_padded_fwd_bwd_small(vlc, H, Hkv, d, theta, il):
    cu, cp = _layout(LENS, PADS)
    total = int(cp[-1])
    q, k, v, g = _inputs(total, H, Hkv, d, seed=H + Hkv + d)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cut, cpt = torch.from_numpy(cu).to(DEV), torch.from_numpy(cp).to(DEV)
    mx = max(LENS)
    o, lse = vlc.varlen_attn_fwd(qd, kd, vd, cut, mx, rope_theta=theta, rope_interleaved=il,
                                 cu_seqlens_padded=cpt)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, cu, theta=theta, interleaved=il, cu_padded=cp)
    real = np.zeros(total, bool)
    real[oracle.real_rows(cu, cp)] = True
    eo = _cmp(o, o_ref, O_MAX, "O")
    assert eo[real].mean() <= O_MEAN
    assert torch.all(o[torch.from_numpy(~real).to(DEV)] == 0)
    lse_c = lse.cpu().numpy()
    assert np.all(np.isneginf(lse_c[:, ~real]))
    assert np.abs(lse_c[:, real] - lse_ref[:, real]).max() <= LSE_MAX
    # dO at padding rows is nonzero garbage too: it must not leak into any gradient
    dq, dk, dv = vlc.varlen_attn_bwd(gd, qd, kd, vd, o, lse, cut, mx, rope_theta=theta, rope_interleaved=il,
                                     cu_seqlens_padded=cpt)
    ref = oracle.attn_bwd(g, q, k, v, cu, theta=theta, interleaved=il, cu_padded=cp)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        _cmp(a, b, G_MAX, name)
        assert torch.all(a[torch.from_numpy(~real).to(DEV)] == 0), name


def _padded_vs_packed(vlc, lens, pads, H, Hkv, d, seed):
    cu, cp = _layout(lens, pads)
    idx = torch.from_numpy(oracle.real_rows(cu, cp)).to(DEV)
    total = int(cp[-1])
    q, k, v, g = _inputs(total, H, Hkv, d, seed, device=DEV)
    cut, cpt = torch.from_numpy(cu).to(DEV), torch.from_numpy(cp).to(DEV)
    mx = int(max(lens))
    o1, l1 = vlc.varlen_attn_fwd(q, k, v, cut, mx, cu_seqlens_padded=cpt)
    g1 = vlc.varlen_attn_bwd(g, q, k, v, o1, l1, cut, mx, cu_seqlens_padded=cpt)
    qp, kp, vp, gp = (x[idx].contiguous() for x in (q, k, v, g))
    o2, l2 = vlc.varlen_attn_fwd(qp, kp, vp, cut, mx)
    g2 = vlc.varlen_attn_bwd(gp, qp, kp, vp, o2, l2, cut, mx)
    assert torch.equal(o1[idx], o2) and torch.equal(l1[:, idx], l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a[idx], b)


def test_padded_real_rows_equal_the_packed_run(vlc):
    # masked tile entries contribute exact zeros, so the real rows match bit for bit
    _padded_vs_packed(vlc, [700, 1, 333, 1030, 5], [1, 200, 0, 62, 9], 8, 4, 128, seed=5)


def test_padded_full_size_equals_packed(vlc):
    # the SFT pack's segments each padded up to a multiple of 64 rows (a context-parallel
    # style alignment), H = 32, d = 128, as bench.py's shapes
    w = synth.workload(1)
    lens = np.diff(w.cu).astype(np.int64)
    pads = (-lens) % 64
    _padded_vs_packed(vlc, lens, pads, w.H, w.H, w.d, seed=13)


def test_padded_bad_offsets_are_reported(vlc):
    cu, cp = _layout([5, 9, 3], [0, 2, 1])
    total = int(cp[-1])
    q, k, v, _ = _inputs(total, 2, 2, 64, seed=1, device=DEV)
    cut = torch.from_numpy(cu).to(DEV)
    bad = cp.copy()
    bad[2] = bad[1] + 8                       # slot 1 (8 rows) shorter than segment 1 (9 tokens)
    for c in (bad, np.where(np.arange(len(cp)) == len(cp) - 1, total + 4, cp).astype(np.int32)):
        with pytest.raises(vlc.VlcError) as ei:
            vlc.varlen_attn_fwd(q, k, v, cut, 9, cu_seqlens_padded=torch.from_numpy(c).to(DEV))
        assert ei.value.bits & vlc.binding.DEVERR_CU_PADDED
