"""GPU parity for the interleaved RoPE pairing (pairs x[2j], x[2j+1] at the frequencies
theta^(-2j/d); the per-segment position reset is unchanged): forward and backward through
the C ABI against the fp64 oracle with the same bounds as the rotate-half tests (O max
2e-2, mean 2e-3, LSE 1e-3, gradients max 5e-2).
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


def _inputs(lens, H, Hkv, d, seed):
    w = synth.custom_workload(lens, H, d)
    gen = torch.Generator().manual_seed(seed)
    q, g = (torch.randn((w.total, H, d), generator=gen).bfloat16() for _ in range(2))
    k, v = (torch.randn((w.total, Hkv, d), generator=gen).bfloat16() for _ in range(2))
    return w, q, k, v, g


def _cmp(got, want, bound, name):
    got = got.float().cpu().numpy()
    assert np.isfinite(got).all(), name
    e = np.abs(got - want)
    assert e.max() <= bound, f"{name} max err {e.max()}"
    return e


LENS = [1, 130, 7, 257, 64, 129, 300]


@pytest.mark.parametrize("H,Hkv,d", [(4, 4, 128), (4, 4, 64), (8, 2, 128), (6, 3, 64)])
@pytest.mark.parametrize("theta", [10000.0, 500000.0])
def test_interleaved_fwd_bwd_small(vlc, H, Hkv, d, theta):
    w, q, k, v, g = _inputs(LENS, H, Hkv, d, seed=H * 7 + Hkv + d)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cu = torch.from_numpy(w.cu).to(DEV)
    o, lse = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, rope_theta=theta, rope_interleaved=True)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.cu, theta=theta, interleaved=True)
    eo = _cmp(o, o_ref, O_MAX, "O")
    assert eo.mean() <= O_MEAN
    _cmp(lse, lse_ref, LSE_MAX, "LSE")
    dq, dk, dv = vlc.varlen_attn_bwd(gd, qd, kd, vd, o, lse, cu, w.max_seqlen, rope_theta=theta,
                                     rope_interleaved=True)
    ref = oracle.attn_bwd(g, q, k, v, w.cu, theta=theta, interleaved=True)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        _cmp(a, b, G_MAX, name)


def test_pairing_matters_and_theta_zero_ignores_it(vlc):
    # the two pairings give different outputs; without RoPE the bit changes nothing
    w, q, k, v, _ = _inputs([200, 90], 4, 4, 128, seed=3)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    cu = torch.from_numpy(w.cu).to(DEV)
    a = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, rope_interleaved=True)[0]
    b = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, rope_interleaved=False)[0]
    assert (a.float() - b.float()).abs().max().item() > 0.05
    c = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, rope_theta=0.0, rope_interleaved=True)[0]
    e = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, rope_theta=0.0)[0]
    assert torch.equal(c, e)


def test_interleaved_is_rotate_half_on_permuted_columns(vlc):
    # moving even columns to the first half and odd ones to the second turns the interleaved
    # rotation into the rotate-half one; scores are sums over all columns, so the interleaved
    # run on (q, k) and the rotate-half run on the permuted (q, k) agree up to summation order,
    # and the gradients agree after permuting dq, dk back
    H, Hkv, d = 8, 4, 128
    w, q, k, v, g = _inputs([700, 1, 333, 1030], H, Hkv, d, seed=11)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cu = torch.from_numpy(w.cu).to(DEV)
    perm = torch.cat([torch.arange(0, d, 2), torch.arange(1, d, 2)]).to(DEV)
    inv = torch.argsort(perm)
    qp, kp = qd[..., perm].contiguous(), kd[..., perm].contiguous()
    o1, l1 = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, rope_interleaved=True)
    o2, l2 = vlc.varlen_attn_fwd(qp, kp, vd, cu, w.max_seqlen)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3
    g1 = vlc.varlen_attn_bwd(gd, qd, kd, vd, o1, l1, cu, w.max_seqlen, rope_interleaved=True)
    g2 = vlc.varlen_attn_bwd(gd, qp, kp, vd, o2, l2, cu, w.max_seqlen)
    for a, b in ((g1[0], g2[0][..., inv]), (g1[1], g2[1][..., inv]), (g1[2], g2[2])):
        assert (a.float() - b.float()).abs().max().item() <= 5e-2


def test_interleaved_full_size_sampled(vlc):
    # the pretraining-window shape (4096-token windows of the pack), sampled segments and
    # heads recomputed by the oracle
    base = synth.workload(4)
    H, d = base.H, base.d
    gen = torch.Generator(device=DEV).manual_seed(21)
    q, k, v, g = (torch.randn((base.total, H, d), generator=gen, device=DEV).bfloat16() for _ in range(4))
    cu = torch.from_numpy(base.cu).to(DEV)
    o, lse = vlc.varlen_attn_fwd(q, k, v, cu, base.max_seqlen, rope_interleaved=True)
    dq, dk, dv = vlc.varlen_attn_bwd(g, q, k, v, o, lse, cu, base.max_seqlen, rope_interleaved=True)
    real = np.nonzero(base.seg_ignore == 0)[0]
    by_len = real[np.argsort(base.lengths[real], kind="stable")]
    pairs = [(int(by_len[-1]), 0), (int(by_len[len(by_len) // 2]), H - 1), (int(by_len[0]), H // 2)]
    qc, kc, vc, gc = (t.cpu() for t in (q, k, v, g))
    o_ref, lse_ref = oracle.attn_fwd(qc, kc, vc, base.cu, seg_heads=pairs, interleaved=True)
    ref = oracle.attn_bwd(gc, qc, kc, vc, base.cu, seg_heads=pairs, interleaved=True)
    for s, h in pairs:
        a, b = int(base.cu[s]), int(base.cu[s + 1])
        _cmp(o[a:b, h], o_ref[a:b, h], O_MAX, "O")
        _cmp(lse[h, a:b], lse_ref[h, a:b], LSE_MAX, "LSE")
        for name, x, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            _cmp(x[a:b, h], r[a:b, h], G_MAX, name)
