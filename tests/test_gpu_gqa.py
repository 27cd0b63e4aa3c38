"""GPU parity for grouped key/value heads (H_kv dividing H; query head h reads key/value
head h // (H // H_kv)): forward and backward through the C ABI against the fp64 oracle,
with the same bounds as the equal-head tests (O max 2e-2, mean 2e-3, LSE 1e-3, gradients
max 5e-2).  dK and dV sum the contributions of their group's query heads.
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


LENS = [1, 130, 7, 257, 64, 129]


@pytest.mark.parametrize("H,Hkv,d", [(8, 2, 128), (8, 1, 64), (6, 3, 128), (4, 4, 64)])
@pytest.mark.parametrize("theta", [10000.0, 0.0])
def test_gqa_fwd_bwd_small(vlc, H, Hkv, d, theta):
    w, q, k, v, g = _inputs(LENS, H, Hkv, d, seed=H * 10 + Hkv + d)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cu = torch.from_numpy(w.cu).to(DEV)
    o, lse = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen, rope_theta=theta)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.cu, theta=theta)
    eo = _cmp(o, o_ref, O_MAX, "O")
    assert eo.mean() <= O_MEAN
    _cmp(lse, lse_ref, LSE_MAX, "LSE")
    dq, dk, dv = vlc.varlen_attn_bwd(gd, qd, kd, vd, o, lse, cu, w.max_seqlen, rope_theta=theta)
    assert dk.shape == k.shape and dv.shape == v.shape
    ref = oracle.attn_bwd(g, q, k, v, w.cu, theta=theta)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        _cmp(a, b, G_MAX, name)


def test_gqa_equals_repeated_heads(vlc):
    # grouped heads give bit-identical O / LSE / dQ to equal heads with k, v repeated per
    # query head, and dK / dV equal to the group sums of the repeated run's gradients
    H, Hkv, d = 8, 2, 128
    w, q, k, v, g = _inputs([300, 45, 600], H, Hkv, d, seed=5)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cu = torch.from_numpy(w.cu).to(DEV)
    kr, vr = (x.repeat_interleave(H // Hkv, dim=1).contiguous() for x in (kd, vd))
    o1, l1 = vlc.varlen_attn_fwd(qd, kd, vd, cu, w.max_seqlen)
    o2, l2 = vlc.varlen_attn_fwd(qd, kr, vr, cu, w.max_seqlen)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = vlc.varlen_attn_bwd(gd, qd, kd, vd, o1, l1, cu, w.max_seqlen)
    g2 = vlc.varlen_attn_bwd(gd, qd, kr, vr, o2, l2, cu, w.max_seqlen)
    assert torch.equal(g1[0], g2[0])
    for a, b in ((g1[1], g2[1]), (g1[2], g2[2])):
        s = b.float().reshape(w.total, Hkv, H // Hkv, d).sum(2)
        err = (a.float() - s).abs() / (1.0 + s.abs())   # bf16 rounding of the summed parts
        assert err.max().item() <= 1e-2


def test_gqa_full_size_sampled(vlc):
    # the pretraining-window fwd+bwd shape with 32 query heads over 8 key/value heads;
    # sampled (segment, key/value head) pairs recomputed by the oracle
    base = synth.workload(4)
    H, Hkv, d = 32, 8, 128
    gen = torch.Generator(device=DEV).manual_seed(9)
    q, g = (torch.randn((base.total, H, d), generator=gen, device=DEV).bfloat16() for _ in range(2))
    k, v = (torch.randn((base.total, Hkv, d), generator=gen, device=DEV).bfloat16() for _ in range(2))
    cu = torch.from_numpy(base.cu).to(DEV)
    o, lse = vlc.varlen_attn_fwd(q, k, v, cu, base.max_seqlen)
    dq, dk, dv = vlc.varlen_attn_bwd(g, q, k, v, o, lse, cu, base.max_seqlen)
    real = np.nonzero(base.seg_ignore == 0)[0]
    lens = base.lengths
    by_len = real[np.argsort(lens[real], kind="stable")]
    pairs = [(int(by_len[(3 * len(by_len)) // 4]), 0), (int(by_len[0]), Hkv - 1),
             (int(by_len[len(by_len) // 2]), 3)]
    qc, kc, vc, gc = (t.cpu() for t in (q, k, v, g))
    ref = oracle.attn_bwd(gc, qc, kc, vc, base.cu, seg_heads=pairs)
    grp = H // Hkv
    for s, hk in pairs:
        a, b = int(base.cu[s]), int(base.cu[s + 1])
        _cmp(dq[a:b, hk * grp:(hk + 1) * grp], ref[0][a:b, hk * grp:(hk + 1) * grp], G_MAX, "dq")
        _cmp(dk[a:b, hk], ref[1][a:b, hk], G_MAX, "dk")
        _cmp(dv[a:b, hk], ref[2][a:b, hk], G_MAX, "dv")
        heads = list(range(hk * grp, (hk + 1) * grp))
        o_ref, lse_ref = oracle.attn_fwd(qc, kc, vc, base.cu, seg_heads=[(s, h) for h in heads])
        for h in heads:
            _cmp(o[a:b, h], o_ref[a:b, h], O_MAX, "O")
            _cmp(lse[h, a:b], lse_ref[h, a:b], LSE_MAX, "LSE")
