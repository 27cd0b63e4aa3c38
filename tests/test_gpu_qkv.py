"""GPU parity for queries and keys/values with segments of their own (cu_seqlens_kv,
bottom-right aligned: query p of a segment with L queries and Lk >= L keys sits at position
p + Lk - L and sees keys 0 .. p + Lk - L): forward and backward through the C ABI against
the fp64 oracle (O max 2e-2, mean 2e-3, LSE 1e-3, gradients max 5e-2).
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


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _inputs(Tq, Tk, H, Hkv, d, seed, device="cpu"):
    gen = torch.Generator(device=device).manual_seed(seed)
    q, g = (torch.randn((Tq, H, d), generator=gen, device=device).bfloat16() for _ in range(2))
    k, v = (torch.randn((Tk, Hkv, d), generator=gen, device=device).bfloat16() for _ in range(2))
    return q, k, v, g


def _cmp(got, want, bound, name):
    got = got.float().cpu().numpy()
    assert np.isfinite(got).all(), name
    e = np.abs(got - np.asarray(want))
    assert e.max() <= bound, f"{name} max err {e.max()}"
    return e


# (L, Lk): square, one-query decode steps, offsets that are and are not tile multiples,
# partial first tiles, several q tiles against a longer key run
LQ = [1, 200, 128, 130, 64, 1, 257, 7, 300]
LK = [1, 300, 384, 1000, 64, 129, 700, 7, 301]


@pytest.mark.parametrize("H,Hkv,d,theta,il", [(4, 4, 128, 10000.0, False), (8, 2, 64, 10000.0, False),
                                              (6, 3, 128, 0.0, False), (4, 2, 128, 500000.0, True)])
def test_qkv_fwd_bwd_small(vlc, H, Hkv, d, theta, il):
    cu, cuk = _cu(LQ), _cu(LK)
    q, k, v, g = _inputs(int(cu[-1]), int(cuk[-1]), H, Hkv, d, seed=H * 3 + Hkv + d)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cut, cukt = torch.from_numpy(cu).to(DEV), torch.from_numpy(cuk).to(DEV)
    kw = dict(rope_theta=theta, rope_interleaved=il, cu_seqlens_kv=cukt, max_seqlen_kv=max(LK))
    o, lse = vlc.varlen_attn_fwd(qd, kd, vd, cut, max(LQ), **kw)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, cu, theta=theta, interleaved=il, cu_kv=cuk)
    eo = _cmp(o, o_ref, O_MAX, "O")
    assert eo.mean() <= O_MEAN
    _cmp(lse, lse_ref, LSE_MAX, "LSE")
    dq, dk, dv = vlc.varlen_attn_bwd(gd, qd, kd, vd, o, lse, cut, max(LQ), **kw)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    ref = oracle.attn_bwd(g, q, k, v, cu, theta=theta, interleaved=il, cu_kv=cuk)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        _cmp(a, b, G_MAX, name)


def test_qkv_equal_lengths_match_self_attention_bitwise(vlc):
    # cu_kv == cu takes the same tiles and masks as the self-attention call
    lens = [700, 1, 333, 129]
    cu = _cu(lens)
    q, k, v, g = _inputs(int(cu[-1]), int(cu[-1]), 8, 4, 128, seed=4, device=DEV)
    cut = torch.from_numpy(cu).to(DEV)
    o1, l1 = vlc.varlen_attn_fwd(q, k, v, cut, max(lens))
    o2, l2 = vlc.varlen_attn_fwd(q, k, v, cut, max(lens), cu_seqlens_kv=cut.clone(), max_seqlen_kv=max(lens))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = vlc.varlen_attn_bwd(g, q, k, v, o1, l1, cut, max(lens))
    g2 = vlc.varlen_attn_bwd(g, q, k, v, o2, l2, cut, max(lens), cu_seqlens_kv=cut.clone(),
                             max_seqlen_kv=max(lens))
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_qkv_tail_queries_match_the_self_attention_rows(vlc):
    # the last L rows of each segment's self-attention, asked as L queries against the whole
    # segment, agree with the self-attention outputs on those rows (up to summation order)
    lk, lq = [900, 300, 1], [128, 201, 1]
    cuk, cu = _cu(lk), _cu(lq)
    qf, k, v, _ = _inputs(int(cuk[-1]), int(cuk[-1]), 4, 4, 128, seed=8, device=DEV)
    tail = torch.from_numpy(np.concatenate([np.arange(a - n, a) for a, n in zip(cuk[1:], lq)])).to(DEV)
    cukt, cut = torch.from_numpy(cuk).to(DEV), torch.from_numpy(cu).to(DEV)
    o_s, l_s = vlc.varlen_attn_fwd(qf, k, v, cukt, max(lk))
    o, lse = vlc.varlen_attn_fwd(qf[tail].contiguous(), k, v, cut, max(lq), cu_seqlens_kv=cukt,
                                 max_seqlen_kv=max(lk))
    assert (o.float() - o_s[tail].float()).abs().max().item() <= 2e-2
    assert (lse - l_s[:, tail]).abs().max().item() <= 1e-3


def test_qkv_full_size_sampled(vlc):
    # chunked-prefill shape: the pretraining-window pack's segments as keys, the last quarter
    # of each as queries; sampled (segment, key/value head) pairs recomputed by the oracle
    base = synth.workload(4)
    lk = np.diff(base.cu).astype(np.int64)
    lq = np.maximum(1, lk // 4)
    cu, cuk = _cu(lq), _cu(lk)
    H, Hkv, d = 32, 8, 128
    q, k, v, g = _inputs(int(cu[-1]), int(cuk[-1]), H, Hkv, d, seed=17, device=DEV)
    cut, cukt = torch.from_numpy(cu).to(DEV), torch.from_numpy(cuk).to(DEV)
    kw = dict(cu_seqlens_kv=cukt, max_seqlen_kv=int(lk.max()))
    o, lse = vlc.varlen_attn_fwd(q, k, v, cut, int(lq.max()), **kw)
    dq, dk, dv = vlc.varlen_attn_bwd(g, q, k, v, o, lse, cut, int(lq.max()), **kw)
    order = np.argsort(lk, kind="stable")
    pairs = [(int(order[-1]), 0), (int(order[len(order) // 2]), Hkv - 1), (int(order[0]), 3)]
    qc, kc, vc, gc = (t.cpu() for t in (q, k, v, g))
    grp = H // Hkv
    ref = oracle.attn_bwd(gc, qc, kc, vc, cu, seg_heads=pairs, cu_kv=cuk)
    for s, hk in pairs:
        a, b = int(cu[s]), int(cu[s + 1])
        ka, kb = int(cuk[s]), int(cuk[s + 1])
        heads = list(range(hk * grp, (hk + 1) * grp))
        o_ref, lse_ref = oracle.attn_fwd(qc, kc, vc, cu, seg_heads=[(s, h) for h in heads], cu_kv=cuk)
        for h in heads:
            _cmp(o[a:b, h], o_ref[a:b, h], O_MAX, "O")
            _cmp(lse[h, a:b], lse_ref[h, a:b], LSE_MAX, "LSE")
        _cmp(dq[a:b, hk * grp:(hk + 1) * grp], ref[0][a:b, hk * grp:(hk + 1) * grp], G_MAX, "dq")
        _cmp(dk[ka:kb, hk], ref[1][ka:kb, hk], G_MAX, "dk")
        _cmp(dv[ka:kb, hk], ref[2][ka:kb, hk], G_MAX, "dv")


def test_qkv_fewer_keys_than_queries_is_reported(vlc):
    cu, cuk = _cu([5, 9]), _cu([5, 8])
    q, k, v, _ = _inputs(14, 13, 2, 2, 64, seed=1, device=DEV)
    with pytest.raises(vlc.VlcError) as ei:
        vlc.varlen_attn_fwd(q, k, v, torch.from_numpy(cu).to(DEV), 9, cu_seqlens_kv=torch.from_numpy(cuk).to(DEV),
                            max_seqlen_kv=8)
    assert ei.value.bits & vlc.binding.DEVERR_QKV
