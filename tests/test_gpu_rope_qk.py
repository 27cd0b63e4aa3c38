"""vlc_rope_qk and the pre-rotated operand option (VLC_QK_ROTATED): one rotation per
training step.  The rotated rows match the oracle's rotation to one bf16 rounding; the
forward and backward on q', k' match the oracle within the usual bounds; the backward on
q', k' is bit-identical to the backward that rotates in its own prep pass (same table,
same arithmetic).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import brute
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
    gen = torch.Generator(device=DEV).manual_seed(seed)
    q, g = (torch.randn((w.total, H, d), generator=gen, device=DEV).bfloat16() for _ in range(2))
    k, v = (torch.randn((w.total, Hkv, d), generator=gen, device=DEV).bfloat16() for _ in range(2))
    return w, q, k, v, g


@pytest.mark.parametrize("il", [False, True])
def test_rotated_rows_match_the_oracle_rotation(vlc, il):
    w, q, k, _, _ = _inputs([1, 300, 2100, 77], 4, 2, 128, seed=3)
    cu = torch.from_numpy(w.cu).to(DEV)
    qr, kr = vlc.rope_qk(q, k, cu, w.max_seqlen, rope_interleaved=il)
    pos = brute.local_positions(w.cu)
    for x, xr in ((q, qr), (k, kr)):
        xs = oracle.bits_to_f64(oracle.bf16_bits(x.cpu()))
        ref = np.stack([oracle.rope_rows(xs[:, h], pos, interleaved=il) for h in range(x.shape[1])], axis=1)
        got = xr.float().cpu().numpy()
        ulp = np.maximum(np.abs(ref), 1e-30) * 2.0 ** -7    # one bf16 rounding step
        assert np.all(np.abs(got - ref) <= ulp + 1e-6)


@pytest.mark.parametrize("il", [False, True])
def test_step_on_rotated_operands(vlc, il):
    w, q, k, v, g = _inputs([1, 130, 7, 2100, 300], 4, 2, 128, seed=11)
    cu = torch.from_numpy(w.cu).to(DEV)
    qr, kr = vlc.rope_qk(q, k, cu, w.max_seqlen, rope_interleaved=il)
    o, lse = vlc.varlen_attn_fwd(qr, kr, v, cu, w.max_seqlen, rope_interleaved=il, qk_rotated=True)
    qc, kc, vc, gc = (t.cpu() for t in (q, k, v, g))
    o_ref, lse_ref = oracle.attn_fwd(qc, kc, vc, w.cu, interleaved=il)
    e = np.abs(o.float().cpu().numpy() - o_ref)
    assert e.max() <= O_MAX and e.mean() <= O_MEAN
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_MAX
    dq, dk, dv = vlc.varlen_attn_bwd(g, qr, kr, v, o, lse, cu, w.max_seqlen, rope_interleaved=il,
                                     qk_rotated=True)
    ref = oracle.attn_bwd(gc, qc, kc, vc, w.cu, interleaved=il)
    for a, b in zip((dq, dk, dv), ref):
        assert np.abs(a.float().cpu().numpy() - b).max() <= G_MAX
    # the backward on q', k' is the backward that rotates in its prep pass, bit for bit
    g2 = vlc.varlen_attn_bwd(g, q, k, v, o, lse, cu, w.max_seqlen, rope_interleaved=il)
    for a, b in zip((dq, dk, dv), g2):
        assert torch.equal(a, b)


def test_rotated_padded_layout(vlc):
    lens, pads = [300, 5, 2100], [20, 0, 44]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cp = np.concatenate([[0], np.cumsum(np.add(lens, pads))]).astype(np.int32)
    total = int(cp[-1])
    gen = torch.Generator(device=DEV).manual_seed(5)
    q, k, v, g = (torch.randn((total, 2, 128), generator=gen, device=DEV).bfloat16() for _ in range(4))
    cut, cpt = torch.from_numpy(cu).to(DEV), torch.from_numpy(cp).to(DEV)
    qr, kr = vlc.rope_qk(q, k, cut, max(lens), cu_seqlens_padded=cpt)
    real = np.zeros(total, bool)
    real[oracle.real_rows(cu, cp)] = True
    pad = torch.from_numpy(~real).to(DEV)
    assert torch.all(qr[pad] == 0) and torch.all(kr[pad] == 0)
    o, lse = vlc.varlen_attn_fwd(qr, kr, v, cut, max(lens), cu_seqlens_padded=cpt, qk_rotated=True)
    o_ref, _ = oracle.attn_fwd(q.cpu(), k.cpu(), v.cpu(), cu, cu_padded=cp)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_MAX
    dq, dk, dv = vlc.varlen_attn_bwd(g, qr, kr, v, o, lse, cut, max(lens), cu_seqlens_padded=cpt, qk_rotated=True)
    ref = oracle.attn_bwd(g.cpu(), q.cpu(), k.cpu(), v.cpu(), cu, cu_padded=cp)
    for a, b in zip((dq, dk, dv), ref):
        assert np.abs(a.float().cpu().numpy() - b).max() <= G_MAX


@pytest.mark.parametrize("il,hkv,d", [(False, 4, 128), (True, 4, 128), (False, 2, 128), (True, 4, 64)])
def test_fwd_rot_returns_the_rotated_operands_for_the_backward(vlc, il, hkv, d):
    # the forward with RoPE in the kernel also writes q' (from the kernel's q-tile rotation) and
    # k' (from its k pass); the backward on them with qk_rotated matches the oracle, and k' is
    # the rotation pass's k' bit for bit (hkv < 4: grouped key/value heads)
    lens = [700, 1, 333, 129, 2300]
    w = synth.custom_workload(lens, 4, d)
    q, k, v, g = synth.make_tensors(w, seed=91, with_grad=True)
    k, v = k[:, :hkv].contiguous(), v[:, :hkv].contiguous()
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    cu = torch.from_numpy(w.cu).to(DEV)
    o, lse, qr, kr = vlc.varlen_attn_fwd_rot(qd, kd, vd, cu, w.max_seqlen, rope_interleaved=il)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.cu, interleaved=il)
    e = o.float().cpu().numpy() - o_ref
    assert np.abs(e).max() <= 2e-2 and np.abs(e).mean() <= 2e-3
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3
    qr1, kr1 = vlc.rope_qk(qd, kd, cu, w.max_seqlen, rope_interleaved=il)
    assert torch.equal(kr, kr1)
    # q' from the in-kernel rotation: the same rotation up to the angle recurrence's last bits
    assert torch.allclose(qr.float(), qr1.float(), rtol=2.0 ** -7, atol=1e-6)
    grads = vlc.varlen_attn_bwd(gd, qr, kr, vd, o, lse, cu, w.max_seqlen, qk_rotated=True, rope_interleaved=il)
    ref = oracle.attn_bwd(g, q, k, v, w.cu, interleaved=il)
    for name, a, b in zip(("dq", "dk", "dv"), grads, ref):
        err = np.abs(a.float().cpu().numpy() - b)
        assert np.isfinite(err).all() and err.max() <= 5e-2, (name, err.max())
