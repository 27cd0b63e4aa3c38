"""GPU parity of the context-parallel split: rotation by explicit positions, the
all-keys-visible forward block, the LSE merge, and whole rings emulated on one GPU
(every rank's blocks run one after another) against the oracle's full attention."""
import numpy as np
import pytest
import torch

import oracle
from oracle import cp as ocp
from variable_length_causal_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def vlc():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as m

    m.load_library()
    return m


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).bfloat16()


@pytest.mark.parametrize("d,il", [(128, False), (64, False), (128, True)])
def test_rope_pos_matches_rope_qk_and_oracle(vlc, d, il):
    lens = [300, 17, 1000, 129]
    w = synth.custom_workload(lens, 3, d)
    q, k, _ = synth.make_tensors(w, seed=11)
    cu = torch.from_numpy(w.cu).to(DEV)
    qd, kd = q.to(DEV), k.to(DEV)
    qr, kr = vlc.rope_qk(qd, kd, cu, w.max_seqlen, rope_interleaved=il)
    seg = np.repeat(np.arange(len(lens)), lens)
    pos = (np.arange(w.total) - w.cu[seg]).astype(np.int32)
    pos_d = torch.from_numpy(pos).to(DEV)
    qp = vlc.rope_pos(qd, pos_d, w.max_seqlen - 1, rope_interleaved=il)
    kp = vlc.rope_pos(kd, pos_d, w.max_seqlen - 1, rope_interleaved=il)
    assert torch.equal(qp, qr) and torch.equal(kp, kr)        # same table, same arithmetic
    # against the oracle's fp64 rotation, rounded to bf16: within one bf16 step
    ref = oracle.rope_rows(q.float().numpy().reshape(-1, d), np.repeat(pos, 3), interleaved=il)
    got = qp.float().cpu().numpy().reshape(-1, d)
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.maximum(np.abs(ref), 1e-30) + 1e-6)


def test_rope_pos_flags_out_of_range_positions(vlc):
    x = _bf16((8, 2, 128), 1).to(DEV)
    pos = torch.tensor([0, 1, 2, 3, 9, 5, -1, 7], dtype=torch.int32, device=DEV)
    with pytest.raises(vlc.VlcError):
        vlc.rope_pos(x, pos, 7)
    out = vlc.rope_pos(x, pos, 7, check=False)
    assert bool((out[4] == 0).all()) and bool((out[6] == 0).all())
    assert bool((out[0] == x[0]).all())                      # position 0 is the identity


@pytest.mark.parametrize("d", [64, 128])
def test_lse_merge_matches_oracle(vlc, d):
    rows, H, n = 333, 3, 5
    g = np.random.default_rng(d)
    o_parts = [_bf16((rows, H, d), 20 + i) for i in range(n)]
    lse_parts = [torch.from_numpy(g.normal(0, 3, (H, rows)).astype(np.float32)) for _ in range(n)]
    lse_parts[1][:, :50] = -float("inf")                     # parts that saw no key
    for lp in lse_parts:
        lp[0, 7] = -float("inf")                             # a row no part saw
    o, lse = vlc.lse_merge([t.to(DEV) for t in o_parts], [t.to(DEV) for t in lse_parts])
    o_ref, lse_ref = ocp.lse_merge([t.double().numpy() for t in o_parts], [t.double().numpy() for t in lse_parts])
    got = o.float().cpu().numpy()
    assert np.all(np.abs(got - o_ref) <= 2.0 ** -8 * np.abs(o_ref) + 1e-6)
    l = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(l[fin] - lse_ref[fin]).max() <= 1e-5 * max(1.0, np.abs(lse_ref[fin]).max())
    assert bool((o[7, 0] == 0).all())


@pytest.mark.parametrize("m", [[200, 77], [128, 256], [1, 513]])
def test_all_keys_visible_block(vlc, m):
    # queries of chunk 1 against the keys of chunk 0 of the same segments: every key precedes
    # every query, so the block has no causal mask (pre-rotated operands)
    H, d = 2, 128
    cu = np.concatenate([[0], np.cumsum(m)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v = _bf16((T, H, d), 31), _bf16((T, H, d), 32), _bf16((T, H, d), 33)
    cud = torch.from_numpy(cu).to(DEV)
    o, lse = vlc.varlen_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cud, max(m), cu_seqlens_kv=cud,
                                 max_seqlen_kv=max(m), qk_rotated=True, keys_all_visible=True)
    seg = np.repeat(np.arange(len(m)), m)
    pos = np.arange(T) - cu[seg]
    o_ref, l_ref = ocp.block_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), seg,
                                       pos + 10 ** 6, seg, pos, 1.0 / np.sqrt(d))
    e = np.abs(o.float().cpu().numpy() - o_ref)
    assert e.max() <= O_MAX and e.mean() <= O_MEAN
    assert np.abs(lse.cpu().numpy() - l_ref).max() <= LSE_MAX
    # without the flag the same call is the causal square block
    o2, l2 = vlc.varlen_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), cud, max(m), cu_seqlens_kv=cud,
                                 max_seqlen_kv=max(m), qk_rotated=True)
    o_ref2, l_ref2 = ocp.block_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), seg, pos,
                                         seg, pos, 1.0 / np.sqrt(d))
    assert np.abs(o2.float().cpu().numpy() - o_ref2).max() <= O_MAX
    assert np.abs(l2.cpu().numpy() - l_ref2).max() <= LSE_MAX


def _ring(vlc, q, k, v, cu, cp, theta=10000.0):
    """Every rank's output rows after a full ring, computed one rank after another."""
    out = []
    for rank in range(cp):
        rows, pos, cu_chunk = vlc.cp_partition(cu, cp, rank)
        rows_d = torch.from_numpy(rows).to(DEV)
        pos_d = torch.from_numpy(pos).to(DEV)
        maxp = int(np.diff(cu).max()) - 1
        loc = {}
        for r2 in range(cp):
            rr, pp, _ = vlc.cp_partition(cu, cp, r2)
            rr_d, pp_d = torch.from_numpy(rr).to(DEV), torch.from_numpy(pp).to(DEV)
            loc[r2] = (vlc.rope_pos(q[rr_d], pp_d, maxp, theta), vlc.rope_pos(k[rr_d], pp_d, maxp, theta),
                       v[rr_d].contiguous())
        half = len(rows) // 2
        cuc = torch.from_numpy(cu_chunk).to(DEV)
        mc = int(np.diff(cu_chunk).max())
        res_o, res_l = [], []
        for qh in (0, 1):
            qs = slice(qh * half, (qh + 1) * half)
            parts_o, parts_l = [], []
            for step in range(cp):
                src = (rank - step) % cp
                for kh in (0, 1):
                    mode = vlc.cp_block_mode(cp, rank, qh, src, kh)
                    if mode == vlc.binding.CP_BLOCK_NONE:
                        continue
                    ks = slice(kh * half, (kh + 1) * half)
                    o_p, l_p = vlc.varlen_attn_fwd(loc[rank][0][qs], loc[src][1][ks], loc[src][2][ks], cuc, mc,
                                                   cu_seqlens_kv=cuc, max_seqlen_kv=mc, qk_rotated=True,
                                                   keys_all_visible=mode == vlc.binding.CP_BLOCK_ALL)
                    parts_o.append(o_p)
                    parts_l.append(l_p)
            o_m, l_m = vlc.lse_merge(parts_o, parts_l)
            res_o.append(o_m)
            res_l.append(l_m)
        out.append((rows, torch.cat(res_o), torch.cat(res_l, dim=1)))
    return out


@pytest.mark.parametrize("cp", [2, 4])
@pytest.mark.parametrize("lens,H,d", [([32768], 2, 128), ([4096, 1024, 2560, 512, 8192, 64], 4, 64)])
def test_context_parallel_ring_matches_full_attention(vlc, cp, lens, H, d):
    w = synth.custom_workload(lens, H, d)
    q, k, v = synth.make_tensors(w, seed=sum(lens) + cp)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    res = _ring(vlc, qd, kd, vd, w.cu, cp)
    covered = np.concatenate([r[0] for r in res])
    assert np.array_equal(np.sort(covered), np.arange(w.total))
    rng = np.random.default_rng(cp + len(lens))
    for rows, o_loc, lse_loc in res:
        pick = rng.choice(len(rows), size=24, replace=False)
        heads = rng.integers(0, H, size=24)
        o_ref, l_ref = oracle.attn_fwd_rows(q, k, v, w.cu, rows[pick], heads)
        got = o_loc[torch.from_numpy(pick).to(DEV), torch.from_numpy(heads).to(DEV)].float().cpu().numpy()
        e = np.abs(got - o_ref)
        assert e.max() <= O_MAX and e.mean() <= O_MEAN
        gl = lse_loc[torch.from_numpy(heads).to(DEV), torch.from_numpy(pick).to(DEV)].cpu().numpy()
        assert np.abs(gl - l_ref).max() <= LSE_MAX


def test_rope_pos_transpose_inverts(vlc):
    x = _bf16((300, 2, 128), 5).to(DEV)
    pos = torch.arange(300, dtype=torch.int32, device=DEV) * 7 % 1000
    y = vlc.rope_pos(x, pos, 999)
    back = vlc.rope_pos(y, pos, 999, transpose=True)
    assert (back.float() - x.float()).abs().max().item() <= 2e-2    # two bf16 roundings
    # the transpose is the rotation by -p: against the oracle's fp64 rotation
    ref = oracle.rope_rows(x.float().cpu().numpy().reshape(-1, 128), -np.repeat(pos.cpu().numpy(), 2))
    got = vlc.rope_pos(x, pos, 999, transpose=True).float().cpu().numpy().reshape(-1, 128)
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.maximum(np.abs(ref), 1e-30) + 1e-6)


def test_sum_parts(vlc):
    parts = [_bf16((37, 3, 64), 60 + i).to(DEV) for i in range(5)]
    out = vlc.sum_parts(parts)
    ref = sum(p.double() for p in parts)
    assert ((out.double() - ref).abs() <= 2.0 ** -8 * ref.abs() + 1e-6).all()


@pytest.mark.parametrize("cp", [2, 4])
def test_context_parallel_ring_backward_matches_full_gradients(vlc, cp):
    """The ring's backward, all ranks one after another: every block's backward with the
    merged O and LSE of its query half, block gradients summed per query half and per key
    half, then taken back through R(pos)^T; against the oracle's full gradients."""
    lens, H, d = [4096, 1024, 2560, 512, 64, 1000 - 1000 % (2 * cp)], 4, 64
    w = synth.custom_workload(lens, H, d)
    q, k, v, g = synth.make_tensors(w, seed=sum(lens) + 7 * cp, with_grad=True)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    maxp = max(lens) - 1
    loc = {}
    for r in range(cp):
        rows, pos, cu_chunk = vlc.cp_partition(w.cu, cp, r)
        rd, pd = torch.from_numpy(rows).to(DEV), torch.from_numpy(pos).to(DEV)
        loc[r] = dict(rows=rows, pos=pd, qr=vlc.rope_pos(qd[rd], pd, maxp), kr=vlc.rope_pos(kd[rd], pd, maxp),
                      v=vd[rd].contiguous(), g=gd[rd].contiguous())
    cuc = torch.from_numpy(cu_chunk).to(DEV)
    mc = int(np.diff(cu_chunk).max())
    half = len(loc[0]["rows"]) // 2
    sl = lambda h: slice(h * half, (h + 1) * half)
    blocks = {(r, qh): [(src, kh, vlc.cp_block_mode(cp, r, qh, src, kh)) for step in range(cp)
                        for src in [(r - step) % cp] for kh in (0, 1)] for r in range(cp) for qh in (0, 1)}
    blocks = {key: [b for b in val if b[2] != vlc.binding.CP_BLOCK_NONE] for key, val in blocks.items()}
    # forward: merged O and LSE of every query half
    om, lm = {}, {}
    for (r, qh), bl in blocks.items():
        parts = [vlc.varlen_attn_fwd(loc[r]["qr"][sl(qh)], loc[s]["kr"][sl(kh)], loc[s]["v"][sl(kh)], cuc, mc,
                                     cu_seqlens_kv=cuc, max_seqlen_kv=mc, qk_rotated=True,
                                     keys_all_visible=m == vlc.binding.CP_BLOCK_ALL) for s, kh, m in bl]
        om[(r, qh)], lm[(r, qh)] = vlc.lse_merge([a for a, _ in parts], [b for _, b in parts])
    # backward of every block; dq' collected per query half, dk', dv per key half
    dq_p = {key: [] for key in blocks}
    dk_p = {key: [] for key in blocks}
    dv_p = {key: [] for key in blocks}
    for (r, qh), bl in blocks.items():
        for s, kh, m in bl:
            gq, gk, gv = vlc.varlen_attn_bwd(loc[r]["g"][sl(qh)], loc[r]["qr"][sl(qh)], loc[s]["kr"][sl(kh)],
                                             loc[s]["v"][sl(kh)], om[(r, qh)], lm[(r, qh)], cuc, mc, rope_theta=0.0,
                                             cu_seqlens_kv=cuc, max_seqlen_kv=mc,
                                             keys_all_visible=m == vlc.binding.CP_BLOCK_ALL)
            dq_p[(r, qh)].append(gq)
            dk_p[(s, kh)].append(gk)
            dv_p[(s, kh)].append(gv)
    dq = torch.zeros_like(qd)
    dk = torch.zeros_like(kd)
    dv = torch.zeros_like(vd)
    for (r, h), parts in dq_p.items():
        rows_d = torch.from_numpy(loc[r]["rows"][sl(h)]).to(DEV)
        pos_h = loc[r]["pos"][sl(h)].contiguous()
        dq[rows_d] = vlc.rope_pos(vlc.sum_parts(parts), pos_h, maxp, transpose=True)
        dk[rows_d] = vlc.rope_pos(vlc.sum_parts(dk_p[(r, h)]), pos_h, maxp, transpose=True)
        dv[rows_d] = vlc.sum_parts(dv_p[(r, h)])
    ref = oracle.attn_bwd(g, q, k, v, w.cu)
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        e = np.abs(a.float().cpu().numpy() - b)
        assert np.isfinite(e).all() and e.max() <= 5e-2, (name, e.max())
