"""Pins of the fp64 oracle against what the pages and mathematics fix (CPU only).

Each test names the page and section whose value or property it checks.  A
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a mask applied after the softmax, a position that does
not reset) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from tests.conftest import GOLDEN
from variable_length_causal_gb300 import synth


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _rand_qkv(lengths, H, d, seed, with_grad=False):
    w = synth.custom_workload(lengths, H, d)
    return w, synth.make_tensors(w, seed=seed, with_grad=with_grad)


def _f64(t):
    return t.float().double().numpy()


# ------------------------------------------------------------------ cu_seqlens, positions, labels

def test_nine_token_example_positions():
    """charlestar, 'Nine tokens together keep three sample identities'."""
    g = _golden("nine_token_example.json")
    tokens = np.arange(g["total"]) + 1
    pos, _ = oracle.positions_labels(g["cu_seqlens"], tokens)
    assert pos.tolist() == g["position"]
    assert oracle.validate_cu(g["cu_seqlens"], g["total"], g["max_seqlen"]) == 0
    # max_seqlen is the largest segment, not the total nor a bin capacity
    assert oracle.validate_cu(g["cu_seqlens"], g["total"], g["total"]) == oracle.ERR_MAXLEN
    assert oracle.validate_cu(g["cu_seqlens"], g["total"], 3) == oracle.ERR_MAXLEN
    # segment ids agree with numpy's searchsorted (brute)
    assert brute.segment_ids(np.array(g["cu_seqlens"])).tolist() == g["segment"]


@pytest.mark.parametrize("cu,total,maxlen,err", [
    ([1, 3, 5, 9], 9, 4, oracle.ERR_CU_FIRST),
    ([0, 3, 3, 9], 9, 6, oracle.ERR_CU_ORDER),
    ([0, 5, 3, 9], 9, 6, oracle.ERR_CU_ORDER),
    ([0, 3, 5, 9], 10, 4, oracle.ERR_CU_TOTAL),
    ([0, 3, 5, 9], 9, 5, oracle.ERR_MAXLEN),
])
def test_validity_contract(cu, total, maxlen, err):
    """charlestar: cu[0]==0, strictly increasing, cu[-1]==total, max_seqlen == max diff."""
    got = oracle.validate_cu(cu, total, maxlen)
    assert got & err == err
    if err == oracle.ERR_CU_FIRST:
        assert got == oracle.ERR_CU_FIRST | (0 if maxlen == 4 else oracle.ERR_MAXLEN)


def test_preshifted_labels_example():
    """M020 section 06: A=[11,12,13], B=[21,22] -> [12, 13, ignore, 22, ignore], 3 targets."""
    g = _golden("labels_example.json")
    pos, lab = oracle.positions_labels(g["cu_seqlens"], g["tokens"])
    assert pos.tolist() == g["positions"]
    assert lab.tolist() == g["labels_preshifted"]
    assert int(np.sum(lab != -100)) == g["valid_targets"]


def test_internal_shift_gives_same_prediction_pairs():
    """charlestar, 'one cross-boundary prediction pair remains': the internal-shift
    labels (-100 at segment starts, logits[:-1] vs labels[1:]) and the pre-shifted labels
    (-100 at segment ends) supervise the same (input position -> target) pairs, and the
    count is sum (L_r - 1) = 6 for nine tokens."""
    g = _golden("internal_shift_labels.json")
    tok = np.array(g["tokens"])
    cu = np.array(g["cu_seqlens"])
    internal = tok.copy()
    internal[cu[:-1]] = -100
    assert internal.tolist() == g["labels_internal_shift"]
    pairs_internal = {(i, int(internal[i + 1])) for i in range(len(tok) - 1) if internal[i + 1] != -100}
    _, pre = oracle.positions_labels(cu, tok)
    pairs_pre = {(i, int(pre[i])) for i in range(len(tok)) if pre[i] != -100}
    assert pairs_internal == pairs_pre
    assert len(pairs_pre) == g["valid_targets"] == int(np.sum(np.diff(cu) - 1))
    names = g["tokens_symbolic"]
    sym = sorted((names[i], names[i + 1]) for i, _ in pairs_pre)
    assert sym == sorted(tuple(p) for p in g["prediction_pairs_symbolic"])


def test_ignored_segment_labels_all_ignored():
    """llm-compass 'Implementation notes': the padding tail's labels are all -100."""
    cu = [0, 3, 5, 9]
    tok = np.arange(9) + 7
    _, lab = oracle.positions_labels(cu, tok, seg_ignore=[0, 1, 0])
    assert lab[3:5].tolist() == [-100, -100]
    assert lab[:3].tolist() == [8, 9, -100]
    assert lab[5:].tolist() == [13, 14, 15, -100]


def test_positions_labels_random_against_searchsorted():
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 40, size=30)
    cu = np.concatenate([[0], np.cumsum(lens)])
    tok = rng.integers(0, 1000, size=cu[-1])
    ign = (rng.random(30) < 0.2).astype(np.uint8)
    pos, lab = oracle.positions_labels(cu, tok, ign)
    seg = brute.segment_ids(cu)
    assert np.array_equal(pos, brute.local_positions(cu))
    nxt_same = np.append(seg[1:] == seg[:-1], False)
    want = np.where(nxt_same & (ign[seg] == 0), np.append(tok[1:], -100), -100)
    assert np.array_equal(lab, want)


# ------------------------------------------------------------------ attention forward

def test_contamination_counterexample():
    """charlestar, 'EOS is content; isolation happens before softmax': scores all 0,
    V(A)=1, V(b0)=10 -> isolated b0 output 10, whole-pack causal 3.25."""
    g = _golden("contamination_counterexample.json")
    d = 4
    T = 9
    q = torch.zeros(T, 1, d, dtype=torch.bfloat16)
    k = _bf16(np.random.default_rng(0).standard_normal((T, 1, d)))
    v = torch.full((T, 1, d), 5.0, dtype=torch.bfloat16)
    v[0:3] = g["v_values"]["A"]
    v[3] = g["v_values"]["b0"]
    r = g["query_row"]
    o_iso, _ = oracle.attn_fwd(q, k, v, g["cu_seqlens_isolated"])
    o_all, _ = oracle.attn_fwd(q, k, v, g["cu_seqlens_whole_pack"], theta=0.0)
    assert np.allclose(o_iso[r, 0], g["output_isolated"], atol=1e-12)
    assert np.allclose(o_all[r, 0], g["output_whole_pack"], atol=1e-12)


def test_closed_form_zero_queries():
    """With Q = 0 every allowed score is 0: LSE_i = ln(p_i + 1) and O_i is the mean of the
    segment's V rows 0..p_i (uniform softmax over the allowed keys only)."""
    lens = [1, 7, 3, 12, 2]
    w, (q, k, v) = _rand_qkv(lens, 2, 8, seed=3)
    q = torch.zeros_like(q)
    o, lse = oracle.attn_fwd(q, k, v, w.cu)
    pos = brute.local_positions(w.cu)
    assert np.allclose(lse, np.log(pos + 1.0)[None, :], atol=1e-13)
    vf = _f64(v)
    for r in range(len(lens)):
        a, b = w.cu[r], w.cu[r + 1]
        mean = np.cumsum(vf[a:b], axis=0) / np.arange(1, b - a + 1)[:, None, None]
        assert np.allclose(o[a:b], mean, atol=1e-13)


@pytest.mark.parametrize("theta,contract", [(0.0, True), (10000.0, False), (10000.0, True), (500.0, False)])
@pytest.mark.parametrize("d", [8, 16])
def test_against_whole_pack_brute_force(theta, contract, d):
    """Segment-by-segment oracle == full T x T masked softmax (numpy, complex-form RoPE)."""
    lens = [1, 5, 17, 3, 9]
    w, (q, k, v) = _rand_qkv(lens, 3, d, seed=11)
    o, lse = oracle.attn_fwd(q, k, v, w.cu, theta=theta, contract=contract)
    ob, lseb = brute.attention(_f64(q), _f64(k), _f64(v), w.cu, theta=theta, contract=contract)
    tol = 1e-12 if not contract else 1e-9
    assert np.max(np.abs(o - ob)) < tol
    assert np.max(np.abs(lse - lseb)) < tol


def test_against_torch_sdpa_bool_mask():
    """torch CPU fp64 scaled_dot_product_attention with a boolean mask, True = attend
    (charlestar notes PyTorch SDPA's boolean semantics)."""
    lens = [4, 1, 11, 6]
    w, (q, k, v) = _rand_qkv(lens, 2, 16, seed=21)
    pos = brute.local_positions(w.cu)
    qr = brute.rope_complex(_f64(q), pos, 10000.0)
    kr = brute.rope_complex(_f64(k), pos, 10000.0)
    mask = torch.from_numpy(brute.block_causal_allow(w.cu))
    qt = torch.from_numpy(qr).permute(1, 0, 2)
    kt = torch.from_numpy(kr).permute(1, 0, 2)
    vt = torch.from_numpy(_f64(v)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    o, _ = oracle.attn_fwd(q, k, v, w.cu, contract=False)
    assert np.max(np.abs(o - ref.permute(1, 0, 2).numpy())) < 1e-12


def test_packed_equals_per_sample_and_isolation():
    """charlestar, 'change A, B must not change'; M020 section 08: packed run equals the
    per-sample runs, and replacing A's tokens leaves B and C bit-identical."""
    lens = [3, 2, 4]
    w, (q, k, v) = _rand_qkv(lens, 2, 8, seed=2)
    o, lse = oracle.attn_fwd(q, k, v, w.cu)
    for r, L in enumerate(lens):
        a, b = w.cu[r], w.cu[r + 1]
        o1, l1 = oracle.attn_fwd(q[a:b].contiguous(), k[a:b].contiguous(), v[a:b].contiguous(), [0, L])
        assert np.array_equal(o1, o[a:b])
        assert np.array_equal(l1, lse[:, a:b])
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    g = torch.Generator().manual_seed(99)
    q2[:3] = torch.randn(3, 2, 8, generator=g).bfloat16()
    k2[:3] = torch.randn(3, 2, 8, generator=g).bfloat16()
    v2[:3] = torch.randn(3, 2, 8, generator=g).bfloat16()
    o2, lse2 = oracle.attn_fwd(q2, k2, v2, w.cu)
    assert np.array_equal(o2[3:], o[3:]) and np.array_equal(lse2[:, 3:], lse[:, 3:])
    assert not np.array_equal(o2[:3], o[:3])


def test_wrong_cu_changes_a_and_b0():
    """charlestar: writing [0,4,5,9] instead of [0,3,5,9] puts b0 into A's context."""
    g = _golden("nine_token_example.json")
    w, (q, k, v) = _rand_qkv(g["lengths"], 1, 8, seed=4)
    o_ok, _ = oracle.attn_fwd(q, k, v, g["cu_seqlens"])
    o_bad, _ = oracle.attn_fwd(q, k, v, g["wrong_cu_seqlens"])
    assert not np.allclose(o_ok[3], o_bad[3])           # b0 now sees A
    assert not np.allclose(o_ok[4], o_bad[4])           # B's EOS lost b0 from its context
    assert np.array_equal(o_ok[:3], o_bad[:3])          # A's own rows keep their prefix
    assert np.array_equal(o_ok[5:], o_bad[5:])          # C untouched


def test_rows_api_matches_full():
    lens = [130, 7, 260]
    w, (q, k, v) = _rand_qkv(lens, 2, 16, seed=8)
    o, lse = oracle.attn_fwd(q, k, v, w.cu)
    rows = np.array([0, 129, 130, 136, 137, 300, 396])
    heads = np.array([0, 1, 1, 0, 1, 0, 1])
    o_r, l_r = oracle.attn_fwd_rows(q, k, v, w.cu, rows, heads)
    assert np.array_equal(o_r, o[rows, heads])
    assert np.array_equal(l_r, lse[heads, rows])


# ------------------------------------------------------------------ RoPE

def test_rope_closed_forms():
    """R(0) = I; d=2 rotates by angle p; d=4's second pair turns at theta^(-1/2) per step
    (rotate-half pairing (x_j, x_{j+d/2}), fixed frequencies theta^(-2j/d))."""
    x = np.random.default_rng(0).standard_normal((5, 8))
    assert np.array_equal(oracle.rope_rows(x, np.zeros(5)), x)
    p = 3
    out = oracle.rope_rows(np.array([[1.0, 0.0]]), [p])[0]
    assert np.allclose(out, [math.cos(p), math.sin(p)], atol=1e-15)
    out = oracle.rope_rows(np.array([[0.0, 1.0, 0.0, 0.0]]), [p], theta=10000.0)[0]
    ang = p * 10000.0 ** (-0.5)
    assert np.allclose(out, [0.0, math.cos(ang), 0.0, math.sin(ang)], atol=1e-15)


def test_rope_shift_invariance_and_norm():
    """charlestar, 'the pure-RoPE argument': (R(m+c)q)^T (R(n+c)k) = q^T R(n-m) k."""
    rng = np.random.default_rng(1)
    d = 64
    for _ in range(20):
        q, k = rng.standard_normal((2, d))
        m, n, c = rng.integers(0, 4000, size=3)
        a = oracle.rope_rows(q[None], [m + c])[0] @ oracle.rope_rows(k[None], [n + c])[0]
        b = oracle.rope_rows(q[None], [m])[0] @ oracle.rope_rows(k[None], [n])[0]
        assert abs(a - b) < 1e-9 * (1 + abs(b))
        assert abs(np.linalg.norm(oracle.rope_rows(q[None], [m])[0]) - np.linalg.norm(q)) < 1e-12
    x = rng.standard_normal((7, 32))
    pos = rng.integers(0, 30000, size=7)
    assert np.allclose(oracle.rope_rows(x, pos), brute.rope_complex(x, pos, 10000.0), atol=1e-9)


def test_rope_exact_mode_reset_invariance():
    """In exact mode, resetting positions per segment or counting them across the pack gives
    the same attention output (the shift cancels inside each segment's scores)."""
    lens = [6, 9]
    w, (q, k, v) = _rand_qkv(lens, 1, 16, seed=6)
    o, _ = oracle.attn_fwd(q, k, v, w.cu, contract=False)
    # second segment alone, but with its q/k pre-rotated by the pack offset c = 6
    a, b = w.cu[1], w.cu[2]
    qf, kf = _f64(q[a:b]), _f64(k[a:b])
    c = np.full(b - a, a)
    qs = brute.rope_complex(qf, c, 10000.0)
    ks = brute.rope_complex(kf, c, 10000.0)
    o2, _ = oracle.attn_fwd_f64(qs, ks, _f64(v[a:b]), [0, b - a])
    assert np.max(np.abs(o2 - o[a:b])) < 1e-12


def test_round_bf16_against_torch():
    """brute.round_bf16 (integer RNE on binary64) agrees with torch's float32->bf16 rounding on
    float32-representable values, where a single rounding happens."""
    x = np.random.default_rng(3).standard_normal(100000).astype(np.float32)
    x = np.concatenate([x, (np.arange(-512, 512) / 256.0 + 1.0 / 512).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(brute.round_bf16(x.astype(np.float64)), ref)


# ------------------------------------------------------------------ attention backward

def _fd_check(lens, H, d, theta, seed, Hkv=None):
    rng = np.random.default_rng(seed)
    w = synth.custom_workload(lens, H, d)
    T = w.total
    Hkv = H if Hkv is None else Hkv
    q, g = (rng.standard_normal((T, H, d)) for _ in range(2))
    k, v = (rng.standard_normal((T, Hkv, d)) for _ in range(2))
    dq, dk, dv = oracle.attn_bwd_f64(g, q, k, v, w.cu, theta=theta)
    eps = 1e-6

    def f(qq, kk, vv):
        o, _ = oracle.attn_fwd_f64(qq, kk, vv, w.cu, theta=theta)
        return float(np.sum(o * g))

    for name, x, gx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        idx = [tuple(rng.integers(0, s) for s in x.shape) for _ in range(12)]
        for ix in idx:
            xp, xm = x.copy(), x.copy()
            xp[ix] += eps
            xm[ix] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num = (f(*args_p) - f(*args_m)) / (2 * eps)
            assert abs(num - gx[ix]) < 1e-6 * (1 + abs(num)), (name, ix, num, gx[ix])


@pytest.mark.parametrize("theta", [0.0, 10000.0])
def test_backward_finite_differences(theta):
    """charlestar, 'change A, B must not change' (its CPU recheck uses finite differences
    for the Q/K/V gradients)."""
    _fd_check([3, 1, 5], 2, 8, theta, seed=7)


@pytest.mark.parametrize("theta", [0.0, 10000.0])
def test_backward_finite_differences_grouped_heads(theta):
    # four query heads sharing two key/value heads: dK and dV sum the group's contributions
    _fd_check([4, 2, 3], 4, 8, theta, seed=8, Hkv=2)


def _rope_torch(x, pos, d, theta=10000.0):
    half = d // 2
    wfreq = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones(len(pos), half, dtype=torch.float64), pos[:, None] * wfreq[None])
    z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


@pytest.mark.parametrize("H,Hkv", [(4, 2), (8, 1), (6, 3)])
def test_grouped_heads_against_torch_sdpa_autograd(H, Hkv):
    # torch fp64 SDPA with enable_gqa (query head h reads key/value head h // (H // Hkv)) and a
    # boolean block mask, differentiated by autograd, against the oracle's forward and backward
    lens = [5, 1, 7, 3]
    d = 16
    w = synth.custom_workload(lens, H, d)
    g0 = torch.Generator().manual_seed(31)
    q, g = (torch.randn((w.total, H, d), generator=g0).bfloat16() for _ in range(2))
    k, v = (torch.randn((w.total, Hkv, d), generator=g0).bfloat16() for _ in range(2))
    pos = torch.from_numpy(brute.local_positions(w.cu)).double()
    qt, kt, vt = (torch.from_numpy(_f64(x)).requires_grad_() for x in (q, k, v))
    mask = torch.from_numpy(brute.block_causal_allow(w.cu))
    o = torch.nn.functional.scaled_dot_product_attention(
        _rope_torch(qt, pos, d).permute(1, 0, 2), _rope_torch(kt, pos, d).permute(1, 0, 2),
        vt.permute(1, 0, 2), attn_mask=mask, enable_gqa=True).permute(1, 0, 2)
    (o * torch.from_numpy(_f64(g))).sum().backward()
    o_orc, _ = oracle.attn_fwd(q, k, v, w.cu, contract=False)
    assert np.max(np.abs(o_orc - o.detach().numpy())) < 1e-12
    dq, dk, dv = oracle.attn_bwd(g, q, k, v, w.cu, contract=False)
    assert dk.shape == (w.total, Hkv, d)
    assert np.max(np.abs(dq - qt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dk - kt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dv - vt.grad.numpy())) < 1e-11


def test_backward_against_torch_autograd():
    """Whole-pack torch fp64 autograd (complex-form RoPE, boolean-mask SDPA) vs the oracle."""
    lens = [5, 2, 9]
    w, (q, k, v, g) = _rand_qkv(lens, 2, 16, seed=12, with_grad=True)
    pos = torch.from_numpy(brute.local_positions(w.cu)).double()
    qt = torch.from_numpy(_f64(q)).requires_grad_()
    kt = torch.from_numpy(_f64(k)).requires_grad_()
    vt = torch.from_numpy(_f64(v)).requires_grad_()
    half = 8
    wfreq = 10000.0 ** (-2.0 * torch.arange(half, dtype=torch.float64) / 16)
    rot = torch.polar(torch.ones(len(pos), half, dtype=torch.float64), pos[:, None] * wfreq[None])

    def rope(x):
        z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    mask = torch.from_numpy(brute.block_causal_allow(w.cu))
    o = torch.nn.functional.scaled_dot_product_attention(
        rope(qt).permute(1, 0, 2), rope(kt).permute(1, 0, 2), vt.permute(1, 0, 2), attn_mask=mask
    ).permute(1, 0, 2)
    (o * torch.from_numpy(_f64(g))).sum().backward()
    dq, dk, dv = oracle.attn_bwd(g, q, k, v, w.cu, contract=False)
    assert np.max(np.abs(dq - qt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dk - kt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dv - vt.grad.numpy())) < 1e-11


def test_backward_seg_heads_subset_matches_full():
    lens = [4, 9, 3]
    w, (q, k, v, g) = _rand_qkv(lens, 2, 8, seed=13, with_grad=True)
    full = oracle.attn_bwd(g, q, k, v, w.cu)
    part = oracle.attn_bwd(g, q, k, v, w.cu, seg_heads=[(1, 1), (2, 0)])
    for a, b in zip(full, part):
        assert np.array_equal(a[4:13, 1], b[4:13, 1])
        assert np.array_equal(a[13:16, 0], b[13:16, 0])
        assert not b[:4].any()


def test_backward_isolation():
    """Gradients of one segment do not depend on another segment's inputs."""
    lens = [3, 2, 4]
    w, (q, k, v, g) = _rand_qkv(lens, 1, 8, seed=14, with_grad=True)
    base = oracle.attn_bwd(g, q, k, v, w.cu)
    q2 = q.clone()
    q2[:3] = -q2[:3]
    alt = oracle.attn_bwd(g, q2, k, v, w.cu)
    for a, b in zip(base, alt):
        assert np.array_equal(a[3:], b[3:])


# ------------------------------------------------------------------ work lists

def _allowed_tiles(cu, BM, BN):
    """Brute force: every (seg, q_tile, kv_tile) holding at least one allowed pair."""
    tiles = set()
    for r in range(len(cu) - 1):
        L = cu[r + 1] - cu[r]
        for i in range(L):
            for j in range(i + 1):
                tiles.add((r, i // BM, j // BN))
    return tiles


@pytest.mark.parametrize("BM,BN", [(128, 128), (64, 128), (128, 64), (16, 16), (16, 32)])
def test_worklists_cover_exactly_the_allowed_tiles(BM, BN):
    """No item touches another segment or a tile wholly above the diagonal, and every
    allowed (query, key) pair lies in exactly one forward and one backward tile."""
    rng = np.random.default_rng(BM * 7 + BN)
    lens = np.concatenate([rng.integers(1, 300, size=12), [1, BM, BM + 1, BN - 1 if BN > 1 else 1]])
    cu = np.concatenate([[0], np.cumsum(lens)])
    want = _allowed_tiles(cu, BM, BN)
    fwd = oracle.worklist_fwd(cu, BM, BN)
    got_f = []
    for s, qt, lo, hi in fwd:
        got_f += [(s, qt, kt) for kt in range(lo, hi)]
    assert len(got_f) == len(set(got_f)) and set(got_f) == want
    bwd = oracle.worklist_bwd(cu, BM, BN)
    got_b = []
    for s, kt, lo, hi in bwd:
        got_b += [(s, qt, kt) for qt in range(lo, hi)]
    assert len(got_b) == len(set(got_b)) and set(got_b) == want
    # one forward item per q tile, one backward item per kv tile
    assert len(fwd) == int(np.sum(-(-lens // BM)))
    assert len(bwd) == int(np.sum(-(-lens // BN)))


def test_worklist_order():
    """Longest segments first (stable on ties), longest key range first inside a segment."""
    lens = np.array([100, 300, 129, 256, 300, 1, 257])
    cu = np.concatenate([[0], np.cumsum(lens)])
    fwd = oracle.worklist_fwd(cu, 128, 128)
    nq = -(-lens // 128)
    seg_seq = [s for s, *_ in fwd]
    firsts = list(dict.fromkeys(seg_seq))
    assert firsts == sorted(range(len(lens)), key=lambda r: (-nq[r], r))
    for r in range(len(lens)):
        qts = [qt for s, qt, _, _ in fwd if s == r]
        assert qts == list(range(nq[r] - 1, -1, -1))
    bwd = oracle.worklist_bwd(cu, 128, 128)
    for r in range(len(lens)):
        kts = [kt for s, kt, _, _ in bwd if s == r]
        assert kts == list(range(nq[r]))


def test_forward_seg_heads_subset_matches_full():
    lens = [4, 9, 3]
    w, (q, k, v) = _rand_qkv(lens, 2, 8, seed=15)
    o, lse = oracle.attn_fwd(q, k, v, w.cu)
    o2, lse2 = oracle.attn_fwd(q, k, v, w.cu, seg_heads=[(1, 1), (2, 0)])
    assert np.array_equal(o2[4:13, 1], o[4:13, 1]) and np.array_equal(lse2[1, 4:13], lse[1, 4:13])
    assert np.array_equal(o2[13:16, 0], o[13:16, 0]) and not o2[:4].any()


# ------------------------------------------------------------------ shifted cross-entropy (next row)
def test_ce_uniform_logits_closed_form():
    # uniform logits: every valid target costs ln(vocab)
    V = 37
    z = np.zeros((11, V))
    lab = np.array([0, 5, -100, 36, 1, 2, -100, 3, 4, 9, -100], dtype=np.int64)
    st, s, n, sl, sc = oracle.shifted_ce(z, lab, [0, 3, 7, 11])
    assert st == 0 and n == 8
    assert s == pytest.approx(8 * math.log(V), rel=1e-13)
    assert list(sc) == [2, 3, 3]
    assert sl == pytest.approx([2 * math.log(V), 3 * math.log(V), 3 * math.log(V)], rel=1e-13)


def test_ce_token_mean_vs_sample_mean_example():
    # charlestar, "Packing should not decide how much a long sample weighs": A has 2 targets
    # of loss 1, B has 6 of loss 3; token mean (2 + 18) / 8 = 2.5, sample mean (1 + 3) / 2 = 2.
    def row(loss):   # two classes, label 1: CE = ln(1 + e^a) = loss
        return [math.log(math.expm1(loss)), 0.0]
    z = np.array([row(1.0)] * 3 + [row(3.0)] * 7)
    lab = np.array([1, 1, -100] + [1] * 6 + [-100], dtype=np.int64)
    st, s, n, sl, sc = oracle.shifted_ce(z, lab, [0, 3, 10])
    assert st == 0 and list(sc) == [2, 6]
    assert sl == pytest.approx([2.0, 18.0], rel=1e-12)
    assert s / n == pytest.approx(2.5, rel=1e-12)
    assert np.mean(sl / sc) == pytest.approx(2.0, rel=1e-12)


def test_ce_against_torch_cross_entropy():
    # an independent library routine: torch's fp64 cross_entropy with ignore_index = -100
    rng = np.random.default_rng(7)
    T, V = 64, 301
    z = rng.normal(0, 3, size=(T, V))
    lab = rng.integers(0, V, size=T)
    lab[rng.random(T) < 0.2] = -100
    st, s, n, _, _ = oracle.shifted_ce(z, lab)
    ref = torch.nn.functional.cross_entropy(torch.from_numpy(z), torch.from_numpy(lab), ignore_index=-100,
                                            reduction="sum").item()
    assert st == 0 and n == int((lab != -100).sum())
    assert s == pytest.approx(ref, rel=1e-12)


def test_ce_preshifted_equals_internal_shift():
    # charlestar, "After isolation one cross-boundary prediction pair remains": the pre-shifted
    # labels on logit row i and the internal shift (labels = tokens with -100 at every segment
    # start, logits[:-1] against labels[1:]) give the same pairs, hence the same sum and count.
    rng = np.random.default_rng(11)
    lens = [3, 1, 5, 2, 6]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, V = int(cu[-1]), 23
    tokens = rng.integers(0, V, size=T).astype(np.int64)
    z = rng.normal(0, 2, size=(T, V))
    _, lab = oracle.positions_labels(cu, tokens)
    st, s, n, sl, sc = oracle.shifted_ce(z, lab, cu)
    lab2 = tokens.copy()
    lab2[cu[:-1]] = -100
    ref = torch.nn.functional.cross_entropy(torch.from_numpy(z[:-1]), torch.from_numpy(lab2[1:]),
                                            ignore_index=-100, reduction="sum").item()
    assert st == 0 and n == int((lab2[1:] != -100).sum()) == sum(L - 1 for L in lens)
    assert s == pytest.approx(ref, rel=1e-12)
    assert list(sc) == [L - 1 for L in lens]


def test_ce_bf16_bits_and_bad_label():
    rng = np.random.default_rng(3)
    z = rng.normal(0, 2, size=(8, 40)).astype(np.float32)
    bits = oracle.bf16_bits(torch.from_numpy(z).to(torch.bfloat16))
    z64 = oracle.bits_to_f64(bits)
    lab = rng.integers(0, 40, size=8)
    a = oracle.shifted_ce(bits, lab)
    b = oracle.shifted_ce(z64, lab)
    assert a[0] == 0 and a[1] == pytest.approx(b[1], rel=1e-15) and a[2] == b[2]
    lab[3] = 40   # outside the vocabulary: flagged and not counted
    st, s, n, _, _ = oracle.shifted_ce(z64, lab)
    assert st == 1 and n == 7


# ------------------------------------------------------------------ interleaved RoPE pairing
def _rope_interleaved_np(x, pos, theta=10000.0):
    # the complex form of consecutive pairs: z_j = x_2j + i x_2j+1, times e^{i p w_j}
    d = x.shape[-1]
    w = theta ** (-2.0 * np.arange(d // 2) / d)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * np.asarray(pos, np.float64)[:, None] * w[None])
    out = np.empty_like(x)
    out[..., 0::2], out[..., 1::2] = z.real, z.imag
    return out


def test_rope_interleaved_rows_complex_form():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 16))
    pos = rng.integers(0, 5000, size=9)
    assert np.allclose(oracle.rope_rows(x, pos, interleaved=True), _rope_interleaved_np(x, pos), atol=1e-9)
    # the two pairings are the same rotation up to a permutation of the coordinates
    perm = np.concatenate([np.arange(0, 16, 2), np.arange(1, 16, 2)])   # interleaved -> halves
    a = oracle.rope_rows(x[:, perm], pos)
    b = oracle.rope_rows(x, pos, interleaved=True)[:, perm]
    assert np.allclose(a, b, atol=1e-12)


def test_interleaved_attention_against_torch_autograd():
    lens = [6, 1, 9]
    H, Hkv, d = 4, 2, 16
    w = synth.custom_workload(lens, H, d)
    g0 = torch.Generator().manual_seed(41)
    q, g = (torch.randn((w.total, H, d), generator=g0).bfloat16() for _ in range(2))
    k, v = (torch.randn((w.total, Hkv, d), generator=g0).bfloat16() for _ in range(2))
    pos = torch.from_numpy(brute.local_positions(w.cu)).double()
    wfreq = 10000.0 ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones(len(pos), d // 2, dtype=torch.float64), pos[:, None] * wfreq[None])

    def rope(x):
        z = torch.view_as_complex(x.reshape(*x.shape[:-1], d // 2, 2).contiguous()) * rot[:, None, :]
        return torch.view_as_real(z).reshape(x.shape)

    qt, kt, vt = (torch.from_numpy(_f64(x)).requires_grad_() for x in (q, k, v))
    mask = torch.from_numpy(brute.block_causal_allow(w.cu))
    o = torch.nn.functional.scaled_dot_product_attention(
        rope(qt).permute(1, 0, 2), rope(kt).permute(1, 0, 2), vt.permute(1, 0, 2), attn_mask=mask,
        enable_gqa=True).permute(1, 0, 2)
    (o * torch.from_numpy(_f64(g))).sum().backward()
    o_orc, _ = oracle.attn_fwd(q, k, v, w.cu, contract=False, interleaved=True)
    assert np.max(np.abs(o_orc - o.detach().numpy())) < 1e-12
    dq, dk, dv = oracle.attn_bwd(g, q, k, v, w.cu, contract=False, interleaved=True)
    assert np.max(np.abs(dq - qt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dk - kt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dv - vt.grad.numpy())) < 1e-11


def test_interleaved_backward_finite_differences():
    rng = np.random.default_rng(17)
    w = synth.custom_workload([4, 3], 2, 8)
    q, k, v, g = (rng.standard_normal((w.total, 2, 8)) for _ in range(4))
    dq, dk, dv = oracle.attn_bwd_f64(g, q, k, v, w.cu, interleaved=True)
    eps = 1e-6
    for name, x, gx in (("q", q, dq), ("k", k, dk)):
        for ix in [tuple(rng.integers(0, s) for s in x.shape) for _ in range(8)]:
            xp, xm = x.copy(), x.copy()
            xp[ix] += eps
            xm[ix] -= eps
            f = lambda a: float(np.sum(oracle.attn_fwd_f64(*((a, k, v) if name == "q" else (q, a, v)), w.cu,
                                                           interleaved=True)[0] * g))
            num = (f(xp) - f(xm)) / (2 * eps)
            assert abs(num - gx[ix]) < 1e-6 * (1 + abs(num)), (name, ix)


# ------------------------------------------------------------------ padded layouts (cu_padded)
def _padded_case(seed=0):
    lens = [5, 1, 9, 4]
    slots = [8, 3, 9, 7]          # slot >= length; padding after each segment
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cp = np.concatenate([[0], np.cumsum(slots)]).astype(np.int32)
    return lens, slots, cu, cp


def test_padded_attention_against_masked_torch_on_padded_rows():
    # the masked attention written directly on the padded rows: a real query sees the real
    # keys of its own slot at positions <= its own; a padding query sees only itself and its
    # output is zeroed, so nothing flows into or out of padding rows
    lens, slots, cu, cp = _padded_case()
    total, H, Hkv, d = int(cp[-1]), 4, 2, 16
    g0 = torch.Generator().manual_seed(3)
    q, g = (torch.randn((total, H, d), generator=g0).bfloat16() for _ in range(2))
    k, v = (torch.randn((total, Hkv, d), generator=g0).bfloat16() for _ in range(2))
    seg = np.repeat(np.arange(len(slots)), slots)
    pos = np.arange(total) - cp[seg]
    real = pos < np.asarray(lens)[seg]
    allow = (seg[:, None] == seg[None, :]) & (pos[None, :] <= pos[:, None]) & real[None, :] & real[:, None]
    allow |= np.diag(~real)
    posd = torch.from_numpy(pos).double()
    qt, kt, vt = (torch.from_numpy(_f64(x)).requires_grad_() for x in (q, k, v))
    rq, rk = _rope_torch(qt, posd, d), _rope_torch(kt, posd, d)
    kr, vr = (x.repeat_interleave(H // Hkv, dim=1) for x in (rk, vt))
    s = torch.einsum("ihd,jhd->hij", rq, kr) / np.sqrt(d)
    s = s.masked_fill(~torch.from_numpy(allow)[None], float("-inf"))
    lse_t = torch.logsumexp(s, dim=-1)
    o = torch.einsum("hij,jhd->ihd", torch.softmax(s, dim=-1), vr) * torch.from_numpy(real)[:, None, None]
    (o * torch.from_numpy(_f64(g))).sum().backward()
    o_orc, lse_orc = oracle.attn_fwd(q, k, v, cu, contract=False, cu_padded=cp)
    assert np.max(np.abs(o_orc - o.detach().numpy())) < 1e-12
    assert np.max(np.abs(lse_orc[:, real] - lse_t.detach().numpy()[:, real])) < 1e-12
    assert np.all(np.isneginf(lse_orc[:, ~real])) and np.all(o_orc[~real] == 0)
    dq, dk, dv = oracle.attn_bwd(g, q, k, v, cu, contract=False, cu_padded=cp)
    assert np.max(np.abs(dq - qt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dk - kt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dv - vt.grad.numpy())) < 1e-11
    assert np.all(dq[~real] == 0) and np.all(dk[~real] == 0) and np.all(dv[~real] == 0)


def test_padded_equals_unpadded_when_slots_are_tight():
    lens, _, cu, _ = _padded_case()
    w = synth.custom_workload(lens, 2, 16)
    rng = np.random.default_rng(8)
    q, k, v = (torch.from_numpy(rng.standard_normal((w.total, 2, 16))).bfloat16() for _ in range(3))
    a = oracle.attn_fwd(q, k, v, cu)
    b = oracle.attn_fwd(q, k, v, cu, cu_padded=cu)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    with pytest.raises(ValueError):
        oracle.real_rows(cu, np.array([0, 4, 5, 14, 18]))   # first slot shorter than its segment


# ------------------------------------------------------------------ q and kv of different lengths
def _qkv_case():
    lq = [3, 1, 6, 4]
    lk = [7, 1, 6, 9]         # Lk >= Lq; one square segment, one single-token decode step
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cuk = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return lq, lk, cu, cuk


def test_qkv_bottom_right_against_torch_autograd():
    # a mask written on the (query, key) rows directly: query p of segment r sees key j of the
    # same segment iff j <= p + (Lk - Lq); queries rotate at position p + Lk - Lq, keys at j
    lq, lk, cu, cuk = _qkv_case()
    Tq, Tk, H, Hkv, d = int(cu[-1]), int(cuk[-1]), 4, 2, 16
    g0 = torch.Generator().manual_seed(12)
    q, g = (torch.randn((Tq, H, d), generator=g0).bfloat16() for _ in range(2))
    k, v = (torch.randn((Tk, Hkv, d), generator=g0).bfloat16() for _ in range(2))
    sq, sk = np.repeat(np.arange(len(lq)), lq), np.repeat(np.arange(len(lk)), lk)
    off = (np.asarray(lk) - np.asarray(lq))[sq]
    pq = np.arange(Tq) - cu[sq] + off
    pk = np.arange(Tk) - cuk[sk]
    allow = (sq[:, None] == sk[None, :]) & (pk[None, :] <= pq[:, None])
    qt, kt, vt = (torch.from_numpy(_f64(x)).requires_grad_() for x in (q, k, v))
    rq = _rope_torch(qt, torch.from_numpy(pq).double(), d)
    rk = _rope_torch(kt, torch.from_numpy(pk).double(), d)
    o = torch.nn.functional.scaled_dot_product_attention(
        rq.permute(1, 0, 2), rk.permute(1, 0, 2), vt.permute(1, 0, 2), attn_mask=torch.from_numpy(allow),
        enable_gqa=True).permute(1, 0, 2)
    (o * torch.from_numpy(_f64(g))).sum().backward()
    o_orc, lse_orc = oracle.attn_fwd(q, k, v, cu, contract=False, cu_kv=cuk)
    assert np.max(np.abs(o_orc - o.detach().numpy())) < 1e-12
    s = torch.einsum("ihd,jhd->hij", rq.detach(), rk.detach().repeat_interleave(H // Hkv, 1)) / np.sqrt(d)
    lse_t = torch.logsumexp(s.masked_fill(~torch.from_numpy(allow)[None], float("-inf")), -1).numpy()
    assert np.max(np.abs(lse_orc - lse_t)) < 1e-12
    dq, dk, dv = oracle.attn_bwd(g, q, k, v, cu, contract=False, cu_kv=cuk)
    assert dk.shape == (Tk, Hkv, d)
    assert np.max(np.abs(dq - qt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dk - kt.grad.numpy())) < 1e-11
    assert np.max(np.abs(dv - vt.grad.numpy())) < 1e-11


def test_qkv_single_query_with_zero_q_averages_all_values():
    # Lq = 1: the one query sees every key; with q = 0 all scores are 0, so O is the mean of V
    lk = [5, 8]
    cu = np.array([0, 1, 2], np.int32)
    cuk = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    rng = np.random.default_rng(3)
    v = rng.standard_normal((13, 2, 8))
    o, lse = oracle.attn_fwd_f64(np.zeros((2, 2, 8)), rng.standard_normal((13, 2, 8)), v, cu, cu_kv=cuk)
    assert np.allclose(o[0], v[:5].mean(0), atol=1e-14) and np.allclose(o[1], v[5:].mean(0), atol=1e-14)
    assert np.allclose(lse[:, 0], np.log(5)) and np.allclose(lse[:, 1], np.log(8))


def test_qkv_queries_equal_the_tail_of_a_self_attention():
    # the last Lq rows of a self-attention over the Lk-token segment, asked as Lq queries
    # against all Lk keys, give the same outputs and gradients (dk, dv: their share)
    lk, lq = [9, 4], [3, 4]
    cuk = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    rng = np.random.default_rng(21)
    qf, k, v, gf = (rng.standard_normal((13, 2, 8)) for _ in range(4))
    tail = np.concatenate([np.arange(a - n, a) for a, n in zip(cuk[1:], lq)])
    gz = np.zeros_like(gf)
    gz[tail] = gf[tail]
    o_self, lse_self = oracle.attn_fwd_f64(qf, k, v, cuk)
    o, lse = oracle.attn_fwd_f64(qf[tail], k, v, cu, cu_kv=cuk)
    assert np.allclose(o, o_self[tail], atol=1e-13) and np.allclose(lse, lse_self[:, tail], atol=1e-13)
    dq_s, dk_s, dv_s = oracle.attn_bwd_f64(gz, qf, k, v, cuk)
    dq, dk, dv = oracle.attn_bwd_f64(gf[tail], qf[tail], k, v, cu, cu_kv=cuk)
    assert np.allclose(dq, dq_s[tail], atol=1e-12)
    assert np.allclose(dk, dk_s, atol=1e-12) and np.allclose(dv, dv_s, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.attn_fwd_f64(qf, k, v, cuk, cu_kv=cu)     # more queries than keys


def test_qkv_rows_sampler_matches_the_full_forward():
    lq, lk, cu, cuk = _qkv_case()
    rng = np.random.default_rng(2)
    q = torch.from_numpy(rng.standard_normal((int(cu[-1]), 2, 16))).bfloat16()
    k, v = (torch.from_numpy(rng.standard_normal((int(cuk[-1]), 2, 16))).bfloat16() for _ in range(2))
    o, lse = oracle.attn_fwd(q, k, v, cu, cu_kv=cuk)
    rows, heads = np.arange(int(cu[-1])), np.arange(int(cu[-1])) % 2
    o_r, lse_r = oracle.attn_fwd_rows(q, k, v, cu, rows, heads, cu_kv=cuk)
    assert np.array_equal(o_r, o[rows, heads]) and np.array_equal(lse_r, lse[heads, rows])


# ------------------------------------------------------------------ host packing (oracle/packing.py)
from oracle import packing  # noqa: E402


@pytest.mark.parametrize("name", ["table_4_1_example_A", "table_4_1_example_B"])
def test_ffd_reaches_the_pages_lower_bound_examples(name):
    # the worked examples of "Long-context training: remove padding": ceil(T/L) = 2 windows,
    # and the printed padding / saved slot numbers follow from the windows FFD builds
    g = _golden("ledgers.json")[name]
    L, lens = g["L"], g["lengths"]
    bin_of, order, bin_start = packing.ffd(lens, L)
    nbins = len(bin_start) - 1
    assert nbins == g["packs"] == math.ceil(g["T"] / L)
    assert nbins * L == g["packed"]
    assert nbins * L - sum(lens) == g["pack_padding"]
    assert g["fixed"] - nbins * L == g["saved"]
    assert round(100 * (1 - packing.eta(lens, nbins, L)), 1) == round(100 * g["pack_padding"] / g["packed"], 1)
    fills = packing.pack_costs(lens, order, bin_start, "tokens")
    assert fills.max() <= L and sorted(order.tolist()) == list(range(len(lens)))


def test_ffd_on_example_b_by_hand():
    # 1024 opens window 0, 768 joins it (256 left), 512 opens window 1, 256 fills window 0,
    # 96 joins window 1
    _, order, bin_start = packing.ffd([1024, 768, 512, 256, 96], 2048)
    assert [order[bin_start[b]:bin_start[b + 1]].tolist() for b in range(2)] == [[0, 1, 3], [2, 4]]


def test_packers_against_exhaustive_optimum():
    # textbook bounds against the exhaustive optimum OPT: ceil(T/L) <= OPT <= FFD <= 11/9 OPT + 6/9,
    # first-fit <= 1.7 OPT (+1 slack for small cases), next-fit <= 2 OPT
    rng = np.random.default_rng(0)
    worst_ffd = 0.0
    for _ in range(60):
        n = int(rng.integers(3, 8))
        cap = int(rng.integers(10, 21))
        lens = [int(x) for x in rng.integers(1, cap + 1, size=n)]
        opt = packing.brute_min_bins(lens, cap)
        assert math.ceil(sum(lens) / cap) <= opt
        nb = {f.__name__: len(f(lens, cap)[2]) - 1 for f in (packing.ffd, packing.first_fit, packing.next_fit)}
        assert opt <= nb["ffd"] <= math.floor(11 * opt / 9 + 6 / 9)
        assert opt <= nb["first_fit"] <= math.floor(1.7 * opt) + 1
        assert opt <= nb["next_fit"] <= 2 * opt
        worst_ffd = max(worst_ffd, nb["ffd"] / opt)
    # a family where first-fit in arrival order (small items first) is poor and FFD optimal
    lens = [2, 2, 2, 7, 7, 7]
    assert len(packing.ffd(lens, 9)[2]) - 1 == packing.brute_min_bins(lens, 9) == 3
    assert len(packing.first_fit(lens, 9)[2]) - 1 == 4


def test_oversize_samples_get_a_window_of_their_own():
    lens = [10, 3, 25, 4, 12]
    bin_of, order, bin_start = packing.ffd(lens, 12, extra=1)   # 25 + 1 and 12 + 1 exceed 12
    assert packing.oversize_count(lens, 12, extra=1) == 2
    for i in (2, 4):
        w = bin_of[i]
        assert bin_start[w + 1] - bin_start[w] == 1
    sizes = np.asarray(lens) + 1
    for b in range(len(bin_start) - 1):
        members = order[bin_start[b]:bin_start[b + 1]]
        assert len(members) == 1 or sizes[members].sum() <= 12


def test_lpt_against_exhaustive_makespan():
    # Graham's bound for longest-processing-time: LPT <= (4/3 - 1/(3R)) OPT
    rng = np.random.default_rng(1)
    for _ in range(60):
        R = int(rng.integers(2, 4))
        costs = [int(x) for x in rng.integers(1, 50, size=int(rng.integers(R, 8)))]
        rank_of, load = packing.lpt(costs, R)
        assert np.array_equal(np.bincount(rank_of, weights=costs, minlength=R).astype(np.int64), load)
        opt = packing.brute_min_makespan(costs, R)
        assert opt <= load.max() <= (4 / 3 - 1 / (3 * R)) * opt + 1e-9


def test_sum_of_squares_balance_beats_token_balance():
    # charlestar's point: equal token counts can hide unequal attention work; two ranks, one
    # pack of a single 4096-token document and four packs of 1024 short ones (4096 tokens each)
    lens = [4096] + [256] * 64
    bin_of, order, bin_start = packing.ffd(lens, 4096)
    tok = packing.pack_costs(lens, order, bin_start, "tokens")
    sq = packing.pack_costs(lens, order, bin_start, "sumsq")
    assert len(tok) == 5 and np.all(tok == 4096)
    by_tok, _ = packing.lpt(tok, 2)
    by_sq, load_sq = packing.lpt(sq, 2)
    work_tok = np.bincount(by_tok, weights=sq, minlength=2)
    assert load_sq.max() == 4096 ** 2 and load_sq.max() < work_tok.max()
