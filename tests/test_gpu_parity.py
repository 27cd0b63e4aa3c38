"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Integer outputs (positions, labels, work lists, error bits) must match
bit-exactly.  Attention is compared on the same bf16 inputs against the
oracle's contract mode (rotated q/k rounded to bf16), with the stated bounds:
O max |err| <= 2e-2 and mean |err| <= 2e-3, LSE max |err| <= 1e-3, gradients
max |err| <= 5e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from variable_length_causal_gb300 import synth

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX, G_MAX = 2e-2, 2e-3, 1e-3, 5e-2


@pytest.fixture(scope="module")
def vlc():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as m

    m.load_library()
    return m


DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def _cu(w):
    return torch.from_numpy(w.cu).to(DEV)


def _cmp_fwd(o, lse, o_ref, lse_ref, rows=None):
    og = o.float().cpu().numpy()
    lg = lse.cpu().numpy()
    if rows is not None:
        r, h = rows
        og = og[r, h]
        lg = lg[h, r]
    eo = np.abs(og - o_ref)
    el = np.abs(lg - lse_ref)
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    assert eo.max() <= O_MAX, f"O max err {eo.max()}"
    assert eo.mean() <= O_MEAN, f"O mean err {eo.mean()}"
    assert el.max() <= LSE_MAX, f"LSE max err {el.max()}"
    return eo.max(), eo.mean(), el.max()


# ------------------------------------------------------------------ positions and labels

@pytest.mark.parametrize("idx", range(5))
def test_positions_labels_configs(vlc, idx):
    w = synth.workload(idx)
    tok = synth.make_tokens(w)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pos, lab = vlc.build_positions_labels(_cu(w), torch.from_numpy(tok).to(DEV),
                                          torch.from_numpy(w.seg_ignore).to(DEV), err=err)
    pr, lr = oracle.positions_labels(w.cu, tok, w.seg_ignore)
    assert np.array_equal(pos.cpu().numpy(), pr)
    assert np.array_equal(lab.cpu().numpy(), lr)
    assert int(err.item()) == 0


@pytest.mark.parametrize("lens", [[1], [9], [3, 2, 4], [1, 1, 1, 1, 1], [5, 1, 7, 1, 2, 3, 8, 1, 1]])
def test_positions_labels_edges(vlc, lens):
    w = synth.custom_workload(lens, 1, 64)
    tok = np.arange(w.total, dtype=np.int64) * 7 + 3
    pos, lab = vlc.build_positions_labels(_cu(w), torch.from_numpy(tok).to(DEV))
    pr, lr = oracle.positions_labels(w.cu, tok)
    assert np.array_equal(pos.cpu().numpy(), pr) and np.array_equal(lab.cpu().numpy(), lr)


def test_positions_labels_random_many_segments(vlc):
    rng = np.random.default_rng(17)
    lens = rng.integers(1, 50, size=3000)
    w = synth.custom_workload(lens, 1, 64)
    tok = rng.integers(0, 50000, size=w.total)
    ign = (rng.random(len(lens)) < 0.1).astype(np.uint8)
    pos, lab = vlc.build_positions_labels(_cu(w), torch.from_numpy(tok).to(DEV),
                                          torch.from_numpy(ign).to(DEV))
    pr, lr = oracle.positions_labels(w.cu, tok, ign)
    assert np.array_equal(pos.cpu().numpy(), pr) and np.array_equal(lab.cpu().numpy(), lr)


@pytest.mark.parametrize("cu,total", [([1, 3, 5, 9], 9), ([0, 3, 3, 9], 9), ([0, 5, 3, 9], 9),
                                      ([0, 3, 5, 9], 10)])
def test_positions_labels_error_bits(vlc, cu, total):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    tok = torch.arange(total, dtype=torch.int64, device=DEV)
    vlc.build_positions_labels(cu_t, tok, err=err)
    want = oracle.validate_cu(cu, total, max(np.diff(cu))) & ~oracle.ERR_MAXLEN
    assert int(err.item()) == want


# ------------------------------------------------------------------ work lists

def _wl_cases():
    out = [synth.workload(i).cu for i in range(4)]
    rng = np.random.default_rng(3)
    for _ in range(3):
        lens = rng.integers(1, 600, size=int(rng.integers(1, 400)))
        out.append(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    out.append(np.array([0, 1], np.int32))
    out.append(np.concatenate([[0], np.cumsum([128, 128, 127, 129, 1, 256, 255])]).astype(np.int32))
    return out


@pytest.mark.parametrize("ci", range(9))
@pytest.mark.parametrize("kind,BM,BN", [(0, 128, 128), (1, 64, 128), (0, 64, 64), (1, 128, 64)])
def test_worklist_bit_exact(vlc, ci, kind, BM, BN):
    cu = _wl_cases()[ci]
    lens = np.diff(cu)
    items, order, bits = vlc.build_worklist(torch.from_numpy(cu).to(DEV), int(cu[-1]), int(lens.max()),
                                            kind, BM, BN)
    assert bits == 0
    ref = oracle.worklist_fwd(cu, BM, BN) if kind == 0 else oracle.worklist_bwd(cu, BM, BN)
    assert np.array_equal(items.cpu().numpy(), ref)
    nseg = len(lens)
    o = order.cpu().numpy()
    seg_seq = list(dict.fromkeys(ref[:, 0].tolist()))
    assert o[:nseg].tolist() == seg_seq
    tile = BM if kind == 0 else BN
    n_sorted = -(-lens[o[:nseg]] // tile)
    assert o[nseg:].tolist() == np.concatenate([[0], np.cumsum(n_sorted)]).tolist()


@pytest.mark.parametrize("cu,total,maxlen", [([1, 3, 5, 9], 9, 4), ([0, 3, 3, 9], 9, 6),
                                             ([0, 5, 3, 9], 9, 6), ([0, 3, 5, 9], 10, 4),
                                             ([0, 3, 5, 9], 9, 5), ([0, 3, 5, 9], 9, 3)])
def test_worklist_validation_bits(vlc, cu, total, maxlen):
    items, _, bits = vlc.build_worklist(torch.tensor(cu, dtype=torch.int32, device=DEV), total, maxlen)
    assert bits == oracle.validate_cu(cu, total, maxlen)
    assert items.shape[0] == 0


# ------------------------------------------------------------------ forward attention

TINY_CASES = [
    ([3, 2, 4], 2, 64, 10000.0),
    ([1], 1, 128, 10000.0),
    ([1, 1, 1], 3, 128, 10000.0),
    ([127, 128, 129], 2, 128, 10000.0),
    ([255, 256, 257, 1, 2], 2, 128, 10000.0),
    ([300, 17, 513], 3, 64, 10000.0),
    ([200, 55, 140], 2, 128, 0.0),
    ([640], 1, 128, 500.0),
]


@pytest.mark.parametrize("lens,H,d,theta", TINY_CASES)
def test_fwd_small(vlc, lens, H, d, theta):
    w = synth.custom_workload(lens, H, d)
    q, k, v = synth.make_tensors(w, seed=sum(lens) + H + d)
    o, lse = vlc.varlen_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), _cu(w), w.max_seqlen, rope_theta=theta)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.cu, theta=theta)
    _cmp_fwd(o, lse, o_ref, lse_ref)


def test_fwd_tiny_config_full(vlc):
    w = synth.workload(0)
    q, k, v = synth.make_tensors(w)
    o, lse = vlc.varlen_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), _cu(w), w.max_seqlen)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.cu)
    _cmp_fwd(o, lse, o_ref, lse_ref)


def test_fwd_zero_queries_closed_form(vlc):
    """Q = 0: LSE_i = ln(p_i + 1) and O_i = mean of the segment's V rows 0..p_i."""
    w = synth.custom_workload([1, 7, 130, 3], 2, 128)
    _, k, v = synth.make_tensors(w, seed=5)
    q = torch.zeros_like(k)
    o, lse = vlc.varlen_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), _cu(w), w.max_seqlen)
    pos = np.concatenate([np.arange(L) for L in w.lengths])
    assert np.abs(lse.cpu().numpy() - np.log(pos + 1.0)[None]).max() <= LSE_MAX
    o_ref, _ = oracle.attn_fwd(q, k, v, w.cu)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_MAX


def test_fwd_isolation_bitwise(vlc):
    """Change A's q/k/v: every other segment's O and LSE stay bit-identical
    (charlestar, 'change A, B must not change')."""
    w = synth.custom_workload([200, 3, 129, 60], 2, 128)
    q, k, v = (t.to(DEV) for t in synth.make_tensors(w, seed=9))
    o1, l1 = vlc.varlen_attn_fwd(q, k, v, _cu(w), w.max_seqlen)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    for t in (q2, k2, v2):
        t[:200] = torch.randn_like(t[:200].float()).bfloat16()
    o2, l2 = vlc.varlen_attn_fwd(q2, k2, v2, _cu(w), w.max_seqlen)
    assert torch.equal(o1[200:], o2[200:]) and torch.equal(l1[:, 200:], l2[:, 200:])
    assert not torch.equal(o1[:200], o2[:200])


def test_fwd_packed_equals_per_sample_bitwise(vlc):
    """Tiles are segment-local, so a segment computes the same bits alone or packed."""
    lens = [131, 5, 300]
    w = synth.custom_workload(lens, 2, 128)
    q, k, v = (t.to(DEV) for t in synth.make_tensors(w, seed=10))
    o, lse = vlc.varlen_attn_fwd(q, k, v, _cu(w), w.max_seqlen)
    for r, L in enumerate(lens):
        a, b = int(w.cu[r]), int(w.cu[r + 1])
        cu1 = torch.tensor([0, L], dtype=torch.int32, device=DEV)
        o1, l1 = vlc.varlen_attn_fwd(q[a:b].contiguous(), k[a:b].contiguous(), v[a:b].contiguous(), cu1, L)
        assert torch.equal(o1, o[a:b]) and torch.equal(l1, lse[:, a:b])


def test_fwd_bad_cu_is_reported_and_noop(vlc):
    w = synth.custom_workload([3, 2, 4], 1, 64)
    q, k, v = (t.to(DEV) for t in synth.make_tensors(w, seed=1))
    bad = torch.tensor([0, 4, 3, 9], dtype=torch.int32, device=DEV)
    o = torch.full_like(q, 7.0)
    with pytest.raises(vlc.VlcError) as ei:
        vlc.varlen_attn_fwd(q, k, v, bad, 4, out=o)
    assert ei.value.bits & 0x2
    assert torch.all(o == 7.0)


def _sample_rows(w, n, rng):
    """Rows near segment starts/ends and tile edges, plus random ones (real segments)."""
    rows = []
    real = np.nonzero(w.seg_ignore == 0)[0]
    for r in rng.choice(real, size=min(len(real), n // 2), replace=False):
        a, b = int(w.cu[r]), int(w.cu[r + 1])
        cand = [a, b - 1, a + min(127, b - a - 1), a + min(128, b - a - 1), (a + b) // 2]
        rows.append(cand[rng.integers(len(cand))])
    rows += list(rng.integers(0, w.total, size=n - len(rows)))
    heads = rng.integers(0, w.H, size=len(rows))
    return np.asarray(rows, np.int64), heads


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_fwd_full_size_sampled(vlc, idx):
    """Full-size workloads in the bench's launch configuration; sampled rows against the oracle."""
    w = synth.workload(idx)
    q, k, v = synth.make_tensors(w, device=DEV)
    o, lse = vlc.varlen_attn_fwd(q, k, v, _cu(w), w.max_seqlen)
    rng = np.random.default_rng(100 + idx)
    rows, heads = _sample_rows(w, 48, rng)
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    o_ref, lse_ref = oracle.attn_fwd_rows(qc, kc, vc, w.cu, rows, heads)
    _cmp_fwd(o, lse, o_ref, lse_ref, rows=(rows, heads))
    # properties that hold at any size: finite everywhere, LSE >= max score bound ln(1) for row 0
    assert torch.isfinite(lse).all()
    starts = torch.from_numpy(w.cu[:-1].astype(np.int64)).to(DEV)
    # a segment's first row attends only to itself: O equals V there
    assert torch.allclose(o[starts].float(), v[starts].float(), atol=1e-2)


# ------------------------------------------------------------------ backward

def _cmp_grads(got, want, rows=None):
    out = []
    for name, g, r in zip(("dq", "dk", "dv"), got, want):
        gg = g.float().cpu().numpy()
        if rows is not None:
            gg, r = gg[rows], r[rows]
        assert np.isfinite(gg).all(), name
        e = np.abs(gg - r).max()
        assert e <= G_MAX, f"{name} max err {e}"
        out.append(e)
    return out


BWD_CASES = [
    ([3, 2, 4], 2, 64, 10000.0),
    ([1], 1, 128, 10000.0),
    ([127, 128, 129], 2, 128, 10000.0),
    ([255, 1, 257, 64, 65], 2, 128, 10000.0),
    ([300, 17, 200], 2, 64, 10000.0),
    ([190, 66], 2, 128, 0.0),
]


@pytest.mark.parametrize("lens,H,d,theta", BWD_CASES)
def test_bwd_small(vlc, lens, H, d, theta):
    w = synth.custom_workload(lens, H, d)
    q, k, v, g = synth.make_tensors(w, seed=3 * sum(lens) + d, with_grad=True)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    o, lse = vlc.varlen_attn_fwd(qd, kd, vd, _cu(w), w.max_seqlen, rope_theta=theta)
    grads = vlc.varlen_attn_bwd(gd, qd, kd, vd, o, lse, _cu(w), w.max_seqlen, rope_theta=theta)
    ref = oracle.attn_bwd(g, q, k, v, w.cu, theta=theta)
    _cmp_grads(grads, ref)


def test_bwd_tiny_config_full(vlc):
    w = synth.workload(0)
    q, k, v, g = synth.make_tensors(w, with_grad=True)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    o, lse = vlc.varlen_attn_fwd(qd, kd, vd, _cu(w), w.max_seqlen)
    grads = vlc.varlen_attn_bwd(gd, qd, kd, vd, o, lse, _cu(w), w.max_seqlen)
    _cmp_grads(grads, oracle.attn_bwd(g, q, k, v, w.cu))


def test_bwd_isolation_and_determinism(vlc):
    w = synth.custom_workload([150, 3, 140], 2, 128)
    q, k, v, g = (t.to(DEV) for t in synth.make_tensors(w, seed=21, with_grad=True))
    o, lse = vlc.varlen_attn_fwd(q, k, v, _cu(w), w.max_seqlen)
    a = vlc.varlen_attn_bwd(g, q, k, v, o, lse, _cu(w), w.max_seqlen)
    b = vlc.varlen_attn_bwd(g, q, k, v, o, lse, _cu(w), w.max_seqlen)
    for x, y in zip(a, b):
        assert torch.equal(x, y)          # no atomics: bitwise reproducible
    q2, g2 = q.clone(), g.clone()
    q2[:150] = -q2[:150]
    g2[:150] = 2 * g2[:150]
    o2, lse2 = vlc.varlen_attn_fwd(q2, k, v, _cu(w), w.max_seqlen)
    c = vlc.varlen_attn_bwd(g2, q2, k, v, o2, lse2, _cu(w), w.max_seqlen)
    for x, y in zip(a, c):
        assert torch.equal(x[150:], y[150:])


def test_bwd_full_size_sampled(vlc):
    """The pretraining-window fwd+bwd workload at full size; a few (segment, head) pairs
    are recomputed by the oracle and compared row by row."""
    w = synth.workload(4)
    q, k, v, g = synth.make_tensors(w, device=DEV, with_grad=True)
    o, lse = vlc.varlen_attn_fwd(q, k, v, _cu(w), w.max_seqlen)
    dq, dk, dv = vlc.varlen_attn_bwd(g, q, k, v, o, lse, _cu(w), w.max_seqlen)
    lens = w.lengths
    real = np.nonzero(w.seg_ignore == 0)[0]
    longest = int(real[np.argmax(lens[real])])
    shortest = int(real[np.argmin(lens[real])])
    mid = int(real[len(real) // 2])
    pairs = [(longest, 0), (shortest, w.H - 1), (mid, 7)]
    ref = oracle.attn_bwd(g.cpu(), q.cpu(), k.cpu(), v.cpu(), w.cu, seg_heads=pairs)
    for s, h in pairs:
        a, b = int(w.cu[s]), int(w.cu[s + 1])
        got = [t[a:b, h] for t in (dq, dk, dv)]
        want = [r[a:b, h] for r in ref]
        _cmp_grads(got, want)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()


def test_bwd_long_context_sampled(vlc):
    """The long-context buffer (131072 tokens, documents up to 20884 tokens) forward and
    backward at full size in the bench's launch configuration (q, k rotated once, both
    passes on the rotated operands); the gradients of three (segment, head) pairs are
    recomputed by the oracle: a segment of more than 8192 keys whose length is not a
    multiple of 128 (many q steps per key tile, the long-segment paths), a segment of
    exactly 128 tokens, and a mid-length segment with a ragged last tile."""
    w = synth.workload(3)
    q, k, v, g = synth.make_tensors(w, device=DEV, with_grad=True)
    cu = _cu(w)
    qr, kr = vlc.rope_qk(q, k, cu, w.max_seqlen)
    o, lse = vlc.varlen_attn_fwd(qr, kr, v, cu, w.max_seqlen, qk_rotated=True)
    dq, dk, dv = vlc.varlen_attn_bwd(g, qr, kr, v, o, lse, cu, w.max_seqlen, qk_rotated=True)
    # the self-rotating backward on the unrotated operands gives the same bits
    dq2, dk2, dv2 = vlc.varlen_attn_bwd(g, q, k, v, o, lse, cu, w.max_seqlen)
    for a, b in zip((dq, dk, dv), (dq2, dk2, dv2)):
        assert torch.equal(a, b)
    lens = w.lengths
    real = np.nonzero(w.seg_ignore == 0)[0]
    big = [int(r) for r in real if lens[r] > 8192 and lens[r] % 128 != 0]
    exact = [int(r) for r in real if lens[r] == 128]
    ragged = [int(r) for r in real if 1024 < lens[r] < 4096 and lens[r] % 128 != 0]
    assert big and exact and ragged
    pairs = [(min(big, key=lambda r: lens[r]), 5), (exact[0], w.H - 1), (ragged[0], 17)]
    assert lens[pairs[0][0]] > 8192
    ref = oracle.attn_bwd(g.cpu(), q.cpu(), k.cpu(), v.cpu(), w.cu, seg_heads=pairs)
    for s, h in pairs:
        a, b = int(w.cu[s]), int(w.cu[s + 1])
        _cmp_grads([t[a:b, h] for t in (dq, dk, dv)], [r[a:b, h] for r in ref])
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()


def test_fwd_peaky_scores_rescale_paths(vlc):
    """Rows whose max score jumps by far more than 2^8 within a tile and across tiles
    (large-magnitude q/k) exercise the in-row P rescale and the O rescale."""
    w = synth.custom_workload([300, 129, 520], 2, 128)
    q, k, v = synth.make_tensors(w, seed=44)
    g = torch.Generator().manual_seed(45)
    boost = (torch.rand(w.total, 1, 1, generator=g) < 0.05).float() * 12.0 + 1.0
    k = (k.float() * boost).bfloat16()
    q = (q.float() * 3.0).bfloat16()
    o, lse = vlc.varlen_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), _cu(w), w.max_seqlen)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.cu)
    eo = np.abs(o.float().cpu().numpy() - o_ref)
    el = np.abs(lse.cpu().numpy() - lse_ref)
    assert np.isfinite(eo).all()
    assert eo.max() <= O_MAX and eo.mean() <= O_MEAN
    # LSE magnitudes reach ~1e2 here: compare relative to the fp32 scale of the value
    assert (el / np.maximum(1.0, np.abs(lse_ref))).max() <= LSE_MAX


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("il", [False, True])
def test_fwd_rope_without_room_for_rotated_k(vlc, il, d):
    # a workspace without the optional rotated-k region: the forward falls back to the
    # instance whose RoPE warps rotate every staged q and K tile; with the full workspace
    # k is rotated once beforehand and the softmax warps rotate the q tiles
    lens = [2100, 5, 300, 129, 1]
    w = synth.custom_workload(lens, 2, d)
    q, k, v = (t.to(DEV) for t in synth.make_tensors(w, seed=78 + d))
    full = vlc.workspace_bytes(w.nseg, w.total, w.H, d, w.max_seqlen, False)
    krot_bytes = (w.total * w.H * d * 2 + 255) // 256 * 256
    small = torch.empty(full - krot_bytes, dtype=torch.uint8, device=DEV)
    o_ref, lse_ref = oracle.attn_fwd(*(t.cpu() for t in (q, k, v)), w.cu, interleaved=il)
    for ws in (small, None):
        o, lse = vlc.varlen_attn_fwd(q, k, v, _cu(w), w.max_seqlen, rope_interleaved=il, workspace=ws)
        e = o.float().cpu().numpy() - o_ref
        assert np.abs(e).max() <= 2e-2 and np.abs(e).mean() <= 2e-3
        assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("il", [False, True])
def test_fwd_bwd_with_prerotated_keys(vlc, il):
    # with room in the workspace every segment's k is rotated once before the forward (its
    # K tiles are not rotated in-kernel; the q tiles are, by the softmax warps)
    lens = [2100, 5, 300, 2048]
    w = synth.custom_workload(lens, 2, 128)
    q, k, v, g = (t.to(DEV) for t in synth.make_tensors(w, seed=77, with_grad=True))
    o, lse = vlc.varlen_attn_fwd(q, k, v, _cu(w), w.max_seqlen, rope_interleaved=il)
    qc, kc, vc, gc = (t.cpu() for t in (q, k, v, g))
    o_ref, lse_ref = oracle.attn_fwd(qc, kc, vc, w.cu, interleaved=il)
    e = (o.float().cpu().numpy() - o_ref)
    assert np.abs(e).max() <= 2e-2 and np.abs(e).mean() <= 2e-3
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3
    dq, dk, dv = vlc.varlen_attn_bwd(g, q, k, v, o, lse, _cu(w), w.max_seqlen, rope_interleaved=il)
    ref = oracle.attn_bwd(gc, qc, kc, vc, w.cu, interleaved=il)
    for a, b in zip((dq, dk, dv), ref):
        assert np.abs(a.float().cpu().numpy() - b).max() <= 5e-2
