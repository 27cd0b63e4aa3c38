"""GPU parity of the shifted cross-entropy statistics (through the C ABI) against
the fp64 oracle, on the same bf16 logits.

Counts must match exactly.  Sums are fp32 accumulations of fp32 row losses: the
bound is 1e-5 relative on a pack total plus 1e-3 absolute per segment (a
segment holds at most a few thousand targets of ~10 nats each).
"""
import numpy as np
import pytest
import torch

import oracle
from variable_length_causal_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
REL_TOTAL, ABS_SEG, REL_SEG = 1e-5, 1e-3, 1e-5


@pytest.fixture(scope="module")
def vlc():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as m

    m.load_library()
    return m


def _logits(T, V, seed, scale=2.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn((T, V), generator=g) * scale).to(torch.bfloat16)


def _labels(w, seed, vocab):
    tokens = np.random.default_rng(seed).integers(0, vocab, size=w.total).astype(np.int64)
    _, lab = oracle.positions_labels(w.cu, tokens, w.seg_ignore)
    return lab


def _check(vlc, z_cpu, lab, cu):
    z = z_cpu.to(DEV)
    labt = torch.from_numpy(lab).to(DEV)
    cut = None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).to(DEV)
    loss, cnt, sl, sc = vlc.shifted_cross_entropy(z, labt, cut, per_segment=True)
    st, ref, ref_n, ref_sl, ref_sc = oracle.shifted_ce(oracle.bf16_bits(z_cpu), lab, cu)
    assert st == 0
    assert int(cnt.item()) == ref_n
    assert np.array_equal(sc.cpu().numpy().astype(np.int64), ref_sc)
    got = sl.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref_sl) <= ABS_SEG + REL_SEG * np.abs(ref_sl)), np.abs(got - ref_sl).max()
    assert float(loss.item()) == pytest.approx(ref, rel=REL_TOTAL)
    return loss, cnt, sl, sc


@pytest.mark.parametrize("V", [1000, 1003, 8, 257])
def test_ce_small_ragged(vlc, V):
    # the tiny pack's ragged segments (lengths 1..256), one ignored; V = 1003 and 257 take
    # the unaligned scalar path, V = 8 a single vector per row
    w = synth.workload(0)
    ign = w.seg_ignore.copy()
    ign[3] = 1
    w2 = synth.custom_workload(np.diff(w.cu), w.H, w.d, seg_ignore=ign)
    lab = _labels(w2, 5, V)
    _check(vlc, _logits(w2.total, V, 17), lab, w2.cu)


def test_ce_one_segment_and_determinism(vlc):
    T, V = 700, 4096
    z = _logits(T, V, 3)
    lab = np.random.default_rng(4).integers(0, V, size=T).astype(np.int64)
    lab[::7] = -100
    a = _check(vlc, z, lab, None)
    b = vlc.shifted_cross_entropy(z.to(DEV), torch.from_numpy(lab).to(DEV), None, per_segment=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])


def test_ce_all_ignored_segment_and_extreme_logits(vlc):
    # a segment whose targets are all ignored counts 0 and sums 0; large logits stay finite
    lens = [5, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    V = 64
    z = _logits(int(cu[-1]), V, 8, scale=60.0)
    lab = np.random.default_rng(2).integers(0, V, size=int(cu[-1])).astype(np.int64)
    lab[5:14] = -100
    _, _, sl, sc = _check(vlc, z, lab, cu)
    assert int(sc[1].item()) == 0 and float(sl[1].item()) == 0.0


def test_ce_bad_label_is_reported(vlc):
    T, V = 40, 128
    z = _logits(T, V, 9).to(DEV)
    lab = torch.randint(0, V, (T,), dtype=torch.int64)
    lab[7] = V + 3
    with pytest.raises(vlc.VlcError) as ei:
        vlc.shifted_cross_entropy(z, lab.to(DEV))
    assert ei.value.status == vlc.binding.VLC_ERR_LABEL
    loss, cnt = vlc.shifted_cross_entropy(z, lab.to(DEV), check=False)
    assert int(cnt.item()) == T - 1


def test_ce_full_size_sampled_segments(vlc):
    # the SFT pack with a 32000-token vocabulary (4.2 GB of bf16 logits), as bench.py runs
    # it; the oracle recomputes a seeded sample of segments from their own rows
    w = synth.workload(1)
    V = 32000
    g = torch.Generator(device=DEV).manual_seed(77)
    z = (torch.randn((w.total, V), generator=g, device=DEV) * 2.0).to(torch.bfloat16)
    lab = _labels(w, 6, V)
    cut = torch.from_numpy(w.cu).to(DEV)
    loss, cnt, sl, sc = vlc.shifted_cross_entropy(z, torch.from_numpy(lab).to(DEV), cut, per_segment=True)
    assert int(cnt.item()) == int((lab != -100).sum())
    rng = np.random.default_rng(1)
    for r in rng.choice(w.nseg, size=6, replace=False):
        a, b = int(w.cu[r]), int(w.cu[r + 1])
        bits = oracle.bf16_bits(z[a:b].cpu())
        st, ref, ref_n, _, _ = oracle.shifted_ce(bits, lab[a:b])
        assert st == 0 and int(sc[r].item()) == ref_n
        assert abs(float(sl[r].item()) - ref) <= ABS_SEG + REL_SEG * abs(ref)
    assert float(loss.item()) == pytest.approx(float(sl.double().sum().item()), rel=1e-6)
