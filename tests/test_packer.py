"""Host packer (vlc_pack, vlc_shard_packs) against the packing oracle, on CPU: windows and
shard assignments must match bit for bit (integer work), plus invariants at sizes the oracle
does not reach.
"""
import math

import numpy as np
import pytest

from oracle import packing

MODES = {"ffd": packing.ffd, "first_fit": packing.first_fit, "next_fit": packing.next_fit}


@pytest.fixture(scope="module")
def vlc():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as m

    m.load_library()
    return m


def _lengths(seed, n, median, sigma, lo, hi):
    rng = np.random.default_rng(seed)
    return np.clip(np.round(rng.lognormal(np.log(median), sigma, size=n)), lo, hi).astype(np.int32)


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("extra", [0, 1])
def test_pack_matches_oracle(vlc, mode, extra):
    for seed, (n, cap) in enumerate([(1, 16), (7, 16), (300, 4096), (1500, 4096), (900, 700)]):
        L = _lengths(seed, n, cap / 8, 1.0, 1, cap + cap // 4)   # some samples longer than a window
        p = vlc.pack(L, cap, extra=extra, mode=mode)
        bin_of, order, bin_start = MODES[mode](L.tolist(), cap, extra)
        assert np.array_equal(p.bin_of, bin_of)
        assert np.array_equal(p.order, order)
        assert np.array_equal(p.bin_start, bin_start)
        assert p.oversize == packing.oversize_count(L.tolist(), cap, extra)
        assert p.eta == pytest.approx(packing.eta(L, p.nbins, cap), rel=1e-12)


def test_pack_large_sizes_take_the_comparison_sort(vlc):
    # sizes above the counting-sort range, with many ties
    rng = np.random.default_rng(3)
    L = (rng.integers(1, 40, size=400) * (1 << 18)).astype(np.int32)
    cap = 1 << 24
    p = vlc.pack(L, cap)
    bin_of, order, bin_start = packing.ffd(L.tolist(), cap)
    assert np.array_equal(p.order, order) and np.array_equal(p.bin_start, bin_start)


@pytest.mark.parametrize("cost", ["tokens", "sumsq"])
@pytest.mark.parametrize("ranks", [1, 2, 3, 8])
def test_shard_matches_oracle(vlc, cost, ranks):
    L = _lengths(11, 2000, 300, 1.0, 16, 4096)
    p = vlc.pack(L, 4096)
    rank_of, load = vlc.shard_packs(L, p, ranks, cost=cost)
    costs = packing.pack_costs(L, p.order, p.bin_start, cost)
    r2, l2 = packing.lpt(costs, ranks)
    assert np.array_equal(rank_of, r2) and np.array_equal(load, l2)


def test_million_samples_invariants_and_utilisation(vlc):
    # an SFT-like length mix (lognormal median 300, sigma 1.0, clipped to [16, 4096])
    L = _lengths(5, 1_000_000, 300, 1.0, 16, 4095)   # + 1 reserved token fits a window
    cap = 4096
    p = vlc.pack(L, cap, extra=1)
    assert p.oversize == 0
    assert sorted(p.order.tolist()) == list(range(len(L)))
    fill = np.add.reduceat((L.astype(np.int64) + 1)[p.order], p.bin_start[:-1])
    assert fill.max() <= cap and np.array_equal(np.bincount(p.bin_of, minlength=p.nbins),
                                                np.diff(p.bin_start))
    assert p.nbins >= math.ceil(int(L.sum() + len(L)) / cap)
    assert p.eta > 0.99            # FFD fills windows almost completely on this mix
    nf = vlc.pack(L, cap, extra=1, mode="next_fit")
    assert nf.nbins > p.nbins      # streaming wastes more
    rank_of, load = vlc.shard_packs(L, p, 8)
    assert load.max() / load.min() < 1.01
    by_tok, _ = vlc.shard_packs(L, p, 8, cost="tokens")
    sq = np.add.reduceat((L.astype(np.int64) ** 2)[p.order], p.bin_start[:-1])
    work_tok = np.bincount(by_tok, weights=sq, minlength=8)
    assert load.max() <= work_tok.max()


def test_packer_argument_errors(vlc):
    with pytest.raises(ValueError):
        vlc.pack(np.zeros((2, 2), np.int32), 16)
    with pytest.raises(vlc.VlcError):
        vlc.pack(np.array([3, 0, 2], np.int32), 16)        # a zero-length sample
    with pytest.raises(vlc.VlcError):
        vlc.pack(np.array([3, 2], np.int32), 0)
    p = vlc.pack(np.array([3, 2], np.int32), 16)
    with pytest.raises(vlc.VlcError):
        vlc.shard_packs(np.array([3, 2], np.int32), p, 0)
    with pytest.raises(KeyError):
        vlc.pack(np.array([3, 2], np.int32), 16, mode="best_fit")


def test_window_cu_seqlens(vlc):
    L = np.array([1024, 768, 512, 256, 96], np.int32)
    p = vlc.pack(L, 2048)
    assert p.cu_seqlens(L, 0).tolist() == [0, 1024, 1792, 2048]
    assert p.cu_seqlens(L, 1).tolist() == [0, 512, 608]
