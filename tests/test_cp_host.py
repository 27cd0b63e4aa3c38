"""Host side of the context-parallel split (libvlc's vlc_cp_partition, vlc_cp_block_mode)
against the oracle's partition: bit-exact rows, positions and chunk offsets, the error for
a segment length that is not a multiple of 2 * cp, and the block rule of the ring."""
import numpy as np
import pytest

from oracle import cp as ocp


@pytest.fixture(scope="module")
def vlc():
    import __graft_entry__ as g

    g.build()
    import variable_length_causal_gb300 as m

    m.load_library()
    return m


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_partition_matches_oracle(vlc, cp):
    rng = np.random.default_rng(cp)
    lengths = (rng.integers(1, 40, size=13) * 2 * cp).tolist()
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    for rank in range(cp):
        rows, pos, cu_chunk = vlc.cp_partition(cu, cp, rank)
        o_rows, o_pos, o_m = ocp.partition(lengths, cp, rank)
        assert np.array_equal(rows, o_rows)
        assert np.array_equal(pos.astype(np.int64), o_pos)
        assert np.array_equal(np.diff(cu_chunk).astype(np.int64), o_m)


def test_partition_reports_the_first_bad_segment(vlc):
    cu = np.array([0, 8, 14, 22], np.int32)        # 6 is not a multiple of 4
    with pytest.raises(ValueError, match="segment 1"):
        vlc.cp_partition(cu, 2, 0)


@pytest.mark.parametrize("cp", [1, 2, 3, 5])
def test_block_rule(vlc, cp):
    chunk = lambda r, h: r if h == 0 else 2 * cp - 1 - r
    for qr in range(cp):
        for qh in (0, 1):
            for kr in range(cp):
                for kh in (0, 1):
                    cq, ck = chunk(qr, qh), chunk(kr, kh)
                    want = 2 if ck < cq else (1 if ck == cq else 0)
                    assert vlc.cp_block_mode(cp, qr, qh, kr, kh) == want
    # over a full ring every query half sees exactly the chunks up to its own
    for qr in range(cp):
        for qh in (0, 1):
            seen = [chunk(kr, kh) for kr in range(cp) for kh in (0, 1) if vlc.cp_block_mode(cp, qr, qh, kr, kh)]
            assert sorted(seen) == list(range(chunk(qr, qh) + 1))
