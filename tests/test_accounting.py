"""Slot / pair ledgers and workload generators against the pages' printed numbers (CPU)."""
import json
import os

import numpy as np
import pytest

from tests.conftest import GOLDEN
from variable_length_causal_gb300 import synth


def _g(key):
    with open(os.path.join(GOLDEN, "ledgers.json")) as f:
        return json.load(f)[key]


def test_m020_sum_of_squares_vs_padded_pairs():
    g = _g("sum_sq_vs_padded_pairs")
    L = g["lengths"]
    assert synth.score_slots_per_segment(L) == g["score_per_segment"]
    assert synth.batch_score_slots(L, g["batch"]) == g["score_padded_pairs"]
    assert synth.batch_slots(L, g["batch"]) == g["slots_original_order"]
    assert synth.batch_slots(g["grouped_order"], g["batch"]) == g["slots_grouped"]


def test_charlestar_three_ledgers():
    g = _g("three_ledgers")
    L = g["lengths"]
    assert synth.token_slots_padded(L) == g["token_slots_padded"]
    assert int(np.sum(L)) == g["token_slots_packed"] == g["token_slots_whole"]
    assert synth.score_slots_padded(L) == g["score_slots_padded"]
    assert synth.score_slots_per_segment(L) == g["score_slots_per_segment"]
    assert synth.score_slots_whole(L) == g["score_slots_whole"]
    assert synth.causal_pairs(L) == g["causal_pairs_per_segment"]
    assert synth.causal_pairs([sum(L)]) == g["causal_pairs_whole"]
    assert synth.causal_pairs([sum(L)]) - synth.causal_pairs(L) == g["cross_sample_pairs"]


def test_vllbc_long_context_waste():
    g = _g("long_context_waste")
    slots = synth.token_slots_padded(g["lengths"], g["L"])
    assert slots == g["slots"] and sum(g["lengths"]) == g["real"] and slots - g["real"] == g["padding"]
    assert round(100 * synth.padding_waste(g["lengths"], g["L"]), 1) == g["waste_pct_1dp"]


@pytest.mark.parametrize("key", ["table_4_1_example_A", "table_4_1_example_B"])
def test_vllbc_table_4_1(key):
    g = _g(key)
    r = synth.pack_ledger(g["lengths"], g["L"])
    for k in ("T", "fixed", "padding", "packs", "packed", "pack_padding", "saved"):
        assert r[k] == g[k], k
    assert round(100 * r["waste"], 1) == g["waste_pct_1dp"]
    assert round(100 * r["saved_frac"], 1) == g["saved_pct_1dp"]
    if "score_fixed" in g:
        assert round(100 * r["pack_waste"], 1) == g["pack_waste_pct_1dp"]
        assert r["score_fixed_half"] == g["score_fixed"]
        assert r["score_packed_half"] == g["score_packed"]
        assert round(100 * g["score_packed"] / g["score_fixed"], 1) == g["score_ratio_pct_1dp"]


def test_operatorworld_valid_block_fraction():
    g = _g("window_valid_blocks")
    L = g["lengths"]
    assert synth.score_slots_per_segment(L) / synth.score_slots_whole(L) == pytest.approx(g["valid_fraction"])


def test_slot_efficiency_eta():
    # eta = sum L / (B * Lmax): two samples of 2 and 8 padded to 8 -> 10/16
    assert synth.slot_efficiency([2, 8], 2, 8) == pytest.approx(10 / 16)


def test_ffd_first_fit_decreasing():
    # llm-compass: sort descending, first bin with room
    bins = synth.first_fit_decreasing([8, 2, 7, 3], 10)
    assert bins == [[8, 2], [7, 3]]
    bins = synth.first_fit_decreasing([5, 6, 4, 3, 2], 10)
    assert bins == [[6, 4], [5, 3, 2]]


@pytest.mark.parametrize("idx", range(5))
def test_workloads_are_valid_and_deterministic(idx):
    w = synth.workload(idx)
    w2 = synth.workload(idx)
    assert np.array_equal(w.cu, w2.cu) and np.array_equal(w.seg_ignore, w2.seg_ignore)
    assert w.cu[0] == 0 and np.all(np.diff(w.cu) > 0)
    if idx == 0:
        assert w.nseg == 16 and w.lengths.max() <= 256
    elif idx in (1, 2, 4):
        n_bins = 16 if idx == 1 else 32
        assert w.total == n_bins * 4096
        # every bin boundary is a segment boundary; pad segments only at bin ends
        assert set(range(0, w.total + 1, 4096)) <= set(w.cu.tolist())
        ends = w.cu[1:][w.seg_ignore == 1]
        assert np.all(ends % 4096 == 0)
    else:
        assert w.total == 131072 and w.lengths.max() <= 32768


def test_assign_packs_balances_by_quadratic_cost():
    costs = [100.0, 1.0, 1.0, 1.0, 99.0, 2.0]
    a = synth.assign_packs(costs, 2)
    loads = [sum(costs[i] for i in r) for r in a]
    assert sorted(sum(a, [])) == list(range(6))
    assert max(loads) - min(loads) <= 2.0
