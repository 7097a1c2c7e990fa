"""Pins for the oracle's bookkeeping: block schedule (LR-AttnRes Figure 11),
full schedule (MHAR Sec. 2.2) and the storage rounding of block sums."""

import json
import os

import numpy as np
import pytest

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load("block_schedule.json")["cases"],
                         ids=lambda c: f"M{c['M']}_NB{c['NB']}")
def test_block_schedule_golden(orc, case):
    from oracle import schedule
    assert schedule.block_ends(case["M"], case["NB"]) == case["ends"]
    plan = schedule.block_plan(case["M"], case["NB"])
    assert plan["ends"] == case["ends"]
    if "row_ops" in case:
        assert [list(op) for op in plan["row_ops"]] == case["row_ops"]
    if "sites" in case:
        assert plan["sites"] == case["sites"]
    if "site_source_counts" in case:
        assert [len(s) for s in plan["sites"]] == case["site_source_counts"]


def test_block_schedule_properties(orc):
    from oracle import schedule
    for M in range(1, 40):
        for NB in list(range(1, M + 1)) + [None]:
            plan = schedule.block_plan(M, NB)
            nb = M if NB is None else NB
            assert plan["ends"][-1] == M and len(plan["ends"]) == nb
            assert len(plan["sites"]) == M + 1
            # every site reads distinct rows, embedding first, rows in creation order
            for t, rows in enumerate(plan["sites"]):
                assert rows[0] == 0 and len(set(rows)) == len(rows) == sorted(rows).__len__()
                assert rows == sorted(rows) and all(x <= t for x in rows)
                assert rows[-1] == t
            # at most NB completed blocks + embedding + one partial
            assert max(len(s) for s in plan["sites"]) <= nb + 1
    # NB = M is full routing
    assert schedule.block_plan(7, None)["sites"] == schedule.full_sites(8)


def test_full_schedule():
    from oracle import schedule
    s = schedule.full_sites(73)
    assert len(s) == 73 and s[0] == [0] and s[-1] == list(range(73))
    assert sum(len(x) for x in s) == 73 * 74 // 2


@pytest.mark.parametrize("case", _load("bf16_rounding.json")["cases"], ids=lambda c: c["note"][:24])
def test_bf16_rounding_golden(orc, case):
    from oracle import storage
    assert storage.round_to_storage(np.array([case["x"]]), "bf16")[0] == case["bf16"]


def test_bf16_rounding_agrees_with_input_module():
    """Two independent RNE implementations (oracle: frexp/rint on float64; inputs:
    integer bit arithmetic on float32) agree on float32 values."""
    from oracle import storage
    x = synth.misc_normal(5, 77, (200000,), 3.0)
    ours = storage.storage_bits(storage.round_to_storage(x.astype(np.float64), "bf16"), "bf16")
    assert np.array_equal(ours, synth.bf16_bits_from_f32(x))


def test_block_bank_accumulates_and_rounds_once_per_version(orc):
    from oracle import schedule, storage
    plan = schedule.block_plan(6, 3)
    T, d = 3, 8
    outs = [synth.storage_to_f64(synth.sublayer_output(9, j, T, d, "bf16"), "bf16") for j in range(7)]
    rows = storage.block_bank(outs, plan, "bf16")
    assert np.array_equal(rows[2], storage.round_to_storage(outs[1] + outs[2], "bf16"))
    assert np.array_equal(rows[3], outs[3])
    assert np.array_equal(rows[4], storage.round_to_storage(rows[3] + outs[4], "bf16"))
    for r in rows:
        storage.storage_bits(r, "bf16")   # all representable
