"""CPU checks of the offline parameter sweep (no GPU): the enumeration of
settings, the flags and names of a setting, parsing of the bench's JSON
line, and the summary table."""
import json

import pytest

from block_sparse_flash_attn_gb300 import tune

SPACE = {"A": [1, 2, 3], "B": [10, 20]}


def test_scan_is_the_full_product_in_order():
    got = tune.settings(SPACE, "scan")
    assert got == [{"A": a, "B": b} for a in (1, 2, 3) for b in (10, 20)]


def test_sample_is_seeded_distinct_and_bounded():
    a = tune.settings(SPACE, "sample", samples=4, seed=3)
    b = tune.settings(SPACE, "sample", samples=4, seed=3)
    assert a == b and len(a) == 4
    assert len({tuple(sorted(s.items())) for s in a}) == 4
    assert all(s in tune.settings(SPACE, "scan") for s in a)
    assert len(tune.settings(SPACE, "sample", samples=100)) == 6
    with pytest.raises(ValueError):
        tune.settings(SPACE, "grid")


def test_fixed_parameters():
    got = tune.settings(SPACE, "scan", fixed={"A": 2})
    assert got == [{"A": 2, "B": 10}, {"A": 2, "B": 20}]


def test_flags_and_tag():
    s = {"B": 20, "A": 1}
    assert tune.flags(s) == ["-DA=1", "-DB=20"]
    assert tune.tag(s) == tune.tag({"A": 1, "B": 20}) != tune.tag({"A": 2, "B": 20})


def test_parse_bench_takes_the_json_line():
    line = {"metric": "m", "value": 12.5, "ms_per_step": 0.25}
    out = "building...\n" + json.dumps(line) + "\n"
    assert tune.parse_bench(out) == line
    with pytest.raises(ValueError):
        tune.parse_bench("no json here\n")


def test_summary_and_table():
    rows = []
    for tg, st, ms in (("x", {"A": 1}, [2.0, 2.2]), ("y", {"A": 2}, [1.0, 1.2])):
        for i, m in enumerate(ms):
            rows.append({"tag": tg, "setting": st, "workload": 5, "repeat": i,
                         "ms_per_step": m, "value": 100.0 / m})
    summ = tune.summarize(rows)
    assert [r["tag"] for r in summ] == ["y", "x"]          # fastest first
    assert summ[0]["ms_mean"] == pytest.approx(1.1) and summ[0]["ms_std"] == pytest.approx(0.1414, 1e-3)
    text = tune.table(summ)
    assert text.splitlines()[0].startswith("| workload | A |")
    assert "| 5 | 2 | 1.1000 |" in text


def test_space_names_macros_the_sources_define():
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    csrc = os.path.join(root, "block_sparse_flash_attn_gb300", "csrc")
    text = "".join(open(os.path.join(csrc, f)).read() for f in os.listdir(csrc))
    for macro in tune.SPACE:
        assert f"#ifndef {macro}" in text, macro


def test_invalid_stage_combinations_are_skipped():
    space = {"BSATTN_D128_QSTAGES": [1, 2], "BSATTN_D128_KSTAGES": [2, 3],
             "BSATTN_D128_VSTAGES": [2, 3]}
    got = tune.settings(space, "scan")
    assert {"BSATTN_D128_QSTAGES": 2, "BSATTN_D128_KSTAGES": 3, "BSATTN_D128_VSTAGES": 3} not in got
    assert len(got) == 7
    assert all(tune.valid(s) for s in got)
