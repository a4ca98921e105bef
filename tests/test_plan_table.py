"""The plan-table generator: it scores every candidate per cell as a
percentage of the fastest, averages repeated measurements, refuses an
incomplete grid, and writes a header of the committed table's layout."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from allreduce_sum_residual_gb300 import plan_table as pt  # noqa: E402

KEYS = ("stream", "register1", "register2", "register4", "register8", "late1", "late2", "late4",
        "late8")


def _winner(n, H, m):
    # a deterministic, varied winner per cell
    return KEYS[(n * 7 + H // 1024 + m.bit_length()) % len(KEYS)]


def _write(path, cells, bonus=100.0, skip=None):
    with open(path, "w") as f:
        f.write("not json\n")
        for (n, H, m) in cells:
            if (n, H, m) == skip:
                continue
            row = {"n": n, "H": H, "m": m, "bytes": 1, "auto": 1.0}
            for k in KEYS:
                row[k] = 1000.0 + (bonus if k == _winner(n, H, m) else 0.0)
            f.write(json.dumps(row) + "\n")


INPUTS = (1, 2, 3, 4, 8, 16)
HIDDEN = (2048, 4096, 7168)
ROWS = (64, 128, 512, 4096)


def _grid():
    return [(n, H, m) for n in INPUTS for H in HIDDEN for m in ROWS]


def test_keeps_the_fastest_per_cell(tmp_path):
    f = tmp_path / "a.jsonl"
    _write(f, _grid())
    table = pt.choose(pt.load([str(f)]))
    chars = dict(pt.CANDIDATES)
    for cell in _grid():
        assert table[cell][0] == chars[_winner(*cell)]


def test_averages_repeats_within_a_file(tmp_path):
    a = tmp_path / "a.jsonl"
    _write(a, _grid(), bonus=100.0)
    # a repeated line for every cell favours another candidate by less than
    # the first line's margin: the average keeps the first winner
    with open(a, "a") as f:
        for (n, H, m) in _grid():
            row = {"n": n, "H": H, "m": m}
            for k in KEYS:
                row[k] = 1000.0
            row["stream" if _winner(n, H, m) != "stream" else "register1"] = 1050.0
            f.write(json.dumps(row) + "\n")
    table = pt.choose(pt.load([str(a)]))
    chars = dict(pt.CANDIDATES)
    for cell in _grid():
        assert table[cell][0] == chars[_winner(*cell)]


def test_a_later_file_replaces_whole_cells(tmp_path):
    a, b = tmp_path / "a.jsonl", tmp_path / "b.jsonl"
    _write(a, _grid(), bonus=100.0)
    n0, H0, m0 = _grid()[0]
    with open(b, "w") as f:   # one cell re-measured with only two candidates
        f.write(json.dumps({"n": n0, "H": H0, "m": m0, "stream": 900.0, "late2": 1000.0}) + "\n")
    table = pt.choose(pt.load([str(a), str(b)]))
    assert table[(n0, H0, m0)] == ("b", [90, 0, 0, 0, 0, 0, 100, 0, 0])
    chars = dict(pt.CANDIDATES)
    for cell in _grid()[1:]:
        assert table[cell][0] == chars[_winner(*cell)]


def test_refuses_a_missing_cell(tmp_path):
    f = tmp_path / "a.jsonl"
    _write(f, _grid(), skip=(3, 4096, 512))
    with pytest.raises(SystemExit, match="n=3 H=4096 m=512"):
        pt.choose(pt.load([str(f)]))


def test_percentages(tmp_path):
    f = tmp_path / "a.jsonl"
    with open(f, "w") as fh:
        for (n, H, m) in _grid():
            fh.write(json.dumps({"n": n, "H": H, "m": m, "stream": 500.0, "register1": 1000.0,
                                 "register2": 995.0, "register4": None, "register8": 333.0,
                                 "late1": 1010.0}) + "\n")
    table = pt.choose(pt.load([str(f)]))
    for cell in _grid():
        assert table[cell] == ("a", [50, 99, 99, 0, 33, 100, 0, 0, 0])


def test_rendered_header_matches_the_grid(tmp_path):
    f = tmp_path / "a.jsonl"
    _write(f, _grid())
    table = pt.choose(pt.load([str(f)]))
    text = pt.render(table, 152, "test")
    assert "constexpr int kPlanTableSms = 152;" in text
    assert f"kPlanScore[{len(INPUTS)}][{len(HIDDEN)}][{len(ROWS)}][{len(pt.CANDIDATES)}]" in text
    assert "kPlanInputs[6] = {1, 2, 3, 4, 8, 16}" in text
    assert "kPlanPacks[3] = {256, 512, 896}" in text
    assert "kPlanRows[4] = {64, 128, 512, 4096}" in text
    chars = dict(pt.CANDIDATES)
    lines = text.splitlines()
    for n in INPUTS:
        at = lines.index(f"    {{  // n = {n}")
        for i, H in enumerate(HIDDEN):
            comment, data = lines[at + 1 + 2 * i].strip(), lines[at + 2 + 2 * i].strip()
            assert comment == f"// H = {H}: " + "".join(chars[_winner(n, H, m)] for m in ROWS)
            assert data == "{" + ", ".join("{" + ",".join(map(str, table[(n, H, m)][1])) + "}"
                                           for m in ROWS) + "},"


def test_generator_reproduces_the_committed_layout():
    """Re-rendering the committed table's own cells gives the committed file
    back, apart from the sources line."""
    import re
    path = os.path.join(ROOT, "allreduce_sum_residual_gb300", "csrc", "plan_table.cuh")
    text = open(path).read()
    grab = lambda name: [int(x) for x in re.search(name + r"\[\d+\] = \{([^}]*)\}", text).group(1).split(",")]
    inputs, packs, rows = grab("kPlanInputs"), grab("kPlanPacks"), grab("kPlanRows")
    sms = int(re.search(r"kPlanTableSms = (\d+)", text).group(1))
    body = text[text.index("kPlanScore["):]
    nc = len(pt.CANDIDATES)
    cells = [[int(x) for x in c.split(",")] for c in re.findall(r"\{(\d+(?:,\d+){%d})\}" % (nc - 1), body)]
    assert len(cells) == len(inputs) * len(packs) * len(rows)
    chars = [c for _, c in pt.CANDIDATES]
    table, it = {}, iter(cells)
    for n in inputs:
        for P in packs:
            for m in rows:
                pct = next(it)
                table[(n, 8 * P, m)] = (chars[pct.index(max(pct))], pct)
    again = pt.render(table, sms, "x")
    strip = lambda t: [l for l in t.splitlines() if "sources:" not in l]
    assert strip(again) == strip(text)
