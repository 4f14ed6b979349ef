"""Readers for the page-printed fixtures under tests/golden/ (no arithmetic)."""
import os

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(HERE, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def ch37_trace():
    rows, outs, shapes, work, reset = [], {}, {}, {}, {}
    for tok in _lines("ch37_fixture_trace.txt"):
        if tok[0] == "row":
            p, h, j = map(int, tok[1:4])
            rows.append((p, h, j, [float(x) for x in tok[4:6]], [float(x) for x in tok[6:8]], float(tok[8])))
        elif tok[0] == "out":
            outs[int(tok[1])] = [float(x) for x in tok[2:]]
        elif tok[0] == "shape":
            shapes[int(tok[1])] = [int(x) for x in tok[2:]]
        elif tok[0] == "work":
            work = {tok[i]: int(tok[i + 1]) for i in range(1, len(tok), 2)}
        elif tok[0] == "reset":
            reset = {tok[i]: tok[i + 1] for i in range(1, len(tok), 2)}
    return rows, outs, shapes, work, reset


def lcp5_table():
    table, example = {}, {}
    for tok in _lines("lcp5_table.txt"):
        if tok[0].startswith("example"):
            example[tok[0]] = [int(x) for x in tok[1:]]
        elif tok[0] in ("threshold", "observed_max"):
            example[tok[0]] = float(tok[1])
        else:
            table[tok[0]] = dict(query_len=int(tok[1]), cut=int(tok[2]), rows=int(tok[3]),
                                 full_rows=int(tok[4]), in_scope=tok[5] == "yes", policy=tok[5])
    return table, example
