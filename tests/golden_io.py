"""Readers for the text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _triple(s):
    return tuple(int(v) for v in s.split(","))


def window_index_cases():
    """{name: dict(grid, win, shift, padded, flags, n_idx, n_pads, entries=[(dst, src)])}"""
    cases = {}
    with open(os.path.join(GOLDEN, "window_index_worked.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "case":
                name = parts[1]
                cases[name] = dict(grid=_triple(parts[2]), win=_triple(parts[3]),
                                   shift=_triple(parts[4]), padded=_triple(parts[5]),
                                   flags=int(parts[6]), n_idx=int(parts[7]),
                                   n_pads=int(parts[8]), entries=[])
            else:
                cases[parts[0]]["entries"].append((int(parts[1]), int(parts[2])))
    return cases


def gelu_tiny_input():
    rows, bias = [], None
    with open(os.path.join(GOLDEN, "gelu_tiny_input.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            vals = [float(v) for v in parts[1:]]
            if parts[0] == "input":
                rows.append(vals)
            elif parts[0] == "bias":
                bias = vals
    return rows, bias


def shift_region_cases():
    """{name: dict(grid, win, shift, padded, flags, axes, windows={window_id: [labels]})}"""
    cases = {}
    with open(os.path.join(GOLDEN, "shift_regions_worked.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "case":
                cases[parts[1]] = dict(grid=_triple(parts[2]), win=_triple(parts[3]),
                                       shift=_triple(parts[4]), padded=_triple(parts[5]),
                                       flags=int(parts[6]), axes=int(parts[7]), windows={})
            else:
                cases[parts[0]]["windows"][int(parts[1])] = [int(v) for v in parts[2:]]
    return cases
