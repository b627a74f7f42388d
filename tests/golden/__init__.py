"""Readers for the hand-derived fixtures in this folder (no arithmetic of the
method: they parse text)."""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _lines(name):
    with open(os.path.join(HERE, name)) as f:
        for ln in f:
            ln = ln.split("#", 1)[0].strip()
            if ln:
                yield ln.split()


def e2m1_rne_values():
    """[(value, expected_nibble)]"""
    return [(float(p[0]), int(p[1], 16)) for p in _lines("e2m1_rne_values.txt")]


def _payload_fixture(name):
    groups, payload, exps = {}, {}, None
    for p in _lines(name):
        if p[0] == "group":
            g, s = int(p[1]), int(p[2])
            vals = {}
            for kv in p[3:]:
                i, v = kv.split(":")
                vals[int(i)] = float(v)
            groups[g] = (s, vals)
        elif p[0] == "payload":
            payload[int(p[1])] = [int(x, 16) for x in p[2:]]
        elif p[0] == "exponents":
            exps = [int(x, 16) for x in p[1:]]
    pay = np.array([payload[g] for g in range(4)], np.uint8).reshape(-1)
    return groups, pay, np.array(exps, np.uint8)


def pack_layout_row():
    """Returns (row values fp64 [128], payload [64], exponents [4])."""
    groups, pay, exps = _payload_fixture("pack_layout_row.txt")
    row = np.zeros(128, np.float64)
    for g, (s, vals) in groups.items():
        for i, v in vals.items():
            row[32 * g + i] = v * 2.0 ** s
    return row, pay, exps


def midpoint_key_slot():
    """Returns (payload [64], exponents [4])."""
    _, pay, exps = _payload_fixture("midpoint_key_slot.txt")
    return pay, exps
