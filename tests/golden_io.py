"""Readers for the hand-computed fixtures in tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _floats(s):
    return [float(t) for t in s.split()]


def _matrix(s, dtype):
    return np.array([_floats(r) for r in s.split(";")], dtype=dtype)


def act_quant_cases():
    out = []
    for line in _lines("act_quant_int8.txt"):
        tag, rest = line.split(":", 1)
        assert tag == "case"
        name, gs, x, s, q = [p.strip() for p in rest.split("|")]
        out.append(dict(name=name, gs=int(gs), x=np.array(_floats(x), np.float16),
                        s=np.array(_floats(s), np.float32), q=np.array(_floats(q), np.int8)))
    return out


def int4_cases():
    packs, quants = [], []
    for line in _lines("int4_pack.txt"):
        tag, rest = line.split(":", 1)
        parts = [p.strip() for p in rest.split("|")]
        if tag == "pack":
            packs.append((np.array(_floats(parts[0]), np.int8),
                          np.array([int(b, 16) for b in parts[1].split()], np.uint8)))
        else:
            quants.append((np.array(_floats(parts[0]), np.float16), np.float32(float(parts[1])),
                           np.array(_floats(parts[2]), np.int8),
                           np.array([int(b, 16) for b in parts[3].split()], np.uint8)))
    return packs, quants


def linear_cases():
    cases, cur = [], None
    for line in _lines("linear_small.txt"):
        key, val = [p.strip() for p in line.split(":", 1)] if ":" in line else (line, "")
        if key == "test":
            cur = dict(name=val)
        elif key == "end":
            cases.append(cur)
            cur = None
        elif key == "gs":
            cur["gs"] = int(val)
        elif key in ("x", "W", "y"):
            cur[key] = _matrix(val, np.float16)
        elif key in ("sa", "sw"):
            cur[key] = _matrix(val, np.float32)
        elif key in ("xq", "wq"):
            cur[key] = _matrix(val, np.int8)
        elif key == "acc":
            cur[key] = _matrix(val, np.int64)
    return cases


def weight_only_cases():
    """Cases of weight_only_small.txt: each ends with its `y` line."""
    cases, cur = [], None
    for line in _lines("weight_only_small.txt"):
        key, val = [p.strip() for p in line.split(":", 1)]
        if key == "test":
            cur = dict(name=val)
        elif key == "gs":
            cur["gs"] = int(val)
        elif key == "x":
            cur["x"] = _matrix(val, np.float16)
        elif key == "q":
            cur["q"] = _matrix(val, np.int8)
        elif key == "sw":
            cur["sw"] = _matrix(val, np.float32)
        elif key == "y":
            cur["y"] = _matrix(val, np.float16)
            cases.append(cur)
            cur = None
    return cases
