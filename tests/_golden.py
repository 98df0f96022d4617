"""Loader for the hand-worked fixtures in tests/golden/."""
import glob
import os

import numpy as np
import torch

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_bits(values):
    t = torch.tensor(values, dtype=torch.float32)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float32), t), "fixture value not exact in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


def load(path):
    case = {"name": os.path.basename(path), "x": {}, "scales": {}, "codes": {}, "y": []}
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        key, val = [p.strip() for p in line.split(":", 1)]
        if key == "K":
            case["K"] = int(val)
        elif key == "tensor_scale":
            case["tensor_scale"] = float(val)
        elif key.startswith("x"):
            case["x"][int(key[1:])] = [float(v) for v in val.split()]
        elif key.startswith("scales"):
            case["scales"][int(key[6:])] = bytes(int(v, 16) for v in val.split())
        elif key.startswith("codes"):
            case["codes"][int(key[5:])] = bytes(int(v, 16) for v in val.split())
        elif key.startswith("y"):
            lhs, rhs = val.split("->")
            case["y"].append(([float(v) for v in lhs.split()], [float(v) for v in rhs.split()]))
    rows = sorted(case["x"])
    case["X"] = np.stack([bf16_bits(case["x"][r]) for r in rows])
    case["scales_arr"] = np.stack([np.frombuffer(case["scales"][r], np.uint8) for r in rows])
    case["codes_arr"] = np.stack([np.frombuffer(case["codes"][r], np.uint8) for r in rows])
    return case


def all_cases():
    return [load(p) for p in sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))]


def _num(tok: str) -> float:
    return float.fromhex(tok) if ("0x" in tok or "p" in tok) else float(tok)


def load_format(path):
    """A fixture of tests/golden/mxfp4/ or tests/golden/fp8/: rows x<r>,
    optional tensor_scale, per-row scales<r> and codes<r> (hex bytes);
    decimal or hex-float values."""
    case = {"name": os.path.basename(path), "x": {}, "scales": {}, "codes": {}}
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        key, val = [p.strip() for p in line.split(":", 1)]
        if key == "K":
            case["K"] = int(val)
        elif key == "tensor_scale":
            case["tensor_scale"] = _num(val)
        elif key.startswith("x"):
            case["x"][int(key[1:])] = [_num(v) for v in val.split()]
        elif key.startswith("scales"):
            case["scales"][int(key[6:])] = bytes(int(v, 16) for v in val.split())
        elif key.startswith("codes"):
            case["codes"][int(key[5:])] = bytes(int(v, 16) for v in val.split())
    rows = sorted(case["x"])
    case["X"] = np.stack([bf16_bits(case["x"][r]) for r in rows])
    case["codes_arr"] = np.stack([np.frombuffer(case["codes"][r], np.uint8) for r in rows])
    if case["scales"]:
        case["scales_arr"] = np.stack([np.frombuffer(case["scales"][r], np.uint8) for r in rows])
    return case


def format_cases(fmt):
    return [load_format(p) for p in sorted(glob.glob(os.path.join(GOLDEN_DIR, fmt, "*.txt")))]
