import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    """Parse a hand-worked fixture: returns dict with N, K, group, codes, scales,
    zeros and a list of (x_kind, y) cases plus an optional dequantised row."""
    d = {"cases": []}
    xkind = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key in ("N", "K", "group"):
                d[key] = int(vals[0])
            elif key == "codes":
                d["codes"] = np.array([int(v, 16) for v in vals], np.uint8)
            elif key == "zeros":
                d["zeros"] = np.array([int(v, 16) for v in vals], np.uint8)
            elif key == "scales_f16":
                d["scales"] = np.array([int(v, 16) for v in vals], np.uint16)
            elif key == "x":
                xkind = vals[0]
            elif key == "y":
                d["cases"].append((xkind, np.array([float(v) for v in vals], np.float32)))
            elif key == "dequant":
                d["dequant"] = np.array([float(v) for v in vals], np.float32)
            else:
                raise ValueError(f"unknown golden key {key!r} in {name}")
    N, K, g = d["N"], d["K"], d["group"]
    nb = K // g
    d["codes"] = d["codes"].reshape(N, K // 2)
    d["scales"] = d["scales"].reshape(N, nb)
    d["zeros"] = d["zeros"].reshape(N, (nb + 1) // 2)
    return d


def load_golden_blocks(name):
    """Parse a hand-worked block-format fixture: N, K, the raw bytes of every block
    in row order (uint8 [N, K/32, bytes per block]), the (x_kind, y) cases and the
    expected weights of the row(s)."""
    d = {"cases": [], "blocks": []}
    xkind = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key in ("N", "K"):
                d[key] = int(vals[0])
            elif key == "block":
                d["blocks"].append([int(v, 16) for v in vals])
            elif key == "x":
                xkind = vals[0]
            elif key == "y":
                d["cases"].append((xkind, np.array([float(v) for v in vals], np.float32)))
            elif key == "weights":
                d["weights"] = np.array([float(v) for v in vals], np.float32)
            else:
                raise ValueError(f"unknown golden key {key!r} in {name}")
    N, K = d["N"], d["K"]
    d["blocks"] = np.array(d["blocks"], np.uint8).reshape(N, K // 32, -1)
    return d


def golden_x(kind, K):
    if kind == "ones":
        return np.ones((1, K), np.float32)
    if kind == "index":
        return np.arange(K, dtype=np.float32).reshape(1, K)
    raise ValueError(kind)


GOLDEN_FILES = ["hand_1x32_g32.txt", "hand_2x96_g32_zeros.txt", "hand_1x128_g128.txt"]


def pack_codes(q):
    """Test-side packing of integer codes q[N, K] (0..15): even k low nibble."""
    q = np.asarray(q, np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def pack_zeros(z):
    """Test-side packing of zero points z[N, nb]: even group low nibble, pad 0."""
    z = np.asarray(z, np.uint8)
    N, nb = z.shape
    if nb % 2:
        z = np.concatenate([z, np.zeros((N, 1), np.uint8)], axis=1)
    return (z[:, 0::2] | (z[:, 1::2] << 4)).astype(np.uint8)
