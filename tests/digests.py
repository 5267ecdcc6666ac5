"""SHA-256 digests of whole-matrix results, for comparisons at full size.

Stored expected values for the full-size workloads are digests of the oracle's
results (written by ``tests/golden/make_full_digests.py``, which calls only
``oracle/`` and the seeded input generators); the GPU tests digest the CUDA
path's results the same way and compare.  A digest covers one 128-row band of
tiles (8 tile rows), so a mismatch names the band.  Floats are stored as
``float.hex`` strings, exact.
"""
from __future__ import annotations

import hashlib
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "full_digests.json")
BAND_ROWS = 128


def sha(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def tensor_bytes(t) -> np.ndarray:
    """The raw bytes of a CPU torch tensor (bf16 viewed as int16) as numpy."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy()


def input_digests(W, su, sv) -> dict:
    return {"W": sha(tensor_bytes(W)), "su": sha(tensor_bytes(su)), "sv": sha(tensor_bytes(sv))}


def band_digests(codes: np.ndarray, costs, rows: int, cols: int, K: int) -> list:
    """[[codes digest, costs digest] per 128-row band]; codes uint16/int16
    [rows/16, cols/16, 16K], costs fp32 [n_tiles] in row-major tile order (or None)."""
    codes = np.ascontiguousarray(codes).view(np.uint16).reshape(rows // 16, cols // 16, 16 * K)
    tpb = BAND_ROWS // 16
    c2 = None if costs is None else np.ascontiguousarray(costs, dtype=np.float32).reshape(rows // 16, cols // 16)
    out = []
    for b in range(rows // BAND_ROWS):
        out.append([sha(codes[b * tpb:(b + 1) * tpb]),
                    None if c2 is None else sha(c2[b * tpb:(b + 1) * tpb])])
    return out


def fhex(x) -> str:
    return float(x).hex()


def unhex(s: str) -> float:
    return float.fromhex(s)


def load() -> dict:
    if not os.path.exists(GOLDEN):
        return {}
    with open(GOLDEN) as f:
        return json.load(f)


def save(d: dict) -> None:
    tmp = GOLDEN + ".tmp"
    with open(tmp, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")
    os.replace(tmp, GOLDEN)
