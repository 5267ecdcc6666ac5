"""Exhaustive path enumeration on reduced trellises (test helper).

Independent of the oracle: enumerates every state path of a small bitshift
trellis (L state bits, K bits per step, T steps) and sums its branch metrics
left to right in binary32 with numpy, one rounding per operation.
"""
import numpy as np


def all_paths(L, K, T, start_pred=None):
    """Array [n_paths, T] of full states.  Free start when start_pred is None,
    else the first state's predecessor is start_pred."""
    mask = (1 << L) - 1
    if start_pred is None:
        paths = np.arange(1 << L, dtype=np.int64)[:, None]
    else:
        e = np.arange(1 << K, dtype=np.int64)
        paths = (((start_pred << K) | e) & mask)[:, None]
    for _ in range(T - 1):
        last = paths[:, -1]
        e = np.arange(1 << K, dtype=np.int64)
        nxt = ((last[:, None] << K) | e[None, :]) & mask
        paths = np.concatenate([np.repeat(paths, 1 << K, axis=0), nxt.reshape(-1, 1)], axis=1)
    return paths


def path_costs(paths, y, cb):
    y = np.asarray(y, dtype=np.float32)
    cb = np.asarray(cb, dtype=np.float32)
    c = np.zeros(paths.shape[0], dtype=np.float32)
    for t in range(paths.shape[1]):
        d = (y[t] - cb[paths[:, t]]).astype(np.float32)
        q = (d * d).astype(np.float32)
        c = (c + q).astype(np.float32)
    return c


def lexmin_from_end(paths):
    """Index of the path that is lexicographically smallest when its states are
    read from the last to the first."""
    rev = paths[:, ::-1]
    order = np.lexsort(rev.T[::-1])
    return order[0]
