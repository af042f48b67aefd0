"""Worker for the all-fp32-patterns encoder test: kept free of torch so that
spawned worker processes start quickly. Test infrastructure only."""
from multiprocessing import shared_memory

import numpy as np


def nan_mask(lo: int, n: int) -> np.ndarray:
    """True where the fp32 bit pattern lo + i is a NaN."""
    u = np.arange(lo, lo + n, dtype=np.uint64).astype(np.uint32)
    return ((u >> 23) & 0xFF == 0xFF) & (u & 0x7FFFFF != 0)


def _e4m3_nan(q):
    return (q & 0x7F) == 0x7F


def _e5m2_nan(q):
    return ((q >> 2) & 0x1F == 0x1F) & (q & 3 != 0)


def compare_slice(args):
    """Oracle sweeps of patterns [lo, lo + n) against the device codes at
    byte offset `off` of the two shared buffers (e4m3, e5m2). Returns, per
    format, (patterns compared, mismatch count, (pattern, device code, oracle
    code) of the first mismatch)."""
    import oracle
    name4, name5, off, lo, n = args
    nan = nan_mask(lo, n)
    out = []
    for name, sweep, is_nan_code in ((name4, oracle.e4m3_sweep, _e4m3_nan),
                                     (name5, oracle.e5m2_sweep, _e5m2_nan)):
        shm = shared_memory.SharedMemory(name=name)
        try:
            got = np.ndarray((n,), np.uint8, buffer=shm.buf, offset=off).copy()
        finally:
            shm.close()
        want = sweep(lo, lo + n)
        bad = ((got != want) & ~nan) | (nan & ~is_nan_code(got))
        idx = np.flatnonzero(bad)
        out.append((int(want.size), int(idx.size), None if idx.size == 0 else
                    (int(lo + idx[0]), int(got[idx[0]]), int(want[idx[0]]))))
    return out
