"""Seeded synthetic workloads for MoE token dispatch / combine.

This module only draws random inputs. It holds none of the method's arithmetic
(no layout, no permute, no quantiser, no combine): both the CPU oracle and the
CUDA path read the exact bytes produced here.

Workloads (shapes follow the dispatch / combine signatures of the DeepEP API
docs, "dispatch()" section: x [num_tokens, hidden] bf16, topk_idx
[num_tokens, num_topk] int64, topk_weights [num_tokens, num_topk] fp32):

  tiny     T=128   H=256  E=8   K=2 R=2  x~N(0,1), uniform distinct experts,
           weights U(0,1) normalised; the combine input is the dispatched
           rows themselves (identity expert).
  decode   T=256   H=7168 E=256 K=8 R=8  weights = softmax over K of N(0,1)
           logits; y ~N(0,1) [T*K, H].
  prefill  T=8192  H=7168 E=256 K=8 R=8  weights U(0,1) normalised;
           y ~N(0,1) [N, H].
  fp8      as prefill, x ~N(0, 2^2) with floor(0.001*H) outlier channels
           scaled x50 before the bf16 round.
  skewed   T=16384 H=4096 E=64 K=6 R=4  experts drawn without replacement with
           probability proportional to Zipf(s=1.2) over a seeded expert
           permutation (Gumbel-top-k), then each slot dropped (-1) with
           probability 0.05; weights U(0,1) normalised over the valid slots.

Every stream comes from numpy's PCG64 seeded through SeedSequence(seed).spawn:
one child each for x, routing, weights and y. Large arrays are drawn in fixed
row chunks, each from its own grandchild seed, so the bytes do not depend on
how many threads draw them. fp32 -> bf16 uses round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK_ROWS = 2048


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    K: int
    R: int
    x_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_gain: float = 1.0
    routing: str = "uniform"      # "uniform" | "zipf"
    zipf_s: float = 1.2
    drop_p: float = 0.0
    weights: str = "uniform"      # "uniform" | "softmax"
    y: str = "normal"             # "normal" | "identity"
    fp8: bool = False


WORKLOADS = {
    "tiny": Workload("tiny", T=128, H=256, E=8, K=2, R=2, y="identity"),
    "decode": Workload("decode", T=256, H=7168, E=256, K=8, R=8, weights="softmax"),
    "prefill": Workload("prefill", T=8192, H=7168, E=256, K=8, R=8),
    "fp8": Workload("fp8", T=8192, H=7168, E=256, K=8, R=8, x_std=2.0,
                    outlier_frac=0.001, outlier_gain=50.0, fp8=True),
    "skewed": Workload("skewed", T=16384, H=4096, E=64, K=6, R=4, routing="zipf",
                       zipf_s=1.2, drop_p=0.05),
}


def _threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bits.

    Inputs here are finite by construction (normal draws times small gains).
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u = u + np.uint32(0x7FFF)
    u += lsb
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: np.random.SeedSequence, rows: int, cols: int, std: float = 1.0,
                col_gain: np.ndarray | None = None, threads: int | None = None) -> np.ndarray:
    """[rows, cols] bf16 bits of std * N(0,1) (times a per-column gain), chunked."""
    out = np.empty((rows, cols), dtype=np.uint16)
    if rows == 0:
        return out
    nchunks = (rows + CHUNK_ROWS - 1) // CHUNK_ROWS
    kids = seed.spawn(nchunks)

    def work(c: int) -> None:
        r0, r1 = c * CHUNK_ROWS, min(rows, (c + 1) * CHUNK_ROWS)
        g = np.random.Generator(np.random.PCG64(kids[c]))
        a = g.standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        if col_gain is not None:
            a *= col_gain[None, :]
        out[r0:r1] = f32_to_bf16_bits(a)

    n = threads or _threads()
    if n == 1 or nchunks == 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _distinct_topk_by_key(keys: np.ndarray, K: int) -> np.ndarray:
    """Per row, the K column indices of the largest keys, largest first."""
    part = np.argpartition(-keys, K - 1, axis=1)[:, :K]
    kv = np.take_along_axis(keys, part, axis=1)
    order = np.argsort(-kv, axis=1, kind="stable")
    return np.take_along_axis(part, order, axis=1)


def routing(w: Workload, seed: np.random.SeedSequence) -> np.ndarray:
    """topk_idx [T, K] int64: K distinct experts per token, -1 = dropped slot."""
    g = np.random.Generator(np.random.PCG64(seed))
    if w.routing == "uniform":
        keys = g.random((w.T, w.E))
    elif w.routing == "zipf":
        perm = g.permutation(w.E)
        p = np.empty(w.E)
        p[perm] = 1.0 / np.arange(1, w.E + 1, dtype=np.float64) ** w.zipf_s
        p /= p.sum()
        # Gumbel-top-k: the K largest of log p + Gumbel noise are a draw of K
        # distinct items without replacement with probabilities p.
        u = g.random((w.T, w.E))
        keys = np.log(p)[None, :] - np.log(-np.log1p(-u))
    else:
        raise ValueError(w.routing)
    idx = _distinct_topk_by_key(keys, w.K).astype(np.int64)
    if w.drop_p > 0:
        drop = g.random((w.T, w.K)) < w.drop_p
        idx[drop] = -1
    return np.ascontiguousarray(idx)


def weights(w: Workload, idx: np.ndarray, seed: np.random.SeedSequence) -> np.ndarray:
    """topk_weights [T, K] fp32, normalised to sum 1 over each token's valid slots."""
    g = np.random.Generator(np.random.PCG64(seed))
    valid = idx >= 0
    if w.weights == "softmax":
        logits = g.standard_normal((w.T, w.K))
        logits = np.where(valid, logits, -np.inf)
        m = logits.max(axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.where(valid, np.exp(logits - m), 0.0)
    else:
        e = np.where(valid, g.random((w.T, w.K)), 0.0)
    s = e.sum(axis=1, keepdims=True)
    out = np.divide(e, s, out=np.zeros_like(e), where=s > 0)
    return np.ascontiguousarray(out.astype(np.float32))


@dataclasses.dataclass
class Inputs:
    w: Workload
    seed: int
    x: np.ndarray            # [T, H] uint16 (bf16 bits)
    topk_idx: np.ndarray     # [T, K] int64
    topk_weights: np.ndarray  # [T, K] float32
    y: np.ndarray | None     # [N, H] uint16 (bf16 bits); None for the identity expert
    num_valid: int


def make(name_or_w, seed: int = 0, with_y: bool = True, T: int | None = None,
         threads: int | None = None) -> Inputs:
    """Draw one workload. `T` overrides the token count (same recipe, fewer rows)."""
    w = WORKLOADS[name_or_w] if isinstance(name_or_w, str) else name_or_w
    if T is not None:
        w = dataclasses.replace(w, T=T)
    sx, sr, sw, sy = np.random.SeedSequence(seed).spawn(4)
    gain = None
    if w.outlier_frac > 0:
        gain = np.ones(w.H, dtype=np.float32)
        gain[_outlier_cols(w, sx)] = np.float32(w.outlier_gain)
    x = normal_bf16(_child(sx, 0), w.T, w.H, std=w.x_std, col_gain=gain, threads=threads)
    idx = routing(w, sr)
    wt = weights(w, idx, sw)
    n = int((idx >= 0).sum())
    y = None
    if with_y and w.y == "normal":
        y = normal_bf16(sy, n, w.H, threads=threads)
    return Inputs(w=w, seed=seed, x=x, topk_idx=idx, topk_weights=wt, y=y, num_valid=n)


def _child(ss: np.random.SeedSequence, i: int) -> np.random.SeedSequence:
    """The i-th child of `ss`, independent of how many children were spawned before."""
    return np.random.SeedSequence(ss.entropy, spawn_key=tuple(ss.spawn_key) + (i,))


def _outlier_cols(w: Workload, sx: np.random.SeedSequence) -> np.ndarray:
    n_out = int(np.floor(w.outlier_frac * w.H))
    return np.random.Generator(np.random.PCG64(_child(sx, 1))).permutation(w.H)[:n_out]


def outlier_columns(name_or_w, seed: int = 0) -> np.ndarray:
    """The channels that the fp8 workload scales x50 (sorted)."""
    w = WORKLOADS[name_or_w] if isinstance(name_or_w, str) else name_or_w
    return np.sort(_outlier_cols(w, np.random.SeedSequence(seed).spawn(4)[0]))
