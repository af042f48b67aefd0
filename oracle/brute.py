"""Second, independent NumPy formulation of the method, for pinning the oracle.

TEST INFRASTRUCTURE ONLY. It shares nothing with oracle.c: the layout here is a
lexicographic sort of (expert, token, k) keys instead of a counting sort, the
e4m3 encoder is a nearest-value search over the 254 finite codes instead of an
exponent/mantissa split, and combine is summed in float64.
"""
from __future__ import annotations

import numpy as np


def layout(topk_idx: np.ndarray, E: int, R: int) -> dict:
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, K = idx.shape
    L = E // R
    valid = (idx >= 0) & (idx < E)
    t_of = np.repeat(np.arange(T), K).reshape(T, K)
    k_of = np.tile(np.arange(K), T).reshape(T, K)
    ev, tv, kv = idx[valid], t_of[valid], k_of[valid]
    order = np.lexsort((kv, tv, ev))          # primary expert, then token, then k
    rows = np.full((T, K), -1, np.int64)
    vt, vk = tv[order], kv[order]
    rows[vt, vk] = np.arange(len(order))
    cnt = np.bincount(ev, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(cnt)])
    in_rank = np.zeros((T, R), np.uint8)
    for r in range(R):
        in_rank[:, r] = (valid & (idx // L == r)).any(axis=1)
    return dict(
        num_tokens_per_expert=cnt.astype(np.int32),
        num_tokens_per_rank=in_rank.sum(axis=0).astype(np.int32),
        is_token_in_rank=in_rank,
        expert_offsets=offsets.astype(np.int32),
        row_of_slot=rows.astype(np.int32),
        status=int(((idx < -1) | (idx >= E)).any()) * 2,
    )


def layout_aligned(topk_idx: np.ndarray, E: int, R: int, A: int) -> dict:
    """Aligned layout from scratch: aligned starts by cumulative ceil, then
    each valid slot's rank inside its expert by sorting (expert, token, k)."""
    base = layout(topk_idx, E, R)
    cnt = base["num_tokens_per_expert"].astype(np.int64)
    padded = -(-cnt // A) * A
    starts = np.concatenate([[0], np.cumsum(padded)])
    idx = np.asarray(topk_idx, np.int64)
    rows = base["row_of_slot"].astype(np.int64)
    valid = rows >= 0
    rank_in_expert = rows - base["expert_offsets"][np.where(valid, idx, 0)]
    new_rows = np.where(valid, starts[np.where(valid, idx, 0)] + rank_in_expert, -1)
    out = dict(base)
    out["expert_offsets"] = starts.astype(np.int32)
    out["row_of_slot"] = new_rows.astype(np.int32)
    return out


def layout_strided(topk_idx: np.ndarray, E: int, R: int, cap: int) -> dict:
    """Strided layout from the sorted order: rank inside the expert, then e * cap."""
    base = layout(topk_idx, E, R)
    idx = np.asarray(topk_idx, np.int64)
    rows = base["row_of_slot"].astype(np.int64)
    valid = rows >= 0
    e = np.where(valid, idx, 0)
    rank_in_expert = rows - base["expert_offsets"][e]
    keep = valid & (rank_in_expert < cap)
    out = dict(base)
    out["expert_offsets"] = (np.arange(E + 1) * cap).astype(np.int32)
    out["row_of_slot"] = np.where(keep, e * cap + rank_in_expert, -1).astype(np.int32)
    out["status"] = 3 if (valid & ~keep).any() else base["status"]
    return out


def layout_nonexpand(topk_idx: np.ndarray, E: int, R: int) -> dict:
    """Non-expand layout from the unique (token, rank) pairs sorted by (rank, token)."""
    idx = np.asarray(topk_idx, np.int64)
    T, K = idx.shape
    L = E // R
    base = layout(idx, E, R)
    valid = (idx >= 0) & (idx < E)
    rank = np.where(valid, idx // L, -1)
    rows = np.full((T, K), -1, np.int64)
    pairs = sorted({(int(r), t) for t in range(T) for r in rank[t] if r >= 0})
    row_of_pair = {p: i for i, p in enumerate(pairs)}
    for t in range(T):
        seen = set()
        for k in range(K):
            r = int(rank[t, k])
            if r < 0 or r in seen:
                continue
            seen.add(r)
            rows[t, k] = row_of_pair[(r, t)]
    per_rank = base["num_tokens_per_rank"]
    return dict(num_tokens_per_expert=base["num_tokens_per_expert"], num_tokens_per_rank=per_rank,
                is_token_in_rank=base["is_token_in_rank"],
                rank_offsets=np.concatenate([[0], np.cumsum(per_rank)]).astype(np.int32),
                row_of_slot=rows.astype(np.int32), status=base["status"])


def e4m3_values() -> tuple[np.ndarray, np.ndarray]:
    """(codes, values) of the 254 finite OCP E4M3 codes, decoded from their bits."""
    codes, vals = [], []
    for c in range(256):
        s, f, m = c >> 7, (c >> 3) & 15, c & 7
        if f == 15 and m == 7:
            continue                                    # NaN
        v = m * 2.0 ** -9 if f == 0 else (1 + m / 8) * 2.0 ** (f - 7)
        codes.append(c)
        vals.append(-v if s else v)
    return np.array(codes, np.uint8), np.array(vals, np.float64)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite code (ties to the even code), saturating; -0 keeps its sign."""
    return _nearest_code(v, *e4m3_values(), 448.0)


def e5m2_values() -> tuple[np.ndarray, np.ndarray]:
    """(codes, values) of the 248 finite OCP E5M2 codes, decoded from their bits
    (exponent field 31 holds the infinities and NaNs)."""
    codes, vals = [], []
    for c in range(256):
        s, f, m = c >> 7, (c >> 2) & 31, c & 3
        if f == 31:
            continue
        v = m * 2.0 ** -16 if f == 0 else (1 + m / 4) * 2.0 ** (f - 15)
        codes.append(c)
        vals.append(-v if s else v)
    return np.array(codes, np.uint8), np.array(vals, np.float64)


def e5m2_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite e5m2 code (ties to the even code), saturating at 57344."""
    return _nearest_code(v, *e5m2_values(), 57344.0)


def _nearest_code(v, codes, vals, vmax) -> np.ndarray:
    v = np.asarray(v, np.float64).ravel()
    out = np.empty(v.shape, np.uint8)
    for i, x in enumerate(v):
        xs = min(max(x, -vmax), vmax)
        d = np.abs(vals - xs)
        best = d.min()
        cand = codes[d == best]
        if xs == 0.0:
            out[i] = 0x80 if np.signbit(x) else 0x00
            continue
        # a value sits between two codes of the same sign; ties go to the
        # code whose mantissa LSB is 0
        cand = [c for c in cand if (c >> 7) == (1 if xs < 0 else 0)]
        even = [c for c in cand if (c & 1) == 0]
        out[i] = even[0] if len(cand) > 1 and even else cand[0]
    return out


def combine_f64(y_f32: np.ndarray, row_of_slot: np.ndarray, w: np.ndarray | None) -> np.ndarray:
    """Exact-ish float64 combine: sum_k w * y[row] over used slots."""
    T, K = row_of_slot.shape
    H = y_f32.shape[1]
    out = np.zeros((T, H), np.float64)
    for k in range(K):
        r = row_of_slot[:, k]
        m = r >= 0
        wk = np.ones(T) if w is None else w[:, k].astype(np.float64)
        out[m] += wk[m, None] * y_f32[r[m]].astype(np.float64)
    return out
