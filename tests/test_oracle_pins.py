"""Pins for the CPU oracle: each check comes from something other than the
oracle itself -- hand-worked fixtures, an independent NumPy formulation, torch's
own format casts, closed forms and invariants of the method."""
import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from gen import inputs as gi


def _ints(v):
    return np.array([int(x, 0) for x in v], dtype=np.int64)


# ------------------------------------------------------------------ layout

@pytest.mark.parametrize("name", ["layout_hand.txt", "layout_hand_dup.txt"])
def test_layout_golden(golden, name):
    g = golden(name)
    T, K, E, R = (int(g[k][0]) for k in "TKER")
    idx = _ints(g["topk_idx"]).reshape(T, K)
    L = oracle.layout(idx, E, R)
    assert L["status"] == oracle.OK
    np.testing.assert_array_equal(L["num_tokens_per_expert"], _ints(g["num_tokens_per_expert"]))
    np.testing.assert_array_equal(L["expert_offsets"], _ints(g["expert_offsets"]))
    np.testing.assert_array_equal(L["row_of_slot"].ravel(), _ints(g["row_of_slot"]))
    np.testing.assert_array_equal(L["is_token_in_rank"].ravel(), _ints(g["is_token_in_rank"]))
    np.testing.assert_array_equal(L["num_tokens_per_rank"], _ints(g["num_tokens_per_rank"]))


def _random_routing(rng, T, K, E, drop_p=0.0, distinct=True, bad_p=0.0):
    if distinct and K <= E:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :K]
    else:
        idx = rng.integers(0, E, size=(T, K))
    idx = idx.astype(np.int64)
    idx[rng.random((T, K)) < drop_p] = -1
    if bad_p > 0:
        bad = rng.random((T, K)) < bad_p
        idx[bad] = rng.choice([E, E + 5, -2, -100], size=bad.sum())
    return idx


CORNERS = [
    # (T, K, E, R, drop_p, distinct, bad_p)
    (1, 1, 1, 1, 0.0, True, 0.0),
    (1, 4, 8, 2, 0.0, True, 0.0),
    (7, 3, 5, 5, 0.2, True, 0.0),    # E == R
    (33, 2, 6, 1, 0.1, False, 0.0),  # R == 1, duplicates allowed
    (50, 8, 8, 4, 0.0, True, 0.0),   # K == E: every token hits every expert
    (64, 4, 16, 4, 1.0, True, 0.0),  # everything dropped
    (129, 6, 64, 4, 0.05, True, 0.0),
    (300, 2, 32, 8, 0.3, False, 0.0),
    (40, 3, 12, 3, 0.0, True, 0.1),  # invalid ids
]


@pytest.mark.parametrize("case", CORNERS)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_layout_vs_brute(case, seed):
    T, K, E, R, drop_p, distinct, bad_p = case
    rng = np.random.default_rng(seed)
    idx = _random_routing(rng, T, K, E, drop_p, distinct, bad_p)
    a = oracle.layout(idx, E, R)
    b = brute.layout(idx, E, R)
    for key in ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank",
                "expert_offsets", "row_of_slot", "status"]:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_layout_one_expert_takes_all():
    idx = np.full((100, 1), 3, np.int64)
    L = oracle.layout(idx, 8, 2)
    assert L["num_tokens_per_expert"].tolist() == [0, 0, 0, 100, 0, 0, 0, 0]
    assert L["row_of_slot"].ravel().tolist() == list(range(100))
    assert L["num_tokens_per_rank"].tolist() == [100, 0]


def test_layout_k1_is_stable_argsort():
    rng = np.random.default_rng(5)
    e = rng.integers(0, 16, size=500)
    L = oracle.layout(e[:, None], 16, 4)
    order = np.argsort(e, kind="stable")
    rows = np.empty(500, np.int64)
    rows[order] = np.arange(500)
    np.testing.assert_array_equal(L["row_of_slot"].ravel(), rows)


def test_layout_bad_args():
    idx = np.zeros((4, 2), np.int64)
    assert oracle.layout(idx, 6, 4)["status"] == oracle.ERR_ARG  # E % R != 0


def _check_invariants(idx, E, R, L):
    T, K = idx.shape
    valid = idx >= 0
    N = int(valid.sum())
    cnt, off, rows = L["num_tokens_per_expert"], L["expert_offsets"], L["row_of_slot"]
    assert cnt.sum() == N and off[0] == 0 and off[E] == N
    assert (np.diff(off) == cnt).all()
    r = rows[valid]
    assert np.array_equal(np.sort(r), np.arange(N))            # bijection onto [0, N)
    assert (rows[~valid] == -1).all()
    # rows of expert e lie in its range, in strictly increasing (t, k) order
    e_of_row = np.empty(N, np.int64)
    slot_of_row = np.empty(N, np.int64)
    e_of_row[r] = idx[valid]
    slot_of_row[r] = np.flatnonzero(valid.ravel())
    for e in range(E):
        seg = slice(off[e], off[e + 1])
        assert (e_of_row[seg] == e).all()
        assert (np.diff(slot_of_row[seg]) > 0).all()
    Lr = E // R
    slab = np.array([off[(q + 1) * Lr] - off[q * Lr] for q in range(R)])
    assert slab.sum() == N
    ntr = L["num_tokens_per_rank"]
    assert (ntr <= np.minimum(T, slab)).all()
    assert (L["is_token_in_rank"].sum(axis=0) == ntr).all()


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed"])
def test_layout_invariants_on_workloads(name):
    w = gi.WORKLOADS[name]
    inp = gi.make(name, 0, with_y=False)
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    assert L["status"] == oracle.OK
    _check_invariants(inp.topk_idx, w.E, w.R, L)


# ------------------------------------------------------------------ formats

def _torch_bf16_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _torch_e4m3_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _structured_f32_patterns():
    """All sign/exponent/top-mantissa combinations with low bits near the
    rounding midpoints of bf16 (bit 15) and e4m3 (bits 19 and below)."""
    hi = np.arange(1 << 13, dtype=np.uint32) << np.uint32(19)   # sign, exp, top 4 mantissa bits
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x3FFFF, 0x40000, 0x40001, 0x7FFFF,
                     0x10000, 0x18000], np.uint32)
    u = (hi[:, None] | lows[None, :]).ravel()
    f = u.view(np.float32)
    return f[np.isfinite(f)]


def test_bf16_encoder_vs_torch():
    rng = np.random.default_rng(0)
    f = np.concatenate([_structured_f32_patterns(),
                        rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32)])
    f = f[np.isfinite(f)]
    np.testing.assert_array_equal(oracle.f32_to_bf16(f), _torch_bf16_bits(f))


def test_e4m3_encoder_vs_torch():
    rng = np.random.default_rng(1)
    f = np.concatenate([_structured_f32_patterns(),
                        rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
                        (rng.standard_normal(500_000) * 100).astype(np.float32),
                        (rng.standard_normal(500_000) * 0.01).astype(np.float32)])
    f = f[np.isfinite(f)]
    np.testing.assert_array_equal(oracle.f32_to_e4m3(f), _torch_e4m3_bits(f))


def test_e4m3_encoder_vs_brute_search():
    rng = np.random.default_rng(2)
    codes, vals = brute.e4m3_values()
    mids = (np.sort(vals)[1:] + np.sort(vals)[:-1]) / 2
    f = np.concatenate([vals, mids, mids * (1 + 2**-20), mids * (1 - 2**-20), [500.0, -1e30, 464.0, -0.0],
                        rng.standard_normal(3000) * 50]).astype(np.float32)
    np.testing.assert_array_equal(oracle.f32_to_e4m3(f), brute.e4m3_encode(f))


def test_encoders_on_every_bf16_bit_pattern():
    """Every bf16 value (the dispatch's inputs are bf16) through the oracle's
    encoders: bf16 gives back the same bits, e4m3 and e5m2 give torch's
    saturating casts; NaN patterns are outside the contract."""
    u = (np.arange(1 << 16, dtype=np.uint32) << np.uint32(16))
    f = u.view(np.float32)
    fin = np.isfinite(f)
    np.testing.assert_array_equal(oracle.f32_to_bf16(f[fin]), (u[fin] >> 16).astype(np.uint16))
    np.testing.assert_array_equal(oracle.f32_to_e4m3(f[fin]), _torch_e4m3_bits(f[fin]))
    np.testing.assert_array_equal(oracle.f32_to_e5m2(f[fin]), _torch_e5m2_bits(f[fin]))
    assert fin.sum() == (1 << 16) - 2 * 128    # all but the 2 x 128 infinity / NaN patterns


_SWEEP_RANGES = [
    (0x00000000, 1 << 18),                 # +0 and fp32 subnormals
    (0x3A800000 - (1 << 17), 0x3A800000 + (1 << 17)),   # around 2^-10 (fp8 subnormals)
    (0x3F800000 - (1 << 18), 0x3F800000 + (1 << 18)),   # around 1.0
    (0x43E00000 - (1 << 19), 0x43E00000 + (1 << 19)),   # around 448 (e4m3 saturation)
    (0x47600000 - (1 << 19), 0x47600000 + (1 << 19)),   # around 57344 (e5m2 saturation)
    (0xBF800000 - (1 << 18), 0xBF800000 + (1 << 18)),   # around -1.0
    (0x7F7FFFFF - (1 << 16), 0x7F800000),               # the largest finite values
]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_sweep_encodes_each_bit_pattern(fmt):
    """The range encoders the GPU conversion sweep compares against give, for
    each fp32 bit pattern in [lo, hi), torch's saturating cast of that value."""
    sweep = oracle.e4m3_sweep if fmt == "e4m3" else oracle.e5m2_sweep
    for lo, hi in _SWEEP_RANGES:
        f = np.arange(lo, hi, dtype=np.uint64).astype(np.uint32).view(np.float32)
        want = _torch_e4m3_bits(f) if fmt == "e4m3" else _torch_e5m2_bits(f)
        np.testing.assert_array_equal(sweep(lo, hi), want, err_msg=f"{fmt} [{lo:#x}, {hi:#x})")


def test_e4m3_decode_roundtrip():
    codes, vals = brute.e4m3_values()
    dec = oracle.e4m3_to_f32(codes)
    np.testing.assert_array_equal(dec.astype(np.float64), vals)
    np.testing.assert_array_equal(oracle.f32_to_e4m3(vals.astype(np.float32)), codes)


# ------------------------------------------------------------------ fp8 quantiser

def test_fp8_block_golden(golden):
    g = golden("fp8_block_hand.txt")
    x = np.zeros(128, np.float32)
    for kv in g["x"]:
        i, v = kv.split(":")
        x[int(i)] = float(v)
    xb = gi.f32_to_bf16_bits(x)
    assert (gi.bf16_bits_to_f32(xb) == x).all(), "fixture values must be bf16-exact"
    q, s = oracle.quant_row_e4m3(xb)
    assert s[0] == np.float32(float(g["scale"][0]))
    want = np.zeros(128, np.uint8)
    for kv in g["q"]:
        i, v = kv.split(":")
        want[int(i)] = int(v, 16)
    np.testing.assert_array_equal(q, want)


def test_fp8_closed_forms():
    rng = np.random.default_rng(3)
    H = 1024
    x = (rng.standard_normal((64, H)) * 2).astype(np.float32)
    x[0, :128] = 0.0          # an all-zero block
    x[1, 128:256] = -0.0      # all negative zeros
    x[2, 256:384] = 1e-38     # tiny normal values
    xb = gi.f32_to_bf16_bits(x)
    xf = gi.bf16_bits_to_f32(xb).reshape(64, H // 128, 128)
    for t in range(64):
        q, s = oracle.quant_row_e4m3(xb[t])
        qb = q.reshape(-1, 128)
        deq = oracle.e4m3_to_f32(q).reshape(-1, 128).astype(np.float64)
        for b in range(H // 128):
            blk = xf[t, b]
            amax = np.abs(blk).max()
            if amax == 0:
                assert s[b] == 0 and (qb[b] == 0).all()
                continue
            assert s[b] == np.float32(amax) / np.float32(448.0)
            # the block-max element always lands on +-448
            i = int(np.argmax(np.abs(blk)))
            assert qb[b, i] in (0x7E, 0xFE)
            # dequantisation error: half a step of e4m3 at each magnitude
            err = np.abs(deq[b] * s[b] - blk.astype(np.float64))
            bound = np.maximum(np.abs(blk) * 2.0**-4, 2.0**-10 * s[b]) * (1 + 1e-6)
            assert (err <= bound).all()


# ------------------------------------------------------------------ dispatch / combine

def test_dispatch_bf16_moves_rows():
    inp = gi.make("tiny", 0)
    w = inp.w
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    N = int(L["expert_offsets"][-1])
    recv, src, rw = oracle.dispatch_bf16(inp.x, L["row_of_slot"], N, inp.topk_weights)
    for t in range(w.T):
        for k in range(w.K):
            r = L["row_of_slot"][t, k]
            assert (recv[r] == inp.x[t]).all() and src[r] == t and rw[r] == inp.topk_weights[t, k]


def test_combine_golden(golden):
    g = golden("combine_hand.txt")
    H = int(g["H"][0])
    y = gi.f32_to_bf16_bits(np.array([float(v) for v in g["y"]], np.float32)).reshape(-1, H)
    rows = _ints(g["row_of_slot"]).reshape(-1, 2).astype(np.int32)
    w = np.array([float(v) for v in g["topk_weights"]], np.float32).reshape(-1, 2)
    out = oracle.combine(y, rows, w)
    want = np.array([float(v) for v in g["out"]], np.float32).reshape(-1, H)
    np.testing.assert_array_equal(gi.bf16_bits_to_f32(out), want)


def test_combine_one_hot_recovers_rows():
    inp = gi.make("tiny", 1)
    w = inp.w
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    N = int(L["expert_offsets"][-1])
    rng = np.random.default_rng(0)
    y = gi.f32_to_bf16_bits(rng.standard_normal((N, w.H)).astype(np.float32))
    onehot = np.zeros((w.T, w.K), np.float32)
    pick = rng.integers(0, w.K, w.T)
    onehot[np.arange(w.T), pick] = 1.0
    out = oracle.combine(y, L["row_of_slot"], onehot)
    np.testing.assert_array_equal(out, y[L["row_of_slot"][np.arange(w.T), pick]])


def test_combine_identity_expert_recovers_x():
    inp = gi.make("tiny", 0)
    w = inp.w
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    N = int(L["expert_offsets"][-1])
    recv, _, _ = oracle.dispatch_bf16(inp.x, L["row_of_slot"], N)
    out = gi.bf16_bits_to_f32(oracle.combine(recv, L["row_of_slot"], inp.topk_weights))
    x = gi.bf16_bits_to_f32(inp.x)
    # weights sum to 1 within a few fp32 ulps, then one bf16 round
    np.testing.assert_allclose(out, x, rtol=2.0**-7, atol=0)


@pytest.mark.parametrize("name,null_w", [("skewed", False), ("decode", False), ("tiny", True)])
def test_combine_vs_f64(name, null_w):
    inp = gi.make(name, 2, T=96)
    w = inp.w
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    N = int(L["expert_offsets"][-1])
    y = inp.y if inp.y is not None else gi.normal_bf16(np.random.SeedSequence(9), N, w.H)
    wt = None if null_w else inp.topk_weights
    out = gi.bf16_bits_to_f32(oracle.combine(y, L["row_of_slot"], wt)).astype(np.float64)
    yf = gi.bf16_bits_to_f32(y)
    ref = brute.combine_f64(yf, L["row_of_slot"], wt)
    absw = np.ones((w.T, w.K)) if wt is None else np.abs(wt.astype(np.float64))
    mag = brute.combine_f64(np.abs(yf), L["row_of_slot"], absw)
    # fp32 accumulation error (K roundings of at most 2^-24 relative to the
    # running magnitude) plus half a bf16 ulp of the result
    bound = w.K * 2.0**-24 * mag + 2.0**-8 * np.abs(ref) + 1e-30
    assert (np.abs(out - ref) <= bound).all()
    # and dropped-only tokens give +0
    dead = (L["row_of_slot"] < 0).all(axis=1)
    assert (out[dead] == 0).all()


def test_combine_tokens_within_the_f64_bound():
    """The per-token combine used for sampled checks at full size: within the
    float64 bound, and the same rows as the full combine."""
    inp = gi.make("skewed", 4, T=80)
    w = inp.w
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    toks = [0, 3, 17, 41, 79]
    got = oracle.combine_tokens(inp.y, L["row_of_slot"], inp.topk_weights, toks)
    yf = gi.bf16_bits_to_f32(inp.y)
    ref = brute.combine_f64(yf, L["row_of_slot"], inp.topk_weights)[toks]
    mag = brute.combine_f64(np.abs(yf), L["row_of_slot"], np.abs(inp.topk_weights.astype(np.float64)))[toks]
    out = gi.bf16_bits_to_f32(got).astype(np.float64)
    assert (np.abs(out - ref) <= w.K * 2.0**-24 * mag + 2.0**-8 * np.abs(ref) + 1e-30).all()
    np.testing.assert_array_equal(got, oracle.combine(inp.y, L["row_of_slot"], inp.topk_weights)[toks])


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_dispatch_e5m2_rows_are_their_tokens_quantised(mode):
    """Each used slot's row holds its token's e5m2 codes and scales (checked
    against the quantiser, itself pinned above); unused rows stay zero."""
    inp = gi.make("tiny", 5, with_y=False)
    w = inp.w
    L = oracle.layout(inp.topk_idx, w.E, w.R)
    n = int(L["expert_offsets"][-1])
    q, s = oracle.dispatch_e5m2(inp.x, L["row_of_slot"], n + 3, scale_mode=mode)
    seen = np.zeros(n + 3, bool)
    for t, k in zip(*np.nonzero(L["row_of_slot"] >= 0)):
        r = L["row_of_slot"][t, k]
        qt, st = oracle.quant_row_e5m2(inp.x[t], mode)
        np.testing.assert_array_equal(q[r], qt)
        np.testing.assert_array_equal(s[r], st)
        seen[r] = True
    assert seen[:n].all() and not seen[n:].any()
    assert not q[n:].any() and not s[n:].any()


@pytest.mark.parametrize("seed", [0, 1])
def test_dispatch_e4m3_rows_are_their_tokens_quantised(seed):
    """The e4m3 quantise-permute (nccl_ep.cc, ncclEpDispatch, low-latency
    branch: fp32 scales one per 128 channels, [rows, hidden/128]; DeepEP API
    docs, dispatch(): recv_topk_weights) places, for every used slot (t, k),
    token t's codes and scale row at receive row row_of_slot[t, k], writes
    source t and weight w[t, k] there, and leaves every other row untouched.
    The routing has dropped slots, an all-dropped token and repeated experts,
    and each token's weights are distinct, so a weight taken from another
    slot shows; codes and scales are checked against the quantiser, which the
    fixtures and closed forms above pin."""
    rng = np.random.default_rng(40 + seed)
    T, K, E, R, H = 37, 3, 8, 2, 256
    idx = _random_routing(rng, T, K, E, drop_p=0.25, distinct=False)
    idx[5] = -1
    x = gi.f32_to_bf16_bits((rng.standard_normal((T, H)) * 3).astype(np.float32))
    x[7, :128] = 0                         # one all-zero block: scale 0, zero codes
    w = (rng.permutation(T * K).reshape(T, K) + 1).astype(np.float32) / 128.0
    L = oracle.layout(idx, E, R)
    n = int(L["expert_offsets"][-1])
    spare = 4
    q, s, src, rw = oracle.dispatch_e4m3(x, L["row_of_slot"], n + spare, w)
    seen = np.zeros(n + spare, bool)
    for t in range(T):
        qt, st = oracle.quant_row_e4m3(x[t])
        for k in range(K):
            r = L["row_of_slot"][t, k]
            if r < 0:
                continue
            np.testing.assert_array_equal(q[r], qt)
            np.testing.assert_array_equal(s[r].view(np.uint32), st.view(np.uint32))
            assert src[r] == t and rw[r] == w[t, k], (t, k, r)
            assert not seen[r]
            seen[r] = True
    assert seen[:n].all() and not seen[n:].any()
    # the rows no slot names keep what the caller put there
    assert not q[n:].any() and np.isnan(s[n:]).all() and (src[n:] == -1).all() and np.isnan(rw[n:]).all()
    # the all-zero block: scale 0 and zero codes in each of token 7's rows
    for r in L["row_of_slot"][7][L["row_of_slot"][7] >= 0]:
        assert s[r, 0] == 0.0 and not q[r, :128].any()
    # without weights the optional weight output is not written
    q2, s2, src2, rw2 = oracle.dispatch_e4m3(x, L["row_of_slot"], n)
    assert rw2 is None
    np.testing.assert_array_equal(q2, q[:n])
    np.testing.assert_array_equal(src2, src[:n])


# ------------------------------------------------------------------ alignment

def test_layout_aligned_golden(golden):
    g = golden("layout_hand_aligned.txt")
    T, K, E, R, A = (int(g[k][0]) for k in "TKERA")
    idx = _ints(g["topk_idx"]).reshape(T, K)
    L = oracle.layout_aligned(idx, E, R, A)
    assert L["status"] == oracle.OK
    np.testing.assert_array_equal(L["num_tokens_per_expert"], _ints(g["num_tokens_per_expert"]))
    np.testing.assert_array_equal(L["expert_offsets"], _ints(g["expert_offsets"]))
    np.testing.assert_array_equal(L["row_of_slot"].ravel(), _ints(g["row_of_slot"]))
    n_pad = int(L["expert_offsets"][-1])
    recv = np.full((n_pad, 8), 0x7777, np.uint16)
    src = np.full(n_pad, 99, np.int32)
    oracle.fill_pad_rows(L, recv, src=src)
    pad = sorted(int(r) for r in np.flatnonzero(src == -1))
    assert pad == [int(v) for v in g["pad_rows"]]
    assert (recv[pad] == 0).all() and (recv[src != -1] == 0x7777).all()


@pytest.mark.parametrize("A", [1, 2, 3, 8, 64, 128])
@pytest.mark.parametrize("case", CORNERS[:8])
def test_layout_aligned_vs_brute(case, A):
    T, K, E, R, drop_p, distinct, bad_p = case
    rng = np.random.default_rng(A)
    idx = _random_routing(rng, T, K, E, drop_p, distinct, bad_p)
    a = oracle.layout_aligned(idx, E, R, A)
    b = brute.layout_aligned(idx, E, R, A)
    for key in ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank",
                "expert_offsets", "row_of_slot"]:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    off = a["expert_offsets"]
    assert (off % A == 0).all()
    pad = np.diff(off) - a["num_tokens_per_expert"]
    assert ((pad >= 0) & (pad < A)).all()


def test_layout_aligned_one_is_plain_layout():
    inp = gi.make("skewed", 0, with_y=False)
    w = inp.w
    a, b = oracle.layout_aligned(inp.topk_idx, w.E, w.R, 1), oracle.layout(inp.topk_idx, w.E, w.R)
    for key in ["expert_offsets", "row_of_slot", "num_tokens_per_expert"]:
        np.testing.assert_array_equal(a[key], b[key])


def _slots_rows(L, key_of_slot, n_keys):
    """Receive rows of the slots of each key (expert, or rank)."""
    rows = L["row_of_slot"].ravel()
    keys = key_of_slot.ravel()
    return [set(int(r) for r in rows[(keys == k) & (rows >= 0)]) for k in range(n_keys)]


@pytest.mark.parametrize("A", [1, 4, 128])
@pytest.mark.parametrize("seed", range(3))
def test_aligned_layout_follows_expand_mode_prefix_sum_recipe(A, seed):
    """DeepEP API docs, "Prefix Sum Interpretation for Expert Token Counts",
    expand mode: the handle's per-expert prefix sum points at the END of each
    expert's real rows; expert i starts at align(psum[i-1], alignment) (0 for
    i = 0) and holds end - start real rows. With the end of expert i's real
    rows taken as offsets[i] + count[i], that recipe must give back this
    layout's starts and counts, the real rows of expert i must be exactly
    [start, end), and the buffer ends at align(psum[E-1], alignment). With
    alignment 1 it is also "Computing with Handle Metadata": start =
    psum[i-1], end = psum[i]."""
    rng = np.random.default_rng(40 + seed)
    T, K, E, R = 300, 6, 24, 4
    idx = _random_routing(rng, T, K, E, drop_p=0.1)
    L = oracle.layout_aligned(idx, E, R, A)
    assert L["status"] == oracle.OK
    cnt, off = L["num_tokens_per_expert"], L["expert_offsets"]
    psum = off[:E] + cnt

    def align(v):
        return (int(v) + A - 1) // A * A

    by_expert = _slots_rows(L, idx, E)
    for i in range(E):
        start = 0 if i == 0 else align(psum[i - 1])
        end = int(psum[i])
        assert start == off[i] and end - start == cnt[i]
        assert by_expert[i] == set(range(start, end))
        if A == 1:
            assert start == (0 if i == 0 else psum[i - 1])
    assert align(psum[E - 1]) == off[E]


@pytest.mark.parametrize("seed", range(3))
def test_nonexpand_layout_follows_inclusive_prefix_sum_recipe(seed):
    """DeepEP API docs, "Prefix Sum Interpretation for Expert Token Counts",
    non-expand mode: a standard inclusive prefix sum, so destination r holds
    rows [psum[r-1], psum[r]) (from 0 for r = 0). Here one row per (token,
    rank): the count of rank r is its number of distinct tokens, the rows of
    the slots routed to rank r fill that range, and of one token's slots on
    one rank only the first (lowest k) carries the row, the others -1."""
    rng = np.random.default_rng(50 + seed)
    T, K, E, R = 257, 5, 32, 8
    idx = _random_routing(rng, T, K, E, drop_p=0.15)
    L = oracle.layout_nonexpand(idx, E, R)
    assert L["status"] == oracle.OK
    psum = L["rank_offsets"][1:]
    rank_of_slot = np.where(idx >= 0, idx // (E // R), -1)
    by_rank = _slots_rows(L, rank_of_slot, R)
    for r in range(R):
        start = 0 if r == 0 else int(psum[r - 1])
        end = int(psum[r])
        distinct_tokens = len({t for t in range(T) if (rank_of_slot[t] == r).any()})
        assert end - start == distinct_tokens == L["num_tokens_per_rank"][r]
        assert by_rank[r] == set(range(start, end))
    rows = L["row_of_slot"]
    for t in range(T):
        for r in range(R):
            ks = np.flatnonzero(rank_of_slot[t] == r)
            if len(ks):
                assert rows[t, ks[0]] >= 0 and (rows[t, ks[1:]] == -1).all()


# ------------------------------------------------------------------ backward

def _small_routed(seed, T=40, K=3, E=8, R=2, H=24, drop_p=0.2):
    rng = np.random.default_rng(seed)
    idx = _random_routing(rng, T, K, E, drop_p, True, 0.0)
    L = oracle.layout(idx, E, R)
    N = int(L["expert_offsets"][-1])
    y = gi.f32_to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    g = gi.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    w = rng.random((T, K)).astype(np.float32)
    return idx, L, N, y, g, w


def test_combine_backward_vs_numpy():
    idx, L, N, y, g, w = _small_routed(0)
    rows = L["row_of_slot"]
    gy, gw = oracle.combine_backward(g, y, rows, w, N)
    gf, yf = gi.bf16_bits_to_f32(g), gi.bf16_bits_to_f32(y)
    for t in range(rows.shape[0]):
        for k in range(rows.shape[1]):
            r = rows[t, k]
            if r < 0:
                assert gw[t, k] == 0.0
                continue
            # grad_y: the fp32 product rounded once to bf16 (torch's cast as the rounder)
            prod = (np.float32(w[t, k]) * gf[t]).astype(np.float32)
            want = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            np.testing.assert_array_equal(gy[r], want)
            np.testing.assert_allclose(gw[t, k], np.dot(gf[t].astype(np.float64), yf[r].astype(np.float64)),
                                       rtol=1e-12, atol=1e-12)
    covered = np.zeros(N, bool)
    covered[rows[rows >= 0]] = True
    assert covered.all()


def test_combine_backward_adjoint_identity():
    """<grad_out, combine(y)> equals sum over slots of w * <grad_out[t], y[row]> (exact in float64)."""
    idx, L, N, y, g, w = _small_routed(1, T=60, K=4, E=12, R=3, H=40)
    rows = L["row_of_slot"]
    _, gw = oracle.combine_backward(g, y, rows, w, N)
    gf, yf = gi.bf16_bits_to_f32(g).astype(np.float64), gi.bf16_bits_to_f32(y).astype(np.float64)
    fwd = brute.combine_f64(gi.bf16_bits_to_f32(y), rows, w)
    lhs = float((gf * fwd).sum())
    rhs = float((w.astype(np.float64) * gw).sum())
    assert abs(lhs - rhs) <= 1e-9 * max(1.0, abs(lhs))


def test_combine_backward_unit_weights_copy_rows():
    idx, L, N, y, g, w = _small_routed(2)
    rows = L["row_of_slot"]
    gy, _ = oracle.combine_backward(g, y, rows, None, N)
    for t, k in zip(*np.nonzero(rows >= 0)):
        np.testing.assert_array_equal(gy[rows[t, k]], g[t])   # w = 1: exact copy


def test_dispatch_backward_is_unweighted_combine_and_gather():
    idx, L, N, y, g, w = _small_routed(3)
    rows = L["row_of_slot"]
    rng = np.random.default_rng(9)
    grw = rng.standard_normal(N).astype(np.float32)
    gx, gtw = oracle.dispatch_backward(y, grw, rows)
    np.testing.assert_array_equal(gx, oracle.combine(y, rows, None))
    want = np.where(rows >= 0, grw[np.maximum(rows, 0)], 0.0).astype(np.float32)
    np.testing.assert_array_equal(gtw, want)
    # grad_x is the sum of the copies: against float64 within one bf16 rounding plus fp32 adds
    ref = brute.combine_f64(gi.bf16_bits_to_f32(y), rows, None)
    got = gi.bf16_bits_to_f32(gx).astype(np.float64)
    mag = brute.combine_f64(np.abs(gi.bf16_bits_to_f32(y)), rows, None)
    assert (np.abs(got - ref) <= 2.0**-8 * np.abs(ref) + rows.shape[1] * 2.0**-24 * mag + 1e-30).all()


# ------------------------------------------------------------------ fp8 variants

def test_fp8_pow2_golden(golden):
    g = golden("fp8_pow2_hand.txt")
    x = np.zeros(128, np.float32)
    for kv in g["x"]:
        i, v = kv.split(":")
        x[int(i)] = float(v)
    xb = gi.f32_to_bf16_bits(x)
    q, s = oracle.quant_row_e4m3_pow2(xb)
    assert s[0] == np.float32(float(g["scale"][0]))
    _, sb = oracle.quant_row_e4m3_pow2(xb, ue8m0=True)
    assert sb[0] == int(g["ue8m0"][0])
    want = np.zeros(128, np.uint8)
    for kv in g["q"]:
        i, v = kv.split(":")
        want[int(i)] = int(v, 16)
    np.testing.assert_array_equal(q, want)


def test_pow2_ceil_vs_numpy():
    rng = np.random.default_rng(4)
    s = np.concatenate([np.exp2(rng.integers(-140, 120, 200)).astype(np.float32),
                        (rng.random(2000) * 10.0 ** rng.integers(-30, 30, 2000)).astype(np.float32)])
    s = s[(s > 0) & np.isfinite(s)]
    got = np.array([oracle.pow2_ceil(v) for v in s], np.float64)
    want = np.exp2(np.ceil(np.log2(s.astype(np.float64))))
    np.testing.assert_array_equal(got, want)


def test_fp8_pow2_closed_forms():
    rng = np.random.default_rng(5)
    H = 1024
    xf = (rng.standard_normal((32, H)) * 3).astype(np.float32)
    xf[0, :128] = 0.0
    xf[1, 128:256] = 1e-39            # amax/448 below 2^-127: UE8M0 clamps
    xb = gi.f32_to_bf16_bits(xf)
    xv = gi.bf16_bits_to_f32(xb).reshape(32, H // 128, 128)
    for t in range(32):
        q, s = oracle.quant_row_e4m3_pow2(xb[t])
        qu, sb = oracle.quant_row_e4m3_pow2(xb[t], ue8m0=True)
        for b in range(H // 128):
            blk = xv[t, b]
            amax = np.abs(blk).max()
            if amax == 0:
                assert s[b] == 0 and sb[b] == 0 and (q[b*128:(b+1)*128] == 0).all()
                continue
            s0 = np.float32(amax) / np.float32(448.0)
            m, e = np.frexp(np.float64(s[b]))
            assert m == 0.5 and s[b] >= s0 and (s[b] / 2 < s0)      # minimal power of two
            # codes: x / scale is exact, so they equal torch's clamped cast of it
            want = _torch_e4m3_bits((blk / s[b]).astype(np.float32))
            np.testing.assert_array_equal(q[b*128:(b+1)*128], want)
            ue_scale = max(float(s[b]), 2.0**-127)
            assert sb[b] == int(np.log2(ue_scale)) + 127
            want_u = _torch_e4m3_bits((blk / np.float32(ue_scale)).astype(np.float32))
            np.testing.assert_array_equal(qu[b*128:(b+1)*128], want_u)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_dispatch_e4m3_pow2_rows_are_their_tokens_quantised(ue8m0):
    """Each used slot's row holds its token's power-of-two-scale codes and
    scales (checked against the quantiser pinned above); unused rows stay zero."""
    rng = np.random.default_rng(6)
    T, K, E, R, H = 29, 3, 8, 4, 256
    idx = _random_routing(rng, T, K, E, drop_p=0.2, distinct=False)
    x = gi.f32_to_bf16_bits((rng.standard_normal((T, H)) * 5).astype(np.float32))
    L = oracle.layout(idx, E, R)
    n = int(L["expert_offsets"][-1])
    q, s = oracle.dispatch_e4m3_pow2(x, L["row_of_slot"], n + 2, ue8m0)
    seen = np.zeros(n + 2, bool)
    for t, k in zip(*np.nonzero(L["row_of_slot"] >= 0)):
        r = L["row_of_slot"][t, k]
        qt, st = oracle.quant_row_e4m3_pow2(x[t], ue8m0)
        np.testing.assert_array_equal(q[r], qt)
        np.testing.assert_array_equal(s[r], st)
        seen[r] = True
    assert seen[:n].all() and not seen[n:].any()
    assert not q[n:].any() and not s[n:].any()


# ------------------------------------------------------------------ e5m2

def _torch_e5m2_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).clamp(-57344.0, 57344.0)
    return t.to(torch.float8_e5m2).view(torch.uint8).numpy()


def _e5m2_rounding_patterns():
    """All sign/exponent/top-2-mantissa combinations with low bits at and
    around e5m2's rounding midpoint (bit 20) and its subnormal midpoints."""
    hi = np.arange(1 << 11, dtype=np.uint32) << np.uint32(21)
    lows = np.array([0, 1, 0xFFFFF, 0x100000, 0x100001, 0x1FFFFF, 0x80000, 0x180000, 0x7FFFF, 0x40000],
                    np.uint32)
    f = (hi[:, None] | lows[None, :]).ravel().view(np.float32)
    return f[np.isfinite(f)]


def test_e5m2_encoder_vs_torch():
    rng = np.random.default_rng(21)
    f = np.concatenate([_e5m2_rounding_patterns(),
                        rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
                        (rng.standard_normal(500_000) * 3e4).astype(np.float32),
                        (rng.standard_normal(500_000) * 1e-4).astype(np.float32)])
    f = f[np.isfinite(f)]
    np.testing.assert_array_equal(oracle.f32_to_e5m2(f), _torch_e5m2_bits(f))


def test_e5m2_encoder_vs_brute_search():
    rng = np.random.default_rng(22)
    codes, vals = brute.e5m2_values()
    sv = np.sort(vals)
    mids = (sv[1:] + sv[:-1]) / 2
    f = np.concatenate([vals, mids, mids * (1 + 2**-20), mids * (1 - 2**-20),
                        [60000.0, 61440.0, -1e30, 57344.0 * (1 + 2**-20), -0.0, 2.0**-17, 2.0**-18],
                        rng.standard_normal(3000) * 4000]).astype(np.float32)
    np.testing.assert_array_equal(oracle.f32_to_e5m2(f), brute.e5m2_encode(f))


def test_e5m2_decode_all_codes():
    codes, vals = brute.e5m2_values()
    np.testing.assert_array_equal(oracle.e5m2_to_f32(codes).astype(np.float64), vals)
    np.testing.assert_array_equal(oracle.f32_to_e5m2(vals.astype(np.float32)), codes)
    allc = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(allc).view(torch.float8_e5m2).float().numpy()
    got = oracle.e5m2_to_f32(allc)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def _hand_values(tokens, n):
    x = np.zeros(n, np.float32)
    for kv in tokens:
        i, v = kv.split(":")
        x[int(i)] = float.fromhex(v) if "p" in v else float(v)
    return x


def _hand_codes(tokens, n):
    q = np.zeros(n, np.uint8)
    for kv in tokens:
        i, v = kv.split(":")
        q[int(i)] = int(v, 16)
    return q


def test_fp8_e5m2_golden(golden):
    g = golden("fp8_e5m2_hand.txt")
    x = _hand_values(g["x"], 256)
    xb = gi.f32_to_bf16_bits(x)
    assert (gi.bf16_bits_to_f32(xb) == x).all(), "fixture values must be bf16-exact"
    for mode, skey, qkey in [(0, "scale_fp32_bits", "q_fp32"), (1, "scale_pow2_bits", "q_pow2")]:
        q, s = oracle.quant_row_e5m2(xb, mode)
        np.testing.assert_array_equal(s.view(np.uint32), _ints(g[skey]).astype(np.uint32))
        np.testing.assert_array_equal(q, _hand_codes(g[qkey], 256))
    q, sb = oracle.quant_row_e5m2(xb, 2)
    np.testing.assert_array_equal(sb, _ints(g["ue8m0"]))
    np.testing.assert_array_equal(q, _hand_codes(g["q_pow2"], 256))


def test_e5m2_quant_closed_forms():
    """Block max -> +-57344 with fp32 scales; dequantisation within half an
    e5m2 step; power-of-two scales minimal, their codes torch's exact cast."""
    rng = np.random.default_rng(23)
    H = 1024
    xf = (rng.standard_normal((48, H)) * 3).astype(np.float32)
    xf[0, :128] = 0.0
    xf[1, 128:256] = 1e-39                     # bf16 subnormals
    xf[2, 256:384] = np.float32(2.0 ** -133)   # the smallest bf16 subnormal
    xf[3, 384:512] = 3e38
    xf[4, ::3] *= 1e5
    xb = gi.f32_to_bf16_bits(xf)
    xv = gi.bf16_bits_to_f32(xb).reshape(48, H // 128, 128).astype(np.float64)
    for t in range(48):
        q, s = oracle.quant_row_e5m2(xb[t], 0)
        qp, sp = oracle.quant_row_e5m2(xb[t], 1)
        qu, su = oracle.quant_row_e5m2(xb[t], 2)
        for b in range(H // 128):
            blk = xv[t, b]
            qb, qpb, qub = (a[b * 128:(b + 1) * 128] for a in (q, qp, qu))
            amax = np.abs(blk).max()
            if amax == 0:
                assert s[b] == 0 and sp[b] == 0 and su[b] == 0
                assert not qb.any() and not qpb.any() and not qub.any()
                continue
            i = int(np.argmax(np.abs(blk)))
            assert qb[i] & 0x7F == 0x7B                     # the block max saturates the format
            dq = oracle.e5m2_to_f32(qb).astype(np.float64) * np.float64(s[b])
            # half a step: 2^-3 relative for normals; half the subnormal step
            # 2^-16 times the scale; plus fp32 rounding of x / s near 57344
            bound = 2.0 ** -3 * np.abs(blk) + 2.0 ** -17 * float(s[b]) + 2.0 ** -20 * amax
            assert (np.abs(dq - blk) <= bound).all()
            s0 = np.float64(np.float32(amax) / np.float32(57344.0))
            m, _ = np.frexp(np.float64(sp[b]))
            assert m == 0.5 and sp[b] >= s0 and sp[b] / 2 < s0
            np.testing.assert_array_equal(qpb, _torch_e5m2_bits((blk / np.float64(sp[b])).astype(np.float32)))
            ue = max(float(sp[b]), 2.0 ** -127)
            assert su[b] == int(np.log2(ue)) + 127
            np.testing.assert_array_equal(qub, _torch_e5m2_bits((blk / ue).astype(np.float32)))


def test_dispatch_rows_moves_any_row_type():
    idx = _random_routing(np.random.default_rng(6), 30, 3, 8, 0.2, True, 0.0)
    L = oracle.layout(idx, 8, 2)
    N = int(L["expert_offsets"][-1])
    src = np.random.default_rng(7).integers(0, 256, (30, 48), dtype=np.uint8)
    out = oracle.dispatch_rows(src, L["row_of_slot"], N)
    for t, k in zip(*np.nonzero(L["row_of_slot"] >= 0)):
        np.testing.assert_array_equal(out[L["row_of_slot"][t, k]], src[t])


# ------------------------------------------------------------------ dense routing maps

def test_routing_map_golden(golden):
    g = golden("routing_map_hand.txt")
    T, K, E = (int(g[k][0]) for k in "TKE")
    idx = _ints(g["topk_idx"]).reshape(T, K)
    w = np.array([float(v) for v in g["topk_weights"]], np.float32).reshape(T, K)
    rm, pr, st = oracle.topk_to_routing_map(idx, w, E)
    assert st == oracle.OK
    np.testing.assert_array_equal(rm.ravel(), _ints(g["routing_map"]))
    np.testing.assert_array_equal(pr.ravel(), np.array([float(v) for v in g["probs"]], np.float32))
    bi, bw, st = oracle.routing_map_to_topk(rm, pr, K)
    assert st == oracle.OK
    np.testing.assert_array_equal(bi.ravel(), _ints(g["back_topk_idx"]))
    np.testing.assert_array_equal(bw.ravel(), np.array([float(v) for v in g["back_topk_weights"]], np.float32))


@pytest.mark.parametrize("seed", [0, 1])
def test_routing_map_round_trip_vs_numpy(seed):
    inp = gi.make("skewed", seed, T=500, with_y=False)
    w_ = inp.w
    rm, pr, st = oracle.topk_to_routing_map(inp.topk_idx, inp.topk_weights, w_.E)
    # numpy: scatter the valid slots
    want = np.zeros((w_.T, w_.E), np.uint8)
    want_p = np.zeros((w_.T, w_.E), np.float32)
    t, k = np.nonzero(inp.topk_idx >= 0)
    want[t, inp.topk_idx[t, k]] = 1
    want_p[t, inp.topk_idx[t, k]] = inp.topk_weights[t, k]
    np.testing.assert_array_equal(rm, want)
    np.testing.assert_array_equal(pr, want_p)
    # back to sparse: each token's experts sorted ascending, weights follow
    bi, bw, st = oracle.routing_map_to_topk(rm, pr, w_.K)
    for tt in range(w_.T):
        valid = inp.topk_idx[tt] >= 0
        order = np.argsort(inp.topk_idx[tt][valid])
        n = int(valid.sum())
        np.testing.assert_array_equal(bi[tt, :n], inp.topk_idx[tt][valid][order])
        np.testing.assert_array_equal(bw[tt, :n], inp.topk_weights[tt][valid][order])
        assert (bi[tt, n:] == -1).all() and (bw[tt, n:] == 0).all()
    # the layout of the converted routing differs only in slot order inside tokens
    a = oracle.layout(inp.topk_idx, w_.E, w_.R)
    b = oracle.layout(bi, w_.E, w_.R)
    for key in ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "expert_offsets"]:
        np.testing.assert_array_equal(a[key], b[key])


def test_routing_map_repeated_expert_and_no_probs():
    """Hand-worked: a token naming expert 1 twice gets one map entry whose
    probability is the sum of both weights in ascending k (nccl_ep.cc,
    ncclEpDispatch: sparse_to_dense_prob, read as a sum over the slots naming
    the expert): 0.25 + 0.5 = 0.75. A map given without probabilities converts
    back with unit weights, the unweighted convention of the combine (no
    weights means 1), and -1 / 0 in the unused slots."""
    idx = np.array([[1, 1, 3]], np.int64)
    w = np.array([[0.25, 0.5, 0.125]], np.float32)
    rm, pr, st = oracle.topk_to_routing_map(idx, w, 4)
    assert st == oracle.OK
    assert rm.tolist() == [[0, 1, 0, 1]]
    assert pr.tolist() == [[0.0, 0.75, 0.0, 0.125]]
    bi, bw, st = oracle.routing_map_to_topk(rm, None, 3)
    assert st == oracle.OK
    assert bi.tolist() == [[1, 3, -1]] and bw.tolist() == [[1.0, 1.0, 0.0]]


def test_routing_map_too_many_experts():
    rm = np.ones((2, 8), np.uint8)
    _, _, st = oracle.routing_map_to_topk(rm, None, 4)
    assert st == oracle.ERR_ARG


# ------------------------------------------------------------------ strided layout

def test_layout_strided_golden(golden):
    g = golden("layout_hand_strided.txt")
    T, K, E, R, C = (int(g[k][0]) for k in "TKERC")
    idx = _ints(g["topk_idx"]).reshape(T, K)
    L = oracle.layout_strided(idx, E, R, C)
    assert L["status"] == oracle.OK
    np.testing.assert_array_equal(L["num_tokens_per_expert"], _ints(g["num_tokens_per_expert"]))
    np.testing.assert_array_equal(L["expert_offsets"], _ints(g["expert_offsets"]))
    np.testing.assert_array_equal(L["row_of_slot"].ravel(), _ints(g["row_of_slot"]))


@pytest.mark.parametrize("cap", [1, 2, 5, 64, 1000])
@pytest.mark.parametrize("case", CORNERS[:8])
def test_layout_strided_vs_brute(case, cap):
    T, K, E, R, drop_p, distinct, bad_p = case
    idx = _random_routing(np.random.default_rng(cap), T, K, E, drop_p, distinct, bad_p)
    a = oracle.layout_strided(idx, E, R, cap)
    b = brute.layout_strided(idx, E, R, cap)
    for key in ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "expert_offsets",
                "row_of_slot", "status"]:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    r = a["row_of_slot"]
    kept = r[r >= 0]
    assert len(np.unique(kept)) == len(kept)                      # no row used twice
    assert ((kept // cap) == idx[r >= 0]).all()                   # each row inside its expert's block


# ------------------------------------------------------------------ non-expand layout

def test_layout_nonexpand_golden(golden):
    g = golden("layout_hand_nonexpand.txt")
    T, K, E, R = (int(g[k][0]) for k in "TKER")
    idx = _ints(g["topk_idx"]).reshape(T, K)
    L = oracle.layout_nonexpand(idx, E, R)
    assert L["status"] == oracle.OK
    np.testing.assert_array_equal(L["num_tokens_per_rank"], _ints(g["num_tokens_per_rank"]))
    np.testing.assert_array_equal(L["rank_offsets"], _ints(g["rank_offsets"]))
    np.testing.assert_array_equal(L["row_of_slot"].ravel(), _ints(g["row_of_slot"]))
    n = int(L["rank_offsets"][-1])
    ri, rw0 = oracle.nonexpand_recv_topk(idx, None, L["row_of_slot"], E, R, n)
    np.testing.assert_array_equal(ri.ravel(), _ints(g["recv_topk_idx"]))
    assert (rw0 == 0).all()                 # no weights given: every entry 0
    w = np.array([float(v) for v in g["topk_weights"]], np.float32).reshape(T, K)
    ri2, rw = oracle.nonexpand_recv_topk(idx, w, L["row_of_slot"], E, R, n)
    np.testing.assert_array_equal(ri2, ri)
    np.testing.assert_array_equal(rw.ravel(), np.array([float(v) for v in g["recv_topk_weights"]], np.float32))


@pytest.mark.parametrize("case", CORNERS)
def test_layout_nonexpand_vs_brute(case):
    T, K, E, R, drop_p, distinct, bad_p = case
    idx = _random_routing(np.random.default_rng(T), T, K, E, drop_p, distinct, bad_p)
    a = oracle.layout_nonexpand(idx, E, R)
    b = brute.layout_nonexpand(idx, E, R)
    for key in ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "rank_offsets",
                "row_of_slot", "status"]:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    # each (token, rank) pair owns exactly one row; rows of a rank lie in its range
    n = int(a["rank_offsets"][-1])
    r = a["row_of_slot"]
    assert np.array_equal(np.sort(r[r >= 0]), np.arange(n))
    assert n == int(a["is_token_in_rank"].sum())


# ------------------------------------------------------------------ division, not reciprocal

def _reciprocal_traps(F, values, torch_codes, limit=6):
    """(amax, x) bf16 pairs, 0 < x <= amax, for which the fp8 code of RN(x / s)
    differs from that of RN(x * RN(1 / s)), s = RN(amax / F) in fp32: a
    quantiser that multiplies by the reciprocal instead of dividing gets these
    wrong. Found with numpy's IEEE fp32 arithmetic, the fp8 code table and
    torch's fp8 cast only: x is taken next to s times each rounding midpoint
    of the fp8 grid, where the two quotients can fall on either side."""
    v = np.unique(np.abs(values))
    mids = (v[1:] + v[:-1]) / 2
    mids = mids[mids < F]
    e = np.arange(107, 148, dtype=np.uint32)                    # amax in [2^-20, 2^21)
    m = (((e[:, None] << 7) | np.arange(128, dtype=np.uint32)[None, :]).ravel() << 16).view(np.float32)
    s = m / np.float32(F)
    r = np.float32(1.0) / s
    found = []
    for M in mids:
        target = (np.float64(M) * s.astype(np.float64)).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
        for bits in (target, target + np.uint32(0x10000)):
            x = bits.view(np.float32)
            ok = (x > 0) & (x <= m)
            qd, qr = x / s, x * r
            hit = ok & (torch_codes(qd) != torch_codes(qr))
            for i in np.flatnonzero(hit):
                found.append((m[i], x[i], int(torch_codes(qd[i:i + 1])[0])))
                if len(found) >= limit:
                    return found
    return found


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantiser_divides_rather_than_multiplying_by_the_reciprocal(fmt):
    """The reading of the fp8 formula is q = fp8(x / scale) by IEEE division.
    On blocks built around the traps above, the oracle's code for x is the
    code of the true quotient, not of x times the rounded reciprocal."""
    if fmt == "e4m3":
        F, values, codes_of = 448.0, brute.e4m3_values()[1], _torch_e4m3_bits
        quant = lambda row: oracle.quant_row_e4m3(row)
    else:
        F, values, codes_of = 57344.0, brute.e5m2_values()[1], _torch_e5m2_bits
        quant = lambda row: oracle.quant_row_e5m2(row, 0)
    traps = _reciprocal_traps(F, values, codes_of)
    assert len(traps) >= 3, "the search should find traps in this amax range"
    for amax, x, code in traps:
        row = np.zeros(128, np.uint16)
        row[0] = gi.f32_to_bf16_bits(np.array([amax], np.float32))[0]
        row[1] = gi.f32_to_bf16_bits(np.array([x], np.float32))[0]
        q, sc = quant(row)
        assert sc[0] == np.float32(amax) / np.float32(F)
        assert q[1] == code, (fmt, float(amax), float(x))
