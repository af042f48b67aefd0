"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs.

Bars: layout arrays, slot -> row map, permuted bf16 rows, fp8 bytes and
scales, receive-side token ids and weights are bit-exact; combine is within
1 bf16 ulp per element (the stated tolerance; both sides use the same fp32
fused multiply-add order, so the test also reports exact matches).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gen import inputs as gi

pytestmark = pytest.mark.gpu

GUARD = 8          # extra rows / bytes after every output, checked untouched
SENT16 = 0x7BAD    # sentinel bf16 bits in guard rows
SENT8 = 0xA5


@pytest.fixture(scope="module")
def ep():
    import combine_get_dispatch_layout_gb300 as m
    from combine_get_dispatch_layout_gb300.build import build

    build()
    m.lib()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return m


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda() if dtype is None else t.cuda().view(dtype)


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place (sign-magnitude made monotonic)."""
    def mono(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, 0x8000 - u, u)
    return np.abs(mono(a) - mono(b))


class Run:
    """One layout (+ optional dispatch / combine) on the GPU with guard bands."""

    def __init__(self, ep, idx: np.ndarray, E: int, R: int, handle=None):
        self.ep = ep
        self.T, self.K = idx.shape
        self.E, self.R = E, R
        T, K = self.T, self.K
        self.idx = _dev(idx)
        self.cnt = torch.full((E + GUARD,), -7, dtype=torch.int32, device="cuda")
        self.ntr = torch.full((R + GUARD,), -7, dtype=torch.int32, device="cuda")
        self.itr = torch.full((T * R + GUARD,), SENT8, dtype=torch.uint8, device="cuda")
        self.off = torch.full((E + 1 + GUARD,), -7, dtype=torch.int32, device="cuda")
        self.h = ep.ep_layout(self.idx, E, R, self.cnt, self.ntr, self.itr, self.off, handle=handle)
        self.rows = torch.full((T * K + GUARD,), -9, dtype=torch.int32, device="cuda")
        ep.ep_handle_copy_row_of_slot(self.h, self.rows)
        torch.cuda.synchronize()

    def layout(self):
        E, R, T, K = self.E, self.R, self.T, self.K
        c, n, i, o, r = (self.cnt.cpu().numpy(), self.ntr.cpu().numpy(), self.itr.cpu().numpy(),
                         self.off.cpu().numpy(), self.rows.cpu().numpy())
        assert (c[E:] == -7).all() and (n[R:] == -7).all() and (i[T * R:] == SENT8).all()
        assert (o[E + 1:] == -7).all() and (r[T * K:] == -9).all(), "guard band overwritten"
        return dict(num_tokens_per_expert=c[:E], num_tokens_per_rank=n[:R],
                    is_token_in_rank=i[:T * R].reshape(T, R), expert_offsets=o[:E + 1],
                    row_of_slot=r[:T * K].reshape(T, K))


def check_layout(run: Run, ref: dict):
    got = run.layout()
    for k in ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "expert_offsets",
              "row_of_slot"]:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


def dispatch_bf16(ep, run, x, N, weights=None):
    T, H = x.shape
    recv = torch.full((N + GUARD, H), SENT16, dtype=torch.int16, device="cuda")
    src = torch.full((N + GUARD,), -5, dtype=torch.int32, device="cuda")
    rw = torch.full((N + GUARD,), -3.0, dtype=torch.float32, device="cuda") if weights is not None else None
    wt = _dev(weights) if weights is not None else None
    ep.ep_dispatch(run.h, _dev(x.view(np.int16)), ep.EP_DTYPE_BF16, recv, N + GUARD,
                   recv_src_token=src, recv_weights=rw, topk_weights=wt)
    torch.cuda.synchronize()
    r = recv.cpu().numpy().view(np.uint16)
    s = src.cpu().numpy()
    assert (r[N:] == SENT16).all() and (s[N:] == -5).all(), "rows >= N written"
    w = None
    if rw is not None:
        w = rw.cpu().numpy()
        assert (w[N:] == -3.0).all()
        w = w[:N]
    return r[:N], s[:N], w


def dispatch_fp8(ep, run, x, N):
    T, H = x.shape
    q = torch.full((N + GUARD, H), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.full((N + GUARD, H // 128), -1.0, dtype=torch.float32, device="cuda")
    src = torch.full((N + GUARD,), -5, dtype=torch.int32, device="cuda")
    ep.ep_dispatch(run.h, _dev(x.view(np.int16)), ep.EP_DTYPE_FP8_E4M3, q, N + GUARD, recv_scales=sc,
                   recv_src_token=src)
    torch.cuda.synchronize()
    qn, sn = q.cpu().numpy(), sc.cpu().numpy()
    assert (qn[N:] == SENT8).all() and (sn[N:] == -1.0).all(), "rows >= N written"
    return qn[:N], sn[:N], src.cpu().numpy()[:N]


def combine(ep, run, y, weights, H):
    T = run.T
    out = torch.full((T + 1, H), SENT16, dtype=torch.int16, device="cuda")
    yd = _dev(y.view(np.int16)) if y is not None and y.shape[0] > 0 else None
    wt = _dev(weights) if weights is not None else None
    rows = 0 if y is None else y.shape[0]
    if yd is None:
        yd = torch.empty((1, H), dtype=torch.int16, device="cuda")
    ep.ep_combine(run.h, yd, out, topk_weights=wt, y_rows=rows)
    torch.cuda.synchronize()
    o = out.cpu().numpy().view(np.uint16)
    assert (o[T:] == SENT16).all(), "combine wrote past T rows"
    return o[:T]


def assert_combine(got, want):
    assert got.shape == want.shape
    d = bf16_ulp_dist(got, want)
    if d.size == 0:
        return
    assert d.max() <= 1, f"combine off by {d.max()} ulp at {np.argwhere(d > 1)[:5]}"
    # same fp32 fma order on both sides: expect exact equality
    assert (d == 0).all(), f"{int((d > 0).sum())} of {d.size} elements differ by 1 ulp"


def full_path(ep, inp, fp8=False, weights=True):
    w = inp.w
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    assert ref["status"] == oracle.OK
    run = Run(ep, inp.topk_idx, w.E, w.R)
    check_layout(run, ref)
    n, err = ep.ep_handle_query(run.h)
    N = int(ref["expert_offsets"][-1])
    assert (n, err) == (N, 0)
    wt = inp.topk_weights if weights else None
    r_x, r_src, r_w = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], N, wt)
    g_x, g_src, g_w = dispatch_bf16(ep, run, inp.x, N, wt)
    np.testing.assert_array_equal(g_x, r_x)
    np.testing.assert_array_equal(g_src, r_src)
    if wt is not None:
        np.testing.assert_array_equal(g_w.view(np.uint32), r_w.view(np.uint32))
    if fp8:
        r_q, r_s, r_src8, _ = oracle.dispatch_e4m3(inp.x, ref["row_of_slot"], N)
        g_q, g_s, g_src8 = dispatch_fp8(ep, run, inp.x, N)
        np.testing.assert_array_equal(g_s.view(np.uint32), r_s.view(np.uint32))
        np.testing.assert_array_equal(g_q, r_q)
        np.testing.assert_array_equal(g_src8, r_src8)
    y = inp.y if inp.y is not None else r_x          # identity expert
    got = combine(ep, run, y, wt, w.H)
    want = oracle.combine(y, ref["row_of_slot"], wt)
    assert_combine(got, want)
    run.h.destroy()


# ------------------------------------------------------------------ workloads

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny(ep, seed):
    full_path(ep, gi.make("tiny", seed), fp8=True)


# seed 0 is the measured workload; seeds 1 and 2 check robustness
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode(ep, seed):
    full_path(ep, gi.make("decode", seed), fp8=True)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prefill_bf16(ep, seed):
    full_path(ep, gi.make("prefill", seed))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prefill_fp8(ep, seed):
    full_path(ep, gi.make("fp8", seed), fp8=True)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_skewed(ep, seed):
    full_path(ep, gi.make("skewed", seed), fp8=True)


@pytest.mark.parametrize("name,T", [("prefill", 777), ("skewed", 1001), ("fp8", 333)])
def test_ragged_token_counts(ep, name, T):
    full_path(ep, gi.make(name, 3, T=T), fp8=True)


# ------------------------------------------------------------------ edge cases

def _workload(T, H, E, K, R, **kw):
    return gi.Workload("edge", T=T, H=H, E=E, K=K, R=R, **kw)


@pytest.mark.parametrize("w", [
    _workload(1, 128, 1, 1, 1),                          # T=1, K=1, E=R=1
    _workload(37, 264, 5, 3, 5, drop_p=0.3),             # E == R, ragged H (not a multiple of 256)
    _workload(100, 384, 16, 4, 1, drop_p=0.1),           # R == 1, odd number of fp8 blocks
    _workload(513, 640, 64, 6, 4, routing="zipf", drop_p=0.05),
    _workload(300, 8, 8, 8, 2),                          # H = 8 (one vector), K == E
    _workload(64, 1152, 32, 32, 8),                      # K = 32 (maximum top-k)
    _workload(200, 136, 4096, 8, 1024),                  # maximum E and R
    _workload(300, 128, 512, 8, 64),                     # R > 32 on the single-cluster path
    _workload(500, 128, 256, 8, 32, drop_p=0.1),         # R = 32: every rank bit in use
    _workload(21504, 64, 64, 6, 4, routing="zipf"),      # K = 6: largest routing of the 8-round cluster kernel
    _workload(21505, 64, 64, 6, 4, routing="zipf"),      # one token more: its packed 16-round instance
    _workload(43520, 64, 64, 6, 4, routing="zipf"),      # K = 6: largest single-cluster routing (512 slots a warp)
    _workload(43521, 64, 64, 6, 4, routing="zipf"),      # one token more: multi-block path
    _workload(32768, 64, 256, 8, 8, drop_p=0.02),        # 2^18 slots on the single cluster
    _workload(8000, 128, 4096, 8, 1024, drop_p=0.02),    # maximum E and R, 64k slots (multi-block)
    _workload(9000, 128, 2048, 32, 256, drop_p=0.02),    # maximum top-k above 2^18 slots
])
def test_edge_shapes(ep, w):
    inp = gi.make(w, 11)
    full_path(ep, inp, fp8=(w.H % 128 == 0))


@pytest.mark.parametrize("T", [480, 521, 522, 560])
def test_dispatch_across_its_item_size_switch(ep, T):
    """A bf16 dispatch grid below one wave of resident warps moves one 16-byte
    vector per lane instead of two. At H=7168 the two-vector grid has 14 items
    a token, so on a 152-SM GB300 (7296 resident warps) the switch falls
    between 521 and 522 tokens; both sides, with fp8 and the aligned layout's
    pad rows, must match the oracle."""
    inp = gi.make("prefill", 21, T=T)
    full_path(ep, inp, fp8=True)
    full_path_aligned(ep, gi.make("prefill", 22, T=T), 64)


@pytest.mark.parametrize("T,K,E,R,ctas", [
    (128, 2, 8, 2, 4),        # the tiny routing: 256 slots
    (64, 8, 256, 8, 4),       # 512 slots
    (256, 8, 256, 8, 8),      # the decode routing: 2048 slots, one round for each of 64 warps
    (512, 8, 256, 8, 16),     # 4096 slots
])
def test_small_routings_take_smaller_clusters(ep, T, K, E, R, ctas):
    """A small routing runs on the fewest CTAs (at least 4) that give each warp
    at most one 32-slot round; its outputs still match the oracle."""
    if ep.ep_layout_cluster_ctas(1024, 8, 256, 8) < 16:
        pytest.skip("this GPU does not co-schedule 16-CTA clusters")
    assert ep.ep_layout_cluster_ctas(T, K, E, R) == ctas
    idx = np.argsort(np.random.default_rng(T).random((T, E)), axis=1)[:, :K].astype(np.int64)
    run = Run(ep, idx, E, R)
    assert ep.ep_handle_layout_kernels(run.h) == 1
    check_layout(run, oracle.layout(idx, E, R))
    run.h.destroy()


@pytest.mark.parametrize("T,K,E,R,kernels", [
    (21504, 6, 64, 4, 1),     # 8 rounds a warp: the unpacked cluster instance
    (21505, 6, 64, 4, 1),     # 9 rounds: the packed 16-round instance
    (43520, 6, 64, 4, 1),     # 16 rounds: the largest single-cluster routing at top-6
    (43521, 6, 64, 4, 3),     # one token more: the three-kernel path
    (32768, 8, 256, 8, 1),    # 2^18 slots: the largest single-cluster routing
    (32769, 8, 256, 8, 3),    # above 2^18 slots
])
def test_layout_path_at_the_boundaries(ep, T, K, E, R, kernels):
    """The boundary routings take the path their size implies. These limits
    assume 16-CTA clusters; on a GPU that co-schedules only 8 the cluster
    holds half as many slots and the test is skipped."""
    if ep.ep_layout_cluster_ctas(1024, 8, 256, 8) < 16:
        pytest.skip("this GPU does not co-schedule 16-CTA clusters")
    assert ep.ep_layout_cluster_ctas(T, K, E, R) == (16 if kernels == 1 else 0)
    w = _workload(T, 64, E, K, R, routing="zipf")
    inp = gi.make(w, 13, with_y=False)
    run = Run(ep, inp.topk_idx, E, R)
    assert ep.ep_handle_layout_kernels(run.h) == kernels
    check_layout(run, oracle.layout(inp.topk_idx, E, R))
    run.h.destroy()


def test_large_routing_multiblock_path(ep):
    """Routings above 2^18 slots take the multi-block layout path."""
    w = _workload(40000, 128, 64, 8, 4, routing="zipf", drop_p=0.05)
    full_path(ep, gi.make(w, 12), fp8=True)


def test_all_dropped(ep):
    w = _workload(50, 256, 8, 2, 2, drop_p=1.0)
    inp = gi.make(w, 0)
    assert inp.num_valid == 0
    full_path(ep, inp, fp8=True)


def test_empty_tokens(ep):
    idx = np.zeros((0, 4), np.int64)
    run = Run(ep, idx, 8, 2)
    got = run.layout()
    assert (got["num_tokens_per_expert"] == 0).all() and (got["expert_offsets"] == 0).all()
    assert (got["num_tokens_per_rank"] == 0).all()
    assert ep.ep_handle_query(run.h) == (0, 0)


def test_one_expert_takes_all(ep):
    idx = np.full((4000, 1), 5, np.int64)
    x = gi.normal_bf16(np.random.SeedSequence(4), 4000, 256)
    inp = gi.Inputs(w=_workload(4000, 256, 8, 1, 4), seed=0, x=x, topk_idx=idx,
                    topk_weights=np.ones((4000, 1), np.float32),
                    y=gi.normal_bf16(np.random.SeedSequence(5), 4000, 256), num_valid=4000)
    full_path(ep, inp, fp8=True)


def test_duplicate_experts_in_token(ep):
    rng = np.random.default_rng(0)
    idx = rng.integers(0, 6, size=(500, 4)).astype(np.int64)
    idx[rng.random((500, 4)) < 0.1] = -1
    x = gi.normal_bf16(np.random.SeedSequence(6), 500, 128)
    N = int((idx >= 0).sum())
    inp = gi.Inputs(w=_workload(500, 128, 6, 4, 3), seed=0, x=x, topk_idx=idx,
                    topk_weights=rng.random((500, 4)).astype(np.float32),
                    y=gi.normal_bf16(np.random.SeedSequence(7), N, 128), num_valid=N)
    full_path(ep, inp, fp8=True)


def test_combine_signed_zeros_and_null_weights(ep):
    rng = np.random.default_rng(1)
    T, K, E, R, H = 64, 4, 8, 2, 256
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    N = T * K
    y = gi.normal_bf16(np.random.SeedSequence(8), N, H)
    y[::3, ::5] = 0x8000        # -0
    y[1::3, ::7] = 0x0000       # +0
    inp = gi.Inputs(w=_workload(T, H, E, K, R), seed=0, x=gi.normal_bf16(np.random.SeedSequence(9), T, H),
                    topk_idx=idx, topk_weights=np.zeros((T, K), np.float32), y=y, num_valid=N)
    full_path(ep, inp)                     # all-zero weights: every output is +0
    full_path(ep, inp, weights=False)      # NULL weights: plain sums


def test_fp8_special_blocks(ep):
    rng = np.random.default_rng(2)
    T, H = 48, 1024
    xf = (rng.standard_normal((T, H)) * 2).astype(np.float32)
    xf[0, :128] = 0.0
    xf[1, 128:256] = -0.0
    xf[2, 256:384] = 1e-38
    xf[3, 384:512] = 3e38
    xf[4, :] = np.float32(2.0 ** -133)    # bf16 subnormal amax
    xf[5, ::2] *= 1e4
    x = gi.f32_to_bf16_bits(xf)
    idx = np.argsort(rng.random((T, 16)), axis=1)[:, :3].astype(np.int64)
    inp = gi.Inputs(w=_workload(T, H, 16, 3, 4), seed=0, x=x, topk_idx=idx,
                    topk_weights=np.full((T, 3), 1 / 3, np.float32), y=None, num_valid=3 * T)
    full_path(ep, inp, fp8=True)


def _sweep_inputs(amaxes):
    """Blocks holding every finite bf16 pattern of magnitude <= amax, with amax
    itself as the block's last element, for each amax."""
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = gi.bf16_bits_to_f32(pats)
    pats = pats[np.isfinite(f)]
    rows = []
    for amax in amaxes:
        vals = gi.bf16_bits_to_f32(pats)
        vals = vals[np.abs(vals) <= amax]
        per = 127
        nblk = (len(vals) + per - 1) // per
        blk = np.zeros((nblk, 128), np.float32)
        flat = np.zeros(nblk * per, np.float32)
        flat[:len(vals)] = vals
        blk[:, :per] = flat.reshape(nblk, per)
        blk[:, per] = amax
        rows.append(blk)
    allb = np.concatenate(rows)
    H = 1024
    nb = (len(allb) + 7) // 8
    pad = np.zeros((nb * 8 - len(allb), 128), np.float32)
    x = gi.f32_to_bf16_bits(np.concatenate([allb, pad]).reshape(nb, H))
    idx = np.zeros((nb, 1), np.int64)
    return gi.Inputs(w=_workload(nb, H, 1, 1, 1), seed=0, x=x, topk_idx=idx,
                     topk_weights=np.ones((nb, 1), np.float32), y=None, num_valid=nb)


def test_fp8_encoder_sweep_all_bf16(ep):
    """Every finite bf16 pattern through the quantiser under several block scales."""
    full_path(ep, _sweep_inputs([448.0, 1.0, 3.0, 1e-3, 7.5e7, 2.0 ** -120]), fp8=True)


def test_invalid_expert_ids(ep):
    rng = np.random.default_rng(3)
    T, K, E, R = 200, 4, 16, 4
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    idx[5, 1] = E
    idx[17, 0] = -3
    idx[100, 3] = 1 << 40
    ref = oracle.layout(idx, E, R)
    assert ref["status"] == oracle.ERR_EXPERT
    run = Run(ep, idx, E, R)
    check_layout(run, ref)                       # bad slots are treated as dropped
    n, err = ep.ep_handle_query(run.h)
    assert err == ep.EP_ERR_INVALID_EXPERT and n == int(ref["expert_offsets"][-1])
    x = torch.zeros((T, 128), dtype=torch.bfloat16, device="cuda")
    recv = torch.zeros((T * K, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch(run.h, x, ep.EP_DTYPE_BF16, recv, T * K)
    assert e.value.status == ep.EP_ERR_INVALID_EXPERT
    # a fresh layout with valid ids clears the latch on the same handle
    idx2 = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    run2 = Run(ep, idx2, E, R, handle=run.h)
    check_layout(run2, oracle.layout(idx2, E, R))
    assert ep.ep_handle_query(run2.h)[1] == 0
    ep.ep_dispatch(run2.h, x, ep.EP_DTYPE_BF16, recv, T * K)
    run.h.destroy()


def test_capacity_errors(ep):
    rng = np.random.default_rng(4)
    T, K, E, R, H = 100, 4, 8, 2, 64
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    idx[rng.random((T, K)) < 0.5] = -1
    N = int((idx >= 0).sum())
    run = Run(ep, idx, E, R)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    small = torch.zeros((N - 1, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch(run.h, x, ep.EP_DTYPE_BF16, small, N - 1)
    assert e.value.status == ep.EP_ERR_CAPACITY
    exact = torch.zeros((N, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_dispatch(run.h, x, ep.EP_DTYPE_BF16, exact, N)     # exactly N rows is enough
    out = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EPError) as e:
        ep.ep_combine(run.h, small, out)
    assert e.value.status == ep.EP_ERR_CAPACITY
    ep.ep_combine(run.h, exact, out)
    run.h.destroy()


def test_cached_row_count_follows_each_layout(ep):
    """N is read from the device once per layout; a new layout on the same
    handle must not be checked against the previous layout's N."""
    rng = np.random.default_rng(41)
    T, K, E, R, H = 300, 4, 16, 4, 64
    idx_a = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    idx_a[rng.random((T, K)) < 0.5] = -1
    idx_b = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    idx_b[rng.random((T, K)) < 0.1] = -1
    n_a, n_b = int((idx_a >= 0).sum()), int((idx_b >= 0).sum())
    assert n_a < n_b
    x = _dev(gi.normal_bf16(np.random.SeedSequence(42), T, H).view(np.int16), torch.bfloat16)
    run = Run(ep, idx_a, E, R)
    assert ep.ep_handle_query(run.h)[0] == n_a           # reads and caches N of layout A
    recv_a = torch.zeros((n_a, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_dispatch(run.h, x, ep.EP_DTYPE_BF16, recv_a, n_a)
    run_b = Run(ep, idx_b, E, R, handle=run.h)           # layout B on the same handle
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch(run_b.h, x, ep.EP_DTYPE_BF16, recv_a, n_a)
    assert e.value.status == ep.EP_ERR_CAPACITY
    recv_b = torch.full((n_b, H), -7.0, dtype=torch.bfloat16, device="cuda")
    ep.ep_dispatch(run_b.h, x, ep.EP_DTYPE_BF16, recv_b, n_b)   # N of B, from the cache now
    out = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(run_b.h, recv_b, out)
    torch.cuda.synchronize()
    ref = oracle.layout(idx_b, E, R)
    x_bits = x.view(torch.int16).cpu().numpy().view(np.uint16)
    r_x, _, _ = oracle.dispatch_bf16(x_bits, ref["row_of_slot"], n_b)
    np.testing.assert_array_equal(recv_b.view(torch.int16).cpu().numpy().view(np.uint16), r_x)
    np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16),
                                  oracle.combine(r_x, ref["row_of_slot"], None))
    # a layout with an invalid id after a clean one: the error is not hidden
    # by the clean layout's cached words
    idx_c = idx_b.copy()
    idx_c[7, 2] = E + 3
    run_c = Run(ep, idx_c, E, R, handle=run.h)
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch(run_c.h, x, ep.EP_DTYPE_BF16, recv_b, n_b)
    assert e.value.status == ep.EP_ERR_INVALID_EXPERT
    run.h.destroy()


def test_handle_reuse_grow_and_shrink(ep):
    h = None
    for (T, K, E, R, seed) in [(64, 2, 8, 2, 0), (5000, 8, 256, 8, 1), (10, 3, 6, 3, 2), (20000, 6, 64, 4, 3)]:
        rng = np.random.default_rng(seed)
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
        run = Run(ep, idx, E, R, handle=h)
        h = run.h
        check_layout(run, oracle.layout(idx, E, R))
    h.destroy()


def test_c_program_runs_the_step_through_the_abi(ep, tmp_path):
    """tests/c_abi_step.c links libep.so and the CUDA runtime directly, with
    no Python between the caller and the library, and runs layout -> bf16
    dispatch -> combine on device buffers it allocates itself; its outputs
    match the oracle."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.join(root, "combine_get_dispatch_layout_gb300")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_step")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(root, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(root, "tests", "c_abi_step.c"),
                    "-L", libdir, "-lep", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe], check=True)
    inp = gi.make("decode", 71)
    w = inp.w
    T, K, E, R, H = w.T, w.K, w.E, w.R, w.H
    n = inp.num_valid
    y = np.zeros((T * K, H), np.uint16)
    y[:n] = inp.y
    inp.topk_idx.astype(np.int64).tofile(tmp_path / "topk_idx.bin")
    inp.x.astype(np.uint16).tofile(tmp_path / "x.bin")
    y.tofile(tmp_path / "y.bin")
    inp.topk_weights.astype(np.float32).tofile(tmp_path / "w.bin")
    r = subprocess.run([exe, str(T), str(K), str(E), str(R), str(H), str(tmp_path)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    ref = oracle.layout(inp.topk_idx, E, R)
    np.testing.assert_array_equal(np.fromfile(tmp_path / "counts.bin", np.int32), ref["num_tokens_per_expert"])
    np.testing.assert_array_equal(np.fromfile(tmp_path / "offsets.bin", np.int32), ref["expert_offsets"])
    r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
    np.testing.assert_array_equal(np.fromfile(tmp_path / "recv.bin", np.uint16).reshape(n, H), r_x)
    r_out = oracle.combine(inp.y, ref["row_of_slot"], inp.topk_weights)
    np.testing.assert_array_equal(np.fromfile(tmp_path / "out.bin", np.uint16).reshape(T, H), r_out)


def test_handle_churn_returns_device_memory(ep):
    """Handles created, grown and destroyed many times give all their device
    memory back (default cudaMalloc hooks, so cudaMemGetInfo sees it)."""
    rng = np.random.default_rng(77)
    shapes = [(64, 2, 8, 2), (3000, 8, 256, 8), (40000, 6, 64, 4)]   # the last takes the multi-block path
    routings = [np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64) for T, K, E, R in shapes]
    dev_idx = [_dev(r) for r in routings]
    outs = [[torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(R, dtype=torch.int32, device="cuda"),
             torch.empty(T, R, dtype=torch.uint8, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda")]
            for T, K, E, R in shapes]

    def churn(n):
        for i in range(n):
            h = None
            for j in (i % 3, (i + 1) % 3, (i + 2) % 3):   # grow and shrink in varying order
                T, K, E, R = shapes[j]
                h = ep.ep_layout(dev_idx[j], E, R, *outs[j], handle=h)
            h.destroy()

    churn(3)                                   # library state that lives for the process
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    churn(200)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free0 - free1 < (2 << 20), (free0, free1)   # within the driver's allocation granularity
    ref = oracle.layout(routings[1], shapes[1][2], shapes[1][3])
    run = Run(ep, routings[1], shapes[1][2], shapes[1][3])
    check_layout(run, ref)
    run.h.destroy()


def test_layout_repeatable_on_same_handle(ep):
    """Back-to-back layouts on one handle (the done-counter reset path)."""
    inp = gi.make("skewed", 5, with_y=False)
    w = inp.w
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    h = None
    for _ in range(5):
        run = Run(ep, inp.topk_idx, w.E, w.R, handle=h)
        h = run.h
        check_layout(run, ref)
    h.destroy()


def test_side_stream(ep):
    """Calls honour the stream they are given."""
    inp = gi.make("decode", 4)
    w = inp.w
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    N = int(ref["expert_offsets"][-1])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        idx = _dev(inp.topk_idx)
        x = _dev(inp.x.view(np.int16), torch.bfloat16)
        cnt = torch.empty(w.E, dtype=torch.int32, device="cuda")
        ntr = torch.empty(w.R, dtype=torch.int32, device="cuda")
        itr = torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda")
        off = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
        h = ep.ep_layout(idx, w.E, w.R, cnt, ntr, itr, off, stream=s)
        recv = torch.empty(N, w.H, dtype=torch.bfloat16, device="cuda")
        ep.ep_dispatch(h, x, ep.EP_DTYPE_BF16, recv, N, stream=s)
    s.synchronize()
    r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], N)
    np.testing.assert_array_equal(_u16(recv), r_x)
    h.destroy()


def test_alloc_hooks(ep):
    """A caller-supplied allocator is used, and its failure is reported."""
    import ctypes

    calls = {"alloc": 0, "free": 0}
    keep = {}

    ALLOC = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t)
    FREE = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p)

    @ALLOC
    def alloc(pp, nbytes):
        calls["alloc"] += 1
        t = torch.empty(int(nbytes), dtype=torch.uint8, device="cuda")
        keep[t.data_ptr()] = t
        pp[0] = t.data_ptr()
        return 0

    @FREE
    def free(p):
        calls["free"] += 1
        keep.pop(p, None)
        return 0

    @ALLOC
    def failing(pp, nbytes):
        return 1

    idx = _dev(np.zeros((10, 2), np.int64))
    outs = [torch.empty(4, dtype=torch.int32, device="cuda"), torch.empty(2, dtype=torch.int32, device="cuda"),
            torch.empty(20, dtype=torch.uint8, device="cuda"), torch.empty(5, dtype=torch.int32, device="cuda")]
    h = ep.ep_layout(idx, 4, 2, *outs, alloc_fn=alloc, free_fn=free)
    torch.cuda.synchronize()
    assert outs[3].cpu().tolist() == [0, 20, 20, 20, 20]
    h.destroy()
    assert calls == {"alloc": 1, "free": 1}
    with pytest.raises(ep.EPError) as e:
        ep.ep_layout(idx, 4, 2, *outs, alloc_fn=failing, free_fn=free)
    assert e.value.status == ep.EP_ERR_ALLOC


def test_layout_path_selection(ep):
    """Routings up to the single-cluster limit take one launch, larger ones three."""
    small = gi.make("prefill", 0, with_y=False)
    big = gi.make(_workload(40000, 128, 64, 8, 4), 0, with_y=False)
    for inp, want in [(small, 1), (big, 3)]:
        w = inp.w
        run = Run(ep, inp.topk_idx, w.E, w.R)
        assert ep.ep_handle_layout_kernels(run.h) == want
        run.h.destroy()


def test_pinned_host_buffers(ep):
    """Host-resident inputs and outputs (pinned, mapped into the unified
    address space) give the same bytes as device buffers."""
    inp = gi.make("decode", 6)
    w = inp.w
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    N = int(ref["expert_offsets"][-1])
    h_idx = torch.from_numpy(inp.topk_idx).pin_memory()
    h_x = torch.from_numpy(inp.x.view(np.int16)).pin_memory()
    h_y = torch.from_numpy(inp.y.view(np.int16)).pin_memory()
    h_w = torch.from_numpy(inp.topk_weights).pin_memory()
    h_out = torch.full((w.T, w.H), SENT16, dtype=torch.int16).pin_memory()
    cnt = torch.empty(w.E, dtype=torch.int32, device="cuda")
    ntr = torch.empty(w.R, dtype=torch.int32, device="cuda")
    itr = torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda")
    off = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
    h = ep.ep_layout(h_idx, w.E, w.R, cnt, ntr, itr, off)
    recv = torch.empty(N, w.H, dtype=torch.int16, device="cuda")
    ep.ep_dispatch(h, h_x, ep.EP_DTYPE_BF16, recv, N)
    ep.ep_combine(h, h_y, h_out, topk_weights=h_w)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(off.cpu().numpy(), ref["expert_offsets"])
    r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], N)
    np.testing.assert_array_equal(recv.cpu().numpy().view(np.uint16), r_x)
    want = oracle.combine(inp.y, ref["row_of_slot"], inp.topk_weights)
    assert_combine(h_out.numpy().view(np.uint16), want)
    h.destroy()


# ------------------------------------------------------------------ aligned layout

def full_path_aligned(ep, inp, A, fp8=True):
    w = inp.w
    T, K, E, R, H = w.T, w.K, w.E, w.R, w.H
    ref = oracle.layout_aligned(inp.topk_idx, E, R, A)
    assert ref["status"] == oracle.OK
    n_pad = int(ref["expert_offsets"][-1])
    idx = _dev(inp.topk_idx)
    cnt = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    ntr = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    itr = torch.full((T, R), SENT8, dtype=torch.uint8, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    h = ep.ep_layout_aligned(idx, E, R, A, cnt, ntr, itr, off)
    rows = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    ep.ep_handle_copy_row_of_slot(h, rows)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref["num_tokens_per_expert"])
    np.testing.assert_array_equal(ntr.cpu().numpy(), ref["num_tokens_per_rank"])
    np.testing.assert_array_equal(itr.cpu().numpy(), ref["is_token_in_rank"])
    np.testing.assert_array_equal(off.cpu().numpy(), ref["expert_offsets"])
    np.testing.assert_array_equal(rows.cpu().numpy(), ref["row_of_slot"])
    assert ep.ep_handle_query(h) == (n_pad, 0)
    # bf16 dispatch: real rows and zeroed pad rows
    r_x, r_src, r_w = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n_pad, inp.topk_weights)
    oracle.fill_pad_rows(ref, r_x, src=r_src, weights=r_w)
    recv = torch.full((n_pad + GUARD, H), SENT16, dtype=torch.int16, device="cuda")
    src = torch.full((n_pad + GUARD,), -5, dtype=torch.int32, device="cuda")
    rw = torch.full((n_pad + GUARD,), -3.0, dtype=torch.float32, device="cuda")
    ep.ep_dispatch(h, _dev(inp.x.view(np.int16)), ep.EP_DTYPE_BF16, recv, n_pad + GUARD,
                   recv_src_token=src, recv_weights=rw, topk_weights=_dev(inp.topk_weights))
    torch.cuda.synchronize()
    g = recv.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(g[:n_pad], r_x)
    assert (g[n_pad:] == SENT16).all()
    np.testing.assert_array_equal(src.cpu().numpy()[:n_pad], r_src)
    np.testing.assert_array_equal(rw.cpu().numpy()[:n_pad].view(np.uint32), r_w.view(np.uint32))
    if fp8 and H % 128 == 0:
        r_q, r_s, _, _ = oracle.dispatch_e4m3(inp.x, ref["row_of_slot"], n_pad)
        oracle.fill_pad_rows(ref, r_q, scales=r_s)
        q = torch.full((n_pad, H), SENT8, dtype=torch.uint8, device="cuda")
        sc = torch.full((n_pad, H // 128), -1.0, dtype=torch.float32, device="cuda")
        ep.ep_dispatch(h, _dev(inp.x.view(np.int16)), ep.EP_DTYPE_FP8_E4M3, q, n_pad, recv_scales=sc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(q.cpu().numpy(), r_q)
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), r_s.view(np.uint32))
    # combine over a padded expert-output buffer
    y = gi.normal_bf16(np.random.SeedSequence(A), n_pad, H)
    out = torch.full((T, H), SENT16, dtype=torch.int16, device="cuda")
    ep.ep_combine(h, _dev(y.view(np.int16)) if n_pad else torch.empty((1, H), dtype=torch.int16, device="cuda"),
                  out, topk_weights=_dev(inp.topk_weights), y_rows=n_pad)
    torch.cuda.synchronize()
    assert_combine(out.cpu().numpy().view(np.uint16), oracle.combine(y, ref["row_of_slot"], inp.topk_weights))
    # the padded total is exactly enough; one row fewer is refused
    if n_pad > 0:
        small = torch.zeros((n_pad - 1, H), dtype=torch.int16, device="cuda")
        with pytest.raises(ep.EPError) as e:
            ep.ep_dispatch(h, _dev(inp.x.view(np.int16)), ep.EP_DTYPE_BF16, small, n_pad - 1)
        assert e.value.status == ep.EP_ERR_CAPACITY
    h.destroy()


@pytest.mark.parametrize("name,A,T", [("tiny", 3, None), ("decode", 16, None), ("skewed", 64, None),
                                      ("prefill", 128, None), ("fp8", 32, 1001), ("skewed", 7, 777)])
def test_aligned_workloads(ep, name, A, T):
    full_path_aligned(ep, gi.make(name, 1, T=T), A)


@pytest.mark.parametrize("w,A", [
    (_workload(50, 256, 8, 2, 2, drop_p=1.0), 8),                     # nothing routed: no pad rows
    (_workload(1, 128, 1, 1, 1), 1024),                               # maximum alignment
    (_workload(40000, 128, 64, 8, 4, routing="zipf", drop_p=0.05), 32),   # multi-block layout path
    (_workload(300, 128, 512, 8, 64), 5),                             # R > 32
])
def test_aligned_edges(ep, w, A):
    full_path_aligned(ep, gi.make(w, 2), A)


def test_aligned_rejects_bad_alignment(ep):
    idx = torch.zeros((4, 2), dtype=torch.int64, device="cuda")
    o = [torch.empty(8, dtype=torch.int32, device="cuda"), torch.empty(2, dtype=torch.int32, device="cuda"),
         torch.empty(8, dtype=torch.uint8, device="cuda"), torch.empty(9, dtype=torch.int32, device="cuda")]
    for A in (0, -1, 1025):
        with pytest.raises(ep.EPError) as e:
            ep.ep_layout_aligned(idx, 8, 2, A, *o)
        assert e.value.status == ep.EP_ERR_INVALID_ARG


# ------------------------------------------------------------------ backward

def _grad_w_bound(g_bits, y_bits, rows, H):
    """|fp32 kernel - float64| bound for the weight gradient: each thread sums
    8 * ceil(H/8/128) products with fused multiply-adds, then a 5-level shuffle
    tree and a 4-term sum, each step adding at most 2^-24 relative to the sum
    of |terms|."""
    n_terms = 8 * (-(-(H // 8) // 128)) + 8
    gf = np.abs(gi.bf16_bits_to_f32(g_bits).astype(np.float64))
    yf = np.abs(gi.bf16_bits_to_f32(y_bits).astype(np.float64))
    T, K = rows.shape
    mag = np.zeros((T, K))
    for k in range(K):
        v = rows[:, k] >= 0
        mag[v, k] = (gf[v] * yf[rows[v, k]]).sum(axis=1)
    return 1.01 * n_terms * 2.0**-24 * mag + 1e-30


def backward_path(ep, inp, A=1, weights=True):
    w = inp.w
    T, K, E, R, H = w.T, w.K, w.E, w.R, w.H
    ref = oracle.layout_aligned(inp.topk_idx, E, R, A)
    n = int(ref["expert_offsets"][-1])
    idx = _dev(inp.topk_idx)
    o = [torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(R, dtype=torch.int32, device="cuda"),
         torch.empty(T, R, dtype=torch.uint8, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda")]
    h = ep.ep_layout_aligned(idx, E, R, A, *o)
    rows = ref["row_of_slot"]
    y = gi.normal_bf16(np.random.SeedSequence(21), n, H)
    g = gi.normal_bf16(np.random.SeedSequence(22), T, H)
    wt = inp.topk_weights if weights else None
    # combine backward
    gy = torch.full((n + GUARD, H), SENT16, dtype=torch.int16, device="cuda")
    gw = torch.full((T, K), -9.0, dtype=torch.float32, device="cuda")
    ep.ep_combine_backward(h, _dev(g.view(np.int16)), y=_dev(y.view(np.int16)) if n else None,
                           topk_weights=_dev(wt) if wt is not None else None, grad_y=gy, grad_topk_weights=gw,
                           y_rows=n, grad_y_capacity=n + GUARD)
    torch.cuda.synchronize()
    r_gy, r_gw = oracle.combine_backward(g, y, rows, wt, n)
    got_gy = gy.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got_gy[:n], r_gy)         # pad rows are zero in both
    assert (got_gy[n:] == SENT16).all()
    got_gw = gw.cpu().numpy().astype(np.float64)
    assert (np.abs(got_gw - r_gw) <= _grad_w_bound(g, y, rows, H)).all()
    assert (got_gw[rows < 0] == 0).all()
    # repeated call: same bits
    gw2 = torch.empty_like(gw)
    ep.ep_combine_backward(h, _dev(g.view(np.int16)), y=_dev(y.view(np.int16)) if n else None,
                           topk_weights=_dev(wt) if wt is not None else None, grad_topk_weights=gw2, y_rows=n)
    torch.cuda.synchronize()
    assert torch.equal(gw, gw2)
    # dispatch backward: grad_x = unweighted combine, weight gradients gathered
    grw = np.random.default_rng(23).standard_normal(max(n, 1)).astype(np.float32)[:n]
    gx = torch.full((T, H), SENT16, dtype=torch.int16, device="cuda")
    gtw = torch.full((T, K), -9.0, dtype=torch.float32, device="cuda")
    ep.ep_dispatch_backward(h, _dev(y.view(np.int16)) if n else torch.empty((1, H), dtype=torch.int16, device="cuda"),
                            gx, grad_recv_weights=_dev(grw) if n else torch.empty(1, device="cuda"),
                            grad_topk_weights=gtw, grad_rows=n)
    torch.cuda.synchronize()
    r_gx, r_gtw = oracle.dispatch_backward(y, grw if n else np.zeros(1, np.float32), rows)
    assert_combine(gx.cpu().numpy().view(np.uint16), r_gx)
    np.testing.assert_array_equal(gtw.cpu().numpy().view(np.uint32), r_gtw.view(np.uint32))
    h.destroy()


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("skewed", 3000), ("prefill", 1024)])
def test_backward_workloads(ep, name, T):
    backward_path(ep, gi.make(name, 4, T=T, with_y=False))


def test_backward_full_prefill(ep):
    backward_path(ep, gi.make("prefill", 0, with_y=False))


@pytest.mark.parametrize("A,weights", [(16, True), (1, False)])
def test_backward_aligned_and_unweighted(ep, A, weights):
    backward_path(ep, gi.make("skewed", 5, T=2000, with_y=False), A=A, weights=weights)


def test_backward_all_dropped(ep):
    backward_path(ep, gi.make(_workload(30, 128, 8, 2, 2, drop_p=1.0), 0, with_y=False))


def test_combine_backward_exact_arithmetic(ep):
    """Small-integer gradients and outputs make every product and partial sum
    exact in fp32, so the weight gradient must equal the exact dot product."""
    rng = np.random.default_rng(31)
    T, K, E, R, H = 96, 4, 16, 4, 1024
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    ref = oracle.layout(idx, E, R)
    n = int(ref["expert_offsets"][-1])
    y = gi.f32_to_bf16_bits(rng.integers(-3, 4, size=(n, H)).astype(np.float32))
    g = gi.f32_to_bf16_bits(rng.integers(-3, 4, size=(T, H)).astype(np.float32))
    run = Run(ep, idx, E, R)
    gw = torch.empty(T, K, dtype=torch.float32, device="cuda")
    ep.ep_combine_backward(run.h, _dev(g.view(np.int16)), y=_dev(y.view(np.int16)), grad_topk_weights=gw)
    torch.cuda.synchronize()
    _, r_gw = oracle.combine_backward(g, y, ref["row_of_slot"], None, n)
    np.testing.assert_array_equal(gw.cpu().numpy().astype(np.float64), r_gw)
    run.h.destroy()


# ------------------------------------------------------------------ fp8 variants

def _layout_dev(ep, inp, A=1):
    w = inp.w
    o = [torch.empty(w.E, dtype=torch.int32, device="cuda"), torch.empty(w.R, dtype=torch.int32, device="cuda"),
         torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda"), torch.empty(w.E + 1, dtype=torch.int32, device="cuda")]
    return ep.ep_layout_aligned(_dev(inp.topk_idx), w.E, w.R, A, *o)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_dispatch_divides_on_reciprocal_traps(ep, fmt):
    """Blocks built around (amax, x) pairs where x / scale and x * (1 / scale)
    give different fp8 codes (found with numpy's IEEE division and torch's fp8
    cast): the fp8 dispatch must give the code of the true quotient, as the
    oracle does. Random data almost never reaches these pairs."""
    from test_oracle_pins import _reciprocal_traps, _torch_e4m3_bits, _torch_e5m2_bits
    from oracle import brute
    if fmt == "e4m3":
        F, values, codes_of, dt = 448.0, brute.e4m3_values()[1], _torch_e4m3_bits, ep.EP_DTYPE_FP8_E4M3
    else:
        F, values, codes_of, dt = 57344.0, brute.e5m2_values()[1], _torch_e5m2_bits, ep.EP_DTYPE_FP8_E5M2
    traps = _reciprocal_traps(F, values, codes_of)
    assert len(traps) >= 3
    T, H = len(traps), 256                     # two blocks per row: the trap block and its mirror
    xf = np.zeros((T, H), np.float32)
    for t, (amax, x, _) in enumerate(traps):
        xf[t, 0], xf[t, 1] = amax, x
        xf[t, 128], xf[t, 200] = -amax, -x
    x_bits = gi.f32_to_bf16_bits(xf)
    idx = np.zeros((T, 1), np.int64)
    w = gi.Workload("traps", T=T, H=H, E=1, K=1, R=1)
    inp = gi.Inputs(w=w, seed=0, x=x_bits, topk_idx=idx, topk_weights=np.ones((T, 1), np.float32), y=None,
                    num_valid=T)
    h = _layout_dev(ep, inp)
    q = torch.full((T, H), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.zeros((T, H // 128), dtype=torch.float32, device="cuda")
    ep.ep_dispatch_ex(h, _dev(x_bits.view(np.int16), torch.bfloat16), q, T, out_dtype=dt, recv_scales=sc)
    torch.cuda.synchronize()
    rows = np.arange(T, dtype=np.int32)[:, None]
    if fmt == "e4m3":
        r_q, r_s, _, _ = oracle.dispatch_e4m3(x_bits, rows, T)
    else:
        r_q, r_s = oracle.dispatch_e5m2(x_bits, rows, T, 0)
    got = q.cpu().numpy()
    np.testing.assert_array_equal(got, r_q)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), r_s.view(np.uint32))
    assert [int(got[t, 1]) for t in range(T)] == [c for _, _, c in traps]
    h.destroy()


def fp8_variant(ep, inp, mode, col_major=False, A=1, fmt=1):
    w = inp.w
    ref = oracle.layout_aligned(inp.topk_idx, w.E, w.R, A)
    n = int(ref["expert_offsets"][-1])
    nb = w.H // 128
    ue = mode == ep.EP_SCALE_UE8M0
    h = _layout_dev(ep, inp, A)
    if fmt == ep.EP_DTYPE_FP8_E5M2:
        r_q, r_s = oracle.dispatch_e5m2(inp.x, ref["row_of_slot"], n, scale_mode=mode)
    elif mode == ep.EP_SCALE_FP32:
        r_q, r_s, _, _ = oracle.dispatch_e4m3(inp.x, ref["row_of_slot"], n)
    else:
        r_q, r_s = oracle.dispatch_e4m3_pow2(inp.x, ref["row_of_slot"], n, ue8m0=ue)
    if A > 1:
        oracle.fill_pad_rows(ref, r_q, scales=None if ue else r_s)
        if ue:   # byte scales of pad rows: 0
            for e in range(w.E):
                lo = ref["expert_offsets"][e] + ref["num_tokens_per_expert"][e]
                r_s[lo:ref["expert_offsets"][e + 1]] = 0
    ld = (n + 3) // 4 * 4 + 4
    sdt = torch.uint8 if ue else torch.float32
    sent = 0xEE if ue else -1.0
    q = torch.full((max(n, 1), w.H), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.full((nb * ld,) if col_major else (max(n, 1), nb), sent, dtype=sdt, device="cuda")
    ep.ep_dispatch_ex(h, _dev(inp.x.view(np.int16)), q, n, out_dtype=fmt, scale_mode=mode, recv_scales=sc,
                      scales_col_major=col_major, scales_ld=ld if col_major else 0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy()[:n], r_q)
    g = sc.cpu().numpy()
    if col_major:
        g = g.reshape(nb, ld)
        got = g[:, :n].T
        assert (g[:, n:] == sent).all(), "column-major scales written past N"
    else:
        got = g[:n]
    if ue:
        np.testing.assert_array_equal(got, r_s)
    else:
        np.testing.assert_array_equal(got.view(np.uint32), r_s.view(np.uint32))
    h.destroy()


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("fp8", 1001), ("skewed", 2000)])
@pytest.mark.parametrize("mode", [1, 2])
def test_fp8_pow2_and_ue8m0(ep, name, T, mode):
    fp8_variant(ep, gi.make(name, 7, T=T, with_y=False), mode)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_fp8_col_major_scales(ep, mode):
    fp8_variant(ep, gi.make("fp8", 8, T=600, with_y=False), mode, col_major=True)


@pytest.mark.parametrize("mode,col", [(0, True), (2, False), (1, True)])
def test_fp8_variants_aligned(ep, mode, col):
    fp8_variant(ep, gi.make("skewed", 9, T=1500, with_y=False), mode, col_major=col, A=32)


def test_fp8_pow2_special_blocks(ep):
    rng = np.random.default_rng(12)
    T, H = 40, 1024
    xf = (rng.standard_normal((T, H)) * 2).astype(np.float32)
    xf[0, :128] = 0.0
    xf[1, 128:256] = 1e-39
    xf[2, 256:384] = 2.0 ** -130
    xf[3, 384:512] = 3e38
    xf[4, :] = np.float32(2.0 ** -133)
    x = gi.f32_to_bf16_bits(xf)
    idx = np.argsort(rng.random((T, 16)), axis=1)[:, :3].astype(np.int64)
    inp = gi.Inputs(w=_workload(T, H, 16, 3, 4), seed=0, x=x, topk_idx=idx,
                    topk_weights=np.full((T, 3), 1 / 3, np.float32), y=None, num_valid=3 * T)
    for mode in (1, 2):
        fp8_variant(ep, inp, mode)


@pytest.mark.parametrize("ue", [False, True])
def test_fp8_input_passthrough(ep, ue):
    inp = gi.make("fp8", 10, T=700, with_y=False)
    w = inp.w
    nb = w.H // 128
    # fp8 tokens and their scales, made by the oracle's quantiser
    codes = np.zeros((w.T, w.H), np.uint8)
    scales = np.zeros((w.T, nb), np.uint8 if ue else np.float32)
    for t in range(w.T):
        codes[t], scales[t] = oracle.quant_row_e4m3_pow2(inp.x[t], ue8m0=ue)
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    n = int(ref["expert_offsets"][-1])
    h = _layout_dev(ep, inp)
    q = torch.full((n, w.H), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.full((n, nb), 0xEE if ue else -1.0, dtype=torch.uint8 if ue else torch.float32, device="cuda")
    src = torch.full((n,), -5, dtype=torch.int32, device="cuda")
    ep.ep_dispatch_ex(h, _dev(codes), q, n, in_dtype=ep.EP_DTYPE_FP8_E4M3,
                      scale_mode=ep.EP_SCALE_UE8M0 if ue else ep.EP_SCALE_FP32,
                      x_scales=_dev(scales), recv_scales=sc, recv_src_token=src, H=w.H)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy(), oracle.dispatch_rows(codes, ref["row_of_slot"], n))
    np.testing.assert_array_equal(sc.cpu().numpy(), oracle.dispatch_rows(scales, ref["row_of_slot"], n))
    _, r_src, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
    np.testing.assert_array_equal(src.cpu().numpy(), r_src)
    h.destroy()


# ------------------------------------------------------------------ e5m2

@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("fp8", 1001), ("skewed", 2000)])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_e5m2_quantise_permute(ep, name, T, mode):
    fp8_variant(ep, gi.make(name, 31, T=T, with_y=False), mode, fmt=ep.EP_DTYPE_FP8_E5M2)


def test_e5m2_full_size(ep):
    """The fp8 prefill workload (T=8192, H=7168, top-8 of 256) quantised to e5m2."""
    fp8_variant(ep, gi.make("fp8", 0, with_y=False), 0, fmt=ep.EP_DTYPE_FP8_E5M2)


@pytest.mark.parametrize("mode,col,A", [(0, True, 1), (2, True, 1), (1, False, 32), (0, True, 32)])
def test_e5m2_col_major_and_aligned(ep, mode, col, A):
    fp8_variant(ep, gi.make("skewed", 32, T=1500, with_y=False), mode, col_major=col, A=A,
                fmt=ep.EP_DTYPE_FP8_E5M2)


def test_e5m2_special_blocks(ep):
    rng = np.random.default_rng(33)
    T, H = 40, 1024
    xf = (rng.standard_normal((T, H)) * 2).astype(np.float32)
    xf[0, :128] = 0.0
    xf[1, 128:256] = 1e-39
    xf[2, 256:384] = 2.0 ** -130
    xf[3, 384:512] = 3e38
    xf[4, :] = np.float32(2.0 ** -133)
    xf[5, ::2] *= 1e4
    xf[6, 512:640] = -0.0
    x = gi.f32_to_bf16_bits(xf)
    idx = np.argsort(rng.random((T, 16)), axis=1)[:, :3].astype(np.int64)
    inp = gi.Inputs(w=_workload(T, H, 16, 3, 4), seed=0, x=x, topk_idx=idx,
                    topk_weights=np.full((T, 3), 1 / 3, np.float32), y=None, num_valid=3 * T)
    for mode in (0, 1, 2):
        fp8_variant(ep, inp, mode, fmt=ep.EP_DTYPE_FP8_E5M2)


@pytest.mark.parametrize("mode", [0, 1])
def test_e5m2_encoder_sweep_all_bf16(ep, mode):
    """Every finite bf16 pattern through the e5m2 quantiser under several block scales."""
    inp = _sweep_inputs([57344.0, 448.0, 1.0, 3.0, 1e-3, 7.5e7, 2.0 ** -120])
    fp8_variant(ep, inp, mode, fmt=ep.EP_DTYPE_FP8_E5M2)


@pytest.mark.parametrize("ue", [False, True])
def test_e5m2_input_passthrough(ep, ue):
    inp = gi.make("fp8", 34, T=500, with_y=False)
    w = inp.w
    nb = w.H // 128
    codes = np.zeros((w.T, w.H), np.uint8)
    scales = np.zeros((w.T, nb), np.uint8 if ue else np.float32)
    for t in range(w.T):
        codes[t], scales[t] = oracle.quant_row_e5m2(inp.x[t], 2 if ue else 0)
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    n = int(ref["expert_offsets"][-1])
    h = _layout_dev(ep, inp)
    q = torch.full((n, w.H), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.full((n, nb), 0xEE if ue else -1.0, dtype=torch.uint8 if ue else torch.float32, device="cuda")
    ep.ep_dispatch_ex(h, _dev(codes), q, n, in_dtype=ep.EP_DTYPE_FP8_E5M2, out_dtype=ep.EP_DTYPE_FP8_E5M2,
                      scale_mode=ep.EP_SCALE_UE8M0 if ue else ep.EP_SCALE_FP32,
                      x_scales=_dev(scales), recv_scales=sc, H=w.H)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q.cpu().numpy(), oracle.dispatch_rows(codes, ref["row_of_slot"], n))
    np.testing.assert_array_equal(sc.cpu().numpy(), oracle.dispatch_rows(scales, ref["row_of_slot"], n))
    h.destroy()


@pytest.mark.parametrize("in_dt,out_dt", [(1, 2), (2, 1), (2, 0), (1, 0), (0, 3), (3, 3)])
def test_dispatch_ex_rejects_fp8_type_mismatch(ep, in_dt, out_dt):
    """fp8 input is moved unchanged, so in and out types must agree; unknown
    types are rejected; nothing is written."""
    inp = gi.make("tiny", 35, with_y=False)
    w = inp.w
    h = _layout_dev(ep, inp)
    n = w.T * w.K
    # sized for the requested output type, so the call reaches the library
    q = torch.full((n, w.H * (2 if out_dt == ep.EP_DTYPE_BF16 else 1)), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.zeros((n, w.H // 128), dtype=torch.float32, device="cuda")
    xs = torch.ones((w.T, w.H // 128), dtype=torch.float32, device="cuda")
    x = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch_ex(h, x, q, n, in_dtype=in_dt, out_dtype=out_dt, x_scales=xs, recv_scales=sc, H=w.H)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (q == SENT8).all()
    h.destroy()


# ------------------------------------------------------------------ dense routing maps

@pytest.mark.parametrize("name,T", [("tiny", None), ("skewed", 3000), ("prefill", 2048)])
def test_routing_map_conversions(ep, name, T):
    inp = gi.make(name, 13, T=T, with_y=False)
    w = inp.w
    r_map, r_probs, st = oracle.topk_to_routing_map(inp.topk_idx, inp.topk_weights, w.E)
    rm = torch.full((w.T, w.E), SENT8, dtype=torch.uint8, device="cuda")
    pr = torch.full((w.T, w.E), -1.0, dtype=torch.float32, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ep.ep_topk_to_routing_map(_dev(inp.topk_idx), w.E, rm, topk_weights=_dev(inp.topk_weights), probs=pr,
                              device_error=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(rm.cpu().numpy(), r_map)
    np.testing.assert_array_equal(pr.cpu().numpy().view(np.uint32), r_probs.view(np.uint32))
    assert err.item() == 0
    r_idx, r_w, _ = oracle.routing_map_to_topk(r_map, r_probs, w.K)
    idx = torch.full((w.T, w.K), -9, dtype=torch.int64, device="cuda")
    wt = torch.full((w.T, w.K), -1.0, dtype=torch.float32, device="cuda")
    ep.ep_routing_map_to_topk(rm, w.K, idx, probs=pr, topk_weights=wt, device_error=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), r_idx)
    np.testing.assert_array_equal(wt.cpu().numpy().view(np.uint32), r_w.view(np.uint32))
    assert err.item() == 0
    # the converted routing runs the whole path like any other
    inp2 = gi.Inputs(w=w, seed=0, x=inp.x, topk_idx=r_idx, topk_weights=r_w,
                     y=gi.normal_bf16(np.random.SeedSequence(14), int((r_idx >= 0).sum()), w.H)
                     if w.y != "identity" else None, num_valid=int((r_idx >= 0).sum()))
    full_path(ep, inp2, fp8=(w.H % 128 == 0))


@pytest.mark.parametrize("E,K,T,offset", [
    (12, 3, 700, 0),       # E % 8 != 0: scalar kernels
    (256, 8, 1000, 1),     # map and probs at odd offsets: scalar kernels
    (4096, 32, 300, 0),    # 16 blocks of 256 experts per token
    (40, 6, 999, 0),       # a partial block
    (64, 4, 513, 0),
])
def test_routing_map_vector_and_scalar_forms(ep, E, K, T, offset):
    """Both conversion directions against the oracle: random top-k with
    duplicate experts and dropped slots; random dense maps with any non-zero
    byte meaning routed, some rows holding more than K experts."""
    rng = np.random.default_rng(E * 100 + K)
    idx = rng.integers(-1, E, (T, K)).astype(np.int64)
    wts = rng.random((T, K)).astype(np.float32)
    r_map, r_probs, _ = oracle.topk_to_routing_map(idx, wts, E)
    mbuf = torch.full((T * E + 64,), SENT8, dtype=torch.uint8, device="cuda")
    pbuf = torch.full((T * E + 16,), -1.0, dtype=torch.float32, device="cuda")
    rm = mbuf[offset:offset + T * E].view(T, E)
    pr = pbuf[offset:offset + T * E].view(T, E)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ep.ep_topk_to_routing_map(_dev(idx), E, rm, topk_weights=_dev(wts), probs=pr, device_error=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(rm.cpu().numpy(), r_map)
    np.testing.assert_array_equal(pr.cpu().numpy().view(np.uint32), r_probs.view(np.uint32))
    assert err.item() == 0
    assert (mbuf[:offset] == SENT8).all() and (mbuf[offset + T * E:] == SENT8).all()

    dense = (rng.random((T, E)) < min(1.0, 1.5 * K / E)) * rng.integers(1, 256, (T, E))
    dense = dense.astype(np.uint8)
    probs = rng.random((T, E)).astype(np.float32)
    r_idx, r_w, st = oracle.routing_map_to_topk(dense, probs, K)
    rm.copy_(torch.from_numpy(dense))
    pr.copy_(torch.from_numpy(probs))
    out_i = torch.full((T, K), -9, dtype=torch.int64, device="cuda")
    out_w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    ep.ep_routing_map_to_topk(rm, K, out_i, probs=pr, topk_weights=out_w, device_error=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_i.cpu().numpy(), r_idx)
    np.testing.assert_array_equal(out_w.cpu().numpy().view(np.uint32), r_w.view(np.uint32))
    over = ((dense != 0).sum(axis=1) > K).any()
    assert err.item() == (ep.EP_ERR_CAPACITY if over else 0)
    assert (st != oracle.OK) == over          # the oracle flags the same inputs


@pytest.mark.parametrize("E", [64, 700])       # vector and scalar kernel forms
def test_routing_map_to_topk_without_probs_gives_unit_weights(ep, E):
    """A map given without probabilities converts to its experts with unit
    weights and 0 in the unused slots, as the oracle does."""
    rng = np.random.default_rng(E)
    T, K = 300, 6
    dense = ((rng.random((T, E)) < 3.0 / E) * rng.integers(1, 256, (T, E))).astype(np.uint8)
    dense[(dense != 0).sum(axis=1) > K] = 0            # keep every row within K experts
    r_idx, r_w, st = oracle.routing_map_to_topk(dense, None, K)
    assert st == oracle.OK
    out_i = torch.full((T, K), -9, dtype=torch.int64, device="cuda")
    out_w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    ep.ep_routing_map_to_topk(_dev(dense), K, out_i, topk_weights=out_w)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_i.cpu().numpy(), r_idx)
    np.testing.assert_array_equal(out_w.cpu().numpy().view(np.uint32), r_w.view(np.uint32))
    assert set(np.unique(r_w).tolist()) <= {0.0, 1.0}


def test_routing_map_errors(ep):
    idx = torch.tensor([[0, 9], [1, -3]], dtype=torch.int64, device="cuda")
    rm = torch.empty((2, 8), dtype=torch.uint8, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ep.ep_topk_to_routing_map(idx, 8, rm, device_error=err)
    torch.cuda.synchronize()
    assert err.item() == ep.EP_ERR_INVALID_EXPERT
    assert rm.cpu().numpy().tolist() == [[1, 0, 0, 0, 0, 0, 0, 0], [0, 1, 0, 0, 0, 0, 0, 0]]
    full = torch.ones((3, 40), dtype=torch.uint8, device="cuda")
    out = torch.empty((3, 4), dtype=torch.int64, device="cuda")
    ep.ep_routing_map_to_topk(full, 4, out, device_error=err)
    torch.cuda.synchronize()
    assert err.item() == ep.EP_ERR_CAPACITY
    assert out.cpu().numpy().tolist() == [[0, 1, 2, 3]] * 3


# ------------------------------------------------------------------ strided (padded 3-D) layout

def strided_path(ep, inp, cap):
    w = inp.w
    T, K, E, R, H = w.T, w.K, w.E, w.R, w.H
    ref = oracle.layout_strided(inp.topk_idx, E, R, cap)
    rows_total = E * cap
    o = [torch.full((E,), -7, dtype=torch.int32, device="cuda"), torch.full((R,), -7, dtype=torch.int32, device="cuda"),
         torch.full((T, R), SENT8, dtype=torch.uint8, device="cuda"),
         torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")]
    h = ep.ep_layout_strided(_dev(inp.topk_idx), E, R, cap, *o)
    rows = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    ep.ep_handle_copy_row_of_slot(h, rows)
    torch.cuda.synchronize()
    for got, key in zip(o, ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "expert_offsets"]):
        np.testing.assert_array_equal(got.cpu().numpy(), ref[key], err_msg=key)
    np.testing.assert_array_equal(rows.cpu().numpy(), ref["row_of_slot"])
    n, err = ep.ep_handle_query(h)
    assert n == rows_total
    assert err == (ep.EP_ERR_CAPACITY if ref["status"] == oracle.ERR_CAPACITY else 0)
    # dispatch into [E, cap, H]: valid rows get their token, the rest keep the sentinel
    recv = torch.full((rows_total, H), SENT16, dtype=torch.int16, device="cuda")
    ep.ep_dispatch(h, _dev(inp.x.view(np.int16)), ep.EP_DTYPE_BF16, recv, rows_total)
    torch.cuda.synchronize()
    want = np.full((rows_total, H), SENT16, np.uint16)
    r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], rows_total)
    used = np.zeros(rows_total, bool)
    used[ref["row_of_slot"][ref["row_of_slot"] >= 0]] = True
    want[used] = r_x[used]
    np.testing.assert_array_equal(recv.cpu().numpy().view(np.uint16), want)
    # combine over [E, cap, H] expert outputs skips dropped slots like the oracle
    y = gi.normal_bf16(np.random.SeedSequence(cap), rows_total, H)
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    ep.ep_combine(h, _dev(y.view(np.int16)), out, topk_weights=_dev(inp.topk_weights))
    torch.cuda.synchronize()
    assert_combine(out.cpu().numpy().view(np.uint16), oracle.combine(y, ref["row_of_slot"], inp.topk_weights))
    # a buffer smaller than E * cap rows is refused
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch(h, _dev(inp.x.view(np.int16)), ep.EP_DTYPE_BF16, recv, rows_total - 1)
    assert e.value.status == ep.EP_ERR_CAPACITY
    h.destroy()


def test_strided_decode(ep):
    strided_path(ep, gi.make("decode", 3, with_y=False), 32)


def test_strided_overflow_drops_slots(ep):
    strided_path(ep, gi.make("skewed", 3, T=2000, with_y=False), 100)


def test_strided_multiblock_path(ep):
    w = _workload(40000, 64, 64, 8, 4, routing="zipf", drop_p=0.05)
    strided_path(ep, gi.make(w, 4, with_y=False), 9000)


def test_strided_tiny_capacity(ep):
    strided_path(ep, gi.make("tiny", 4, with_y=False), 1)


# ------------------------------------------------------------------ non-expand layout

def nonexpand_path(ep, inp):
    w = inp.w
    T, K, E, R, H = w.T, w.K, w.E, w.R, w.H
    ref = oracle.layout_nonexpand(inp.topk_idx, E, R)
    n = int(ref["rank_offsets"][-1])
    o = [torch.full((E,), -7, dtype=torch.int32, device="cuda"), torch.full((R,), -7, dtype=torch.int32, device="cuda"),
         torch.full((T, R), SENT8, dtype=torch.uint8, device="cuda"),
         torch.full((R + 1,), -7, dtype=torch.int32, device="cuda")]
    h = ep.ep_layout_nonexpand(_dev(inp.topk_idx), E, R, *o)
    rows = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    ep.ep_handle_copy_row_of_slot(h, rows)
    torch.cuda.synchronize()
    for got, key in zip(o, ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "rank_offsets"]):
        np.testing.assert_array_equal(got.cpu().numpy(), ref[key], err_msg=key)
    np.testing.assert_array_equal(rows.cpu().numpy(), ref["row_of_slot"])
    assert ep.ep_handle_query(h) == (n, 0)
    # dispatch: one copy per (token, rank)
    r_x, r_src, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
    recv = torch.full((n + GUARD, H), SENT16, dtype=torch.int16, device="cuda")
    src = torch.full((n + GUARD,), -5, dtype=torch.int32, device="cuda")
    ep.ep_dispatch(h, _dev(inp.x.view(np.int16)), ep.EP_DTYPE_BF16, recv, n + GUARD, recv_src_token=src)
    torch.cuda.synchronize()
    g = recv.cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(g[:n], r_x)
    assert (g[n:] == SENT16).all()
    np.testing.assert_array_equal(src.cpu().numpy()[:n], r_src)
    # receive-side top-k per row
    ri = torch.full((n + 1, K), -9, dtype=torch.int64, device="cuda")
    rw = torch.full((n + 1, K), -1.0, dtype=torch.float32, device="cuda")
    ep.ep_nonexpand_recv_topk(h, _dev(inp.topk_idx), E, ri, recv_topk_weights=rw,
                              topk_weights=_dev(inp.topk_weights), recv_capacity=n + 1)
    torch.cuda.synchronize()
    r_ri, r_rw = oracle.nonexpand_recv_topk(inp.topk_idx, inp.topk_weights, ref["row_of_slot"], E, R, n)
    np.testing.assert_array_equal(ri.cpu().numpy()[:n], r_ri)
    np.testing.assert_array_equal(rw.cpu().numpy()[:n].view(np.uint32), r_rw.view(np.uint32))
    assert (ri.cpu().numpy()[n:] == -9).all()
    # unweighted combine: one expert-side row per rank
    y = gi.normal_bf16(np.random.SeedSequence(41), n, H)
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    ep.ep_combine(h, _dev(y.view(np.int16)) if n else torch.empty((1, H), dtype=torch.int16, device="cuda"), out,
                  y_rows=n)
    torch.cuda.synchronize()
    assert_combine(out.cpu().numpy().view(np.uint16), oracle.combine(y, ref["row_of_slot"], None))
    h.destroy()


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("prefill", 2048), ("skewed", 3000)])
def test_nonexpand_workloads(ep, name, T):
    nonexpand_path(ep, gi.make(name, 15, T=T, with_y=False))


def test_nonexpand_recv_topk_refuses_other_handles_and_experts(ep):
    """The rank-local ids depend on E / R, so ep_nonexpand_recv_topk takes only
    a non-expand layout's handle and the E that layout was given; anything
    else is refused before a launch and leaves the outputs untouched."""
    rng = np.random.default_rng(12)
    T, K, E, R = 50, 4, 16, 4
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
    o = [torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(R, dtype=torch.int32, device="cuda"),
         torch.empty((T, R), dtype=torch.uint8, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda")]
    ri = torch.full((T * K, K), -9, dtype=torch.int64, device="cuda")
    h = ep.ep_layout(_dev(idx), E, R, *o)                 # an expand layout
    with pytest.raises(ep.EPError) as e:
        ep.ep_nonexpand_recv_topk(h, _dev(idx), E, ri, recv_capacity=T * K)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
    ep.ep_layout_nonexpand(_dev(idx), E, R, o[0], o[1], o[2], o[3][:R + 1], handle=h)
    for bad_E in (2 * E, E // 2, R):                      # all divisible by R: only the layout's E is right
        with pytest.raises(ep.EPError) as e:
            ep.ep_nonexpand_recv_topk(h, _dev(idx), bad_E, ri, recv_capacity=T * K)
        assert e.value.status == ep.EP_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (ri.cpu().numpy() == -9).all()
    ep.ep_nonexpand_recv_topk(h, _dev(idx), E, ri, recv_capacity=T * K)
    ref = oracle.layout_nonexpand(idx, E, R)
    n = int(ref["rank_offsets"][-1])
    r_ri, _ = oracle.nonexpand_recv_topk(idx, None, ref["row_of_slot"], E, R, n)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ri.cpu().numpy()[:n], r_ri)
    # a later expand layout on the same handle is refused again
    ep.ep_layout(_dev(idx), E, R, *o, handle=h)
    with pytest.raises(ep.EPError) as e:
        ep.ep_nonexpand_recv_topk(h, _dev(idx), E, ri, recv_capacity=T * K)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
    h.destroy()


@pytest.mark.parametrize("w", [
    _workload(300, 128, 512, 8, 64),                                  # R > 32
    _workload(40000, 64, 64, 8, 4, routing="zipf", drop_p=0.05),      # multi-block layout path
    _workload(50, 128, 8, 2, 2, drop_p=1.0),                          # nothing routed
])
def test_nonexpand_edges(ep, w):
    nonexpand_path(ep, gi.make(w, 16, with_y=False))


def test_nonexpand_duplicate_experts_and_invalid_ids(ep):
    rng = np.random.default_rng(17)
    idx = rng.integers(0, 12, size=(200, 4)).astype(np.int64)
    idx[rng.random((200, 4)) < 0.1] = -1
    inp = gi.Inputs(w=_workload(200, 128, 12, 4, 3), seed=0, x=gi.normal_bf16(np.random.SeedSequence(18), 200, 128),
                    topk_idx=idx, topk_weights=rng.random((200, 4)).astype(np.float32), y=None, num_valid=0)
    nonexpand_path(ep, inp)
    bad = idx.copy()
    bad[7, 2] = 99
    ref = oracle.layout_nonexpand(bad, 12, 3)
    o = [torch.empty(12, dtype=torch.int32, device="cuda"), torch.empty(3, dtype=torch.int32, device="cuda"),
         torch.empty(200, 3, dtype=torch.uint8, device="cuda"), torch.empty(4, dtype=torch.int32, device="cuda")]
    h = ep.ep_layout_nonexpand(_dev(bad), 12, 3, *o)
    assert ep.ep_handle_query(h)[1] == ep.EP_ERR_INVALID_EXPERT
    np.testing.assert_array_equal(o[3].cpu().numpy(), ref["rank_offsets"])
    h.destroy()


@pytest.mark.parametrize("name,fp8", [("prefill", False), ("fp8", True), ("decode", False)])
def test_dispatch_overlapping_the_layout(ep, name, fp8):
    """Dispatch launched as the layout's programmatic dependent gives the same bytes."""
    inp = gi.make(name, 19, with_y=False)
    w = inp.w
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    n = int(ref["expert_offsets"][-1])
    idx, x = _dev(inp.topk_idx), _dev(inp.x.view(np.int16))
    o = [torch.empty(w.E, dtype=torch.int32, device="cuda"), torch.empty(w.R, dtype=torch.int32, device="cuda"),
         torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda"), torch.empty(w.E + 1, dtype=torch.int32, device="cuda")]
    h = ep.ep_layout(idx, w.E, w.R, *o)
    recv = torch.full((n, w.H), SENT8 if fp8 else SENT16, dtype=torch.uint8 if fp8 else torch.int16, device="cuda")
    sc = torch.full((n, w.H // 128), -1.0, dtype=torch.float32, device="cuda") if fp8 else None
    for _ in range(3):   # repeated layout -> dispatch pairs on one stream
        ep.ep_layout(idx, w.E, w.R, *o, handle=h)
        ep.ep_dispatch_ex(h, x, recv, n, out_dtype=ep.EP_DTYPE_FP8_E4M3 if fp8 else ep.EP_DTYPE_BF16,
                          recv_scales=sc, overlap_layout=True)
    torch.cuda.synchronize()
    if fp8:
        r_q, r_s, _, _ = oracle.dispatch_e4m3(inp.x, ref["row_of_slot"], n)
        np.testing.assert_array_equal(recv.cpu().numpy(), r_q)
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), r_s.view(np.uint32))
    else:
        r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
        np.testing.assert_array_equal(recv.cpu().numpy().view(np.uint16), r_x)
    h.destroy()


def test_fp8_quotients_near_e4m3_midpoints(ep):
    """Inputs whose x / scale lands within a few fp32 ulps of an e4m3 rounding
    midpoint (where a reciprocal-multiply could round differently from the
    IEEE quotient) still give the oracle's bytes."""
    rng = np.random.default_rng(23)
    xs_all = gi.bf16_bits_to_f32(np.arange(0x3c00, 0x7f00, dtype=np.uint16))   # positive normals
    blocks = []
    for amax_bits in rng.integers(0x3f80, 0x4700, 400).astype(np.uint16):
        amax = gi.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0]
        s = np.float32(amax) / np.float32(448.0)
        xs = xs_all[xs_all <= amax]
        q = (xs / s).astype(np.float32)
        m = (q.view(np.uint32) & 0xFFFFF).astype(np.int64) - 0x80000
        pick = xs[(np.abs(m) <= 8) & (q >= 2.0 ** -6)]
        for i in range(0, len(pick), 127):
            chunk = pick[i:i + 127]
            sign = np.where(rng.random(len(chunk)) < 0.5, -1.0, 1.0).astype(np.float32)
            blk = np.zeros(128, np.float32)
            blk[:len(chunk)] = chunk * sign
            blk[127] = amax
            blocks.append(blk)
    assert len(blocks) >= 8, "the search should find near-midpoint quotients"
    nb = (len(blocks) + 7) // 8 * 8
    allb = np.zeros((nb, 128), np.float32)
    allb[:len(blocks)] = np.stack(blocks)
    H = 1024
    x = gi.f32_to_bf16_bits(allb.reshape(nb // 8, H))
    T = x.shape[0]
    inp = gi.Inputs(w=_workload(T, H, 1, 1, 1), seed=0, x=x, topk_idx=np.zeros((T, 1), np.int64),
                    topk_weights=np.ones((T, 1), np.float32), y=None, num_valid=T)
    full_path(ep, inp, fp8=True)


# ------------------------------------------------------------------ CUDA graphs

@pytest.mark.parametrize("name,fp8", [("decode", False), ("skewed", False), ("tiny", True)])
def test_graph_capture_replays_the_step(ep, name, fp8):
    """layout -> dispatch (overlapped) -> combine captured once into a CUDA
    graph (handle reused, buffers of T*K rows: no allocation, no host wait)
    and replayed for new routings written into the same input buffers."""
    inp = gi.make(name, 50, T=600 if name == "skewed" else None)
    w = inp.w
    cap = w.T * w.K
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        idx = _dev(inp.topk_idx)
        x = _dev(inp.x.view(np.int16), torch.bfloat16)
        wt = _dev(inp.topk_weights)
        y = torch.zeros(cap, w.H, dtype=torch.bfloat16, device="cuda")
        o = [torch.empty(w.E, dtype=torch.int32, device="cuda"), torch.empty(w.R, dtype=torch.int32, device="cuda"),
             torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda"),
             torch.empty(w.E + 1, dtype=torch.int32, device="cuda")]
        recv = torch.empty(cap, w.H, dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
        sc = torch.empty(cap, w.H // 128, dtype=torch.float32, device="cuda") if fp8 else None
        out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
        h = ep.ep_layout(idx, w.E, w.R, *o)          # creates the handle (allocates) before capture
    s.synchronize()

    def step():
        ep.ep_layout(idx, w.E, w.R, *o, handle=h)
        ep.ep_dispatch_ex(h, x, recv, cap, out_dtype=ep.EP_DTYPE_FP8_E4M3 if fp8 else ep.EP_DTYPE_BF16,
                          recv_scales=sc, overlap_layout=True)
        ep.ep_combine(h, y, out, topk_weights=wt)

    with torch.cuda.stream(s):
        step()                                        # warm-up outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    rng = np.random.default_rng(51)
    for rep in range(3):
        # new routing and weights in the captured buffers, and expert outputs
        # for the rows this routing produces
        idx_n = np.argsort(rng.random((w.T, w.E)), axis=1)[:, :w.K].astype(np.int64)
        idx_n[rng.random((w.T, w.K)) < 0.1 * rep] = -1
        wt_n = rng.random((w.T, w.K)).astype(np.float32)
        ref = oracle.layout(idx_n, w.E, w.R)
        n = int(ref["expert_offsets"][-1])
        y_n = gi.normal_bf16(np.random.SeedSequence(52 + rep), n, w.H)
        with torch.cuda.stream(s):
            idx.copy_(torch.from_numpy(idx_n))
            wt.copy_(torch.from_numpy(wt_n))
            y[:n].copy_(torch.from_numpy(y_n.view(np.int16)).view(torch.bfloat16))
            g.replay()                                # on s, after the copies into the captured buffers
        s.synchronize()
        np.testing.assert_array_equal(o[3].cpu().numpy(), ref["expert_offsets"])
        np.testing.assert_array_equal(o[2].cpu().numpy(), ref["is_token_in_rank"])
        np.testing.assert_array_equal(o[1].cpu().numpy(), ref["num_tokens_per_rank"])
        if fp8:
            r_q, r_s, _, _ = oracle.dispatch_e4m3(inp.x, ref["row_of_slot"], n)
            np.testing.assert_array_equal(recv[:n].cpu().numpy(), r_q)
            np.testing.assert_array_equal(sc[:n].cpu().numpy().view(np.uint32), r_s.view(np.uint32))
        else:
            r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
            np.testing.assert_array_equal(_u16(recv[:n]), r_x)
        np.testing.assert_array_equal(_u16(out), oracle.combine(y_n, ref["row_of_slot"], wt_n))
        assert ep.ep_handle_query(h)[0] == n
    del g
    h.destroy()


_FIRST_CALLS_IN_CAPTURE = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import combine_get_dispatch_layout_gb300 as ep
import oracle
from gen import inputs as gi

inp = gi.make("decode", 61)
w = inp.w
cap = w.T * w.K
s = torch.cuda.Stream()
with torch.cuda.stream(s):
    idx = torch.from_numpy(inp.topk_idx).cuda()
    x = torch.from_numpy(inp.x.view(np.int16)).cuda().view(torch.bfloat16)
    wt = torch.from_numpy(inp.topk_weights).cuda()
    y = torch.from_numpy(inp.y.view(np.int16)).cuda().view(torch.bfloat16)
    o = [torch.empty(w.E, dtype=torch.int32, device="cuda"), torch.empty(w.R, dtype=torch.int32, device="cuda"),
         torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda"), torch.empty(w.E + 1, dtype=torch.int32, device="cuda")]
    recv = torch.empty(cap, w.H, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    h = ep.ep_layout(idx, w.E, w.R, *o)
s.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):      # this process's first dispatch and combine
    ep.ep_layout(idx, w.E, w.R, *o, handle=h)
    ep.ep_dispatch_ex(h, x, recv, cap, out_dtype=ep.EP_DTYPE_BF16, overlap_layout=True)
    ep.ep_combine(h, y, out, topk_weights=wt)
with torch.cuda.stream(s):
    g.replay()
s.synchronize()
ref = oracle.layout(inp.topk_idx, w.E, w.R)
n = int(ref["expert_offsets"][-1])
r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
assert np.array_equal(recv[:n].view(torch.int16).cpu().numpy().view(np.uint16), r_x)
assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16),
                      oracle.combine(inp.y, ref["row_of_slot"], inp.topk_weights))
h.destroy()
print("ok")
"""


def test_first_dispatch_of_a_process_inside_a_capture(ep, tmp_path):
    """The library's one-time launch queries must not fall inside a user's
    stream capture: in a fresh process, with only the handle-creating layout
    run eagerly, the first dispatch and combine are captured into a graph,
    replayed, and checked against the oracle."""
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "first_calls.py"
    script.write_text(_FIRST_CALLS_IN_CAPTURE)
    r = subprocess.run([sys.executable, str(script), root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


def test_graph_capture_of_the_whole_chain(ep):
    """Conversions, layout, a plain dispatch (which waits at entry), combine
    and both backward passes captured into one CUDA graph, every kernel a
    programmatic dependent of the one before, then replayed on new inputs
    written into the captured buffers; each output against the oracle."""
    inp = gi.make("decode", 56, with_y=False)
    w = inp.w
    T, K, E, R, H = w.T, w.K, w.E, w.R, w.H
    cap = T * K
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        idx = _dev(inp.topk_idx)
        wt = _dev(inp.topk_weights)
        rm = torch.empty(T, E, dtype=torch.uint8, device="cuda")
        pr = torch.empty(T, E, dtype=torch.float32, device="cuda")
        idx2 = torch.empty(T, K, dtype=torch.int64, device="cuda")
        wt2 = torch.empty(T, K, dtype=torch.float32, device="cuda")
        o = [torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(R, dtype=torch.int32, device="cuda"),
             torch.empty(T, R, dtype=torch.uint8, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda")]
        x = torch.empty(T, H, dtype=torch.int16, device="cuda")
        y = torch.zeros(cap, H, dtype=torch.int16, device="cuda")
        g = torch.empty(T, H, dtype=torch.int16, device="cuda")
        grw = torch.zeros(cap, dtype=torch.float32, device="cuda")
        recv = torch.empty(cap, H, dtype=torch.int16, device="cuda")
        out = torch.empty(T, H, dtype=torch.int16, device="cuda")
        gy = torch.empty(cap, H, dtype=torch.int16, device="cuda")
        gw = torch.empty(T, K, dtype=torch.float32, device="cuda")
        gx = torch.empty(T, H, dtype=torch.int16, device="cuda")
        gtw = torch.empty(T, K, dtype=torch.float32, device="cuda")
        ep.ep_topk_to_routing_map(idx, E, rm, topk_weights=wt, probs=pr)
        ep.ep_routing_map_to_topk(rm, K, idx2, probs=pr, topk_weights=wt2)
        h = ep.ep_layout(idx2, E, R, *o)                # creates the handle before the capture
    s.synchronize()

    def chain():
        ep.ep_topk_to_routing_map(idx, E, rm, topk_weights=wt, probs=pr)
        ep.ep_routing_map_to_topk(rm, K, idx2, probs=pr, topk_weights=wt2)
        ep.ep_layout(idx2, E, R, *o, handle=h)
        ep.ep_dispatch(h, x, ep.EP_DTYPE_BF16, recv, cap)
        ep.ep_combine(h, y, out, topk_weights=wt2)
        ep.ep_combine_backward(h, g, y=y, topk_weights=wt2, grad_y=gy, grad_topk_weights=gw, y_rows=cap,
                               grad_y_capacity=cap)
        ep.ep_dispatch_backward(h, gy, gx, grad_recv_weights=grw, grad_topk_weights=gtw, grad_rows=cap)

    g_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_graph, stream=s):
        chain()
    rng = np.random.default_rng(57)
    for rep in range(2):
        idx_n = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
        idx_n[rng.random((T, K)) < 0.1] = -1
        wt_n = rng.random((T, K)).astype(np.float32)
        x_n = gi.normal_bf16(np.random.SeedSequence(58 + rep), T, H)
        g_n = gi.normal_bf16(np.random.SeedSequence(60 + rep), T, H)
        rm_r, pr_r, st = oracle.topk_to_routing_map(idx_n, wt_n, E)
        assert st == oracle.OK
        idx2_r, wt2_r, st = oracle.routing_map_to_topk(rm_r, pr_r, K)
        assert st == oracle.OK
        L = oracle.layout(idx2_r, E, R)
        rows, n = L["row_of_slot"], int(L["expert_offsets"][-1])
        y_n = gi.normal_bf16(np.random.SeedSequence(62 + rep), n, H)
        grw_n = rng.standard_normal(n).astype(np.float32)
        with torch.cuda.stream(s):
            idx.copy_(torch.from_numpy(idx_n))
            wt.copy_(torch.from_numpy(wt_n))
            x.copy_(torch.from_numpy(x_n.view(np.int16)))
            g.copy_(torch.from_numpy(g_n.view(np.int16)))
            y[:n].copy_(torch.from_numpy(y_n.view(np.int16)))
            grw[:n].copy_(torch.from_numpy(grw_n))
            g_graph.replay()
        s.synchronize()
        np.testing.assert_array_equal(rm.cpu().numpy(), rm_r)
        np.testing.assert_array_equal(idx2.cpu().numpy(), idx2_r)
        np.testing.assert_array_equal(o[3].cpu().numpy(), L["expert_offsets"])
        r_x, _, _ = oracle.dispatch_bf16(x_n, rows, n)
        np.testing.assert_array_equal(_u16(recv[:n]), r_x)
        np.testing.assert_array_equal(_u16(out), oracle.combine(y_n, rows, wt2_r))
        r_gy, r_gw = oracle.combine_backward(g_n, y_n, rows, wt2_r, n)
        np.testing.assert_array_equal(_u16(gy[:n]), r_gy)
        got_gw = gw.cpu().numpy().astype(np.float64)
        assert (np.abs(got_gw - r_gw) <= _grad_w_bound(g_n, y_n, rows, H)).all()
        r_gx, r_gtw = oracle.dispatch_backward(r_gy, grw_n, rows)
        assert_combine(_u16(gx), r_gx)
        np.testing.assert_array_equal(gtw.cpu().numpy().view(np.uint32), r_gtw.view(np.uint32))
    del g_graph
    h.destroy()


def test_capture_refuses_host_waits_and_allocation(ep):
    """Inside a stream capture, calls that would allocate or wait for the
    device are refused with EP_ERR_INVALID_ARG and enqueue nothing; the rest
    of the capture is intact and replays correctly."""
    inp = gi.make("decode", 54)
    w = inp.w
    cap = w.T * w.K
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        idx = _dev(inp.topk_idx)
        x = _dev(inp.x.view(np.int16), torch.bfloat16)
        o = [torch.empty(w.E, dtype=torch.int32, device="cuda"), torch.empty(w.R, dtype=torch.int32, device="cuda"),
             torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda"),
             torch.empty(w.E + 1, dtype=torch.int32, device="cuda")]
        small = torch.empty(cap - 1, w.H, dtype=torch.bfloat16, device="cuda")
        full = torch.full((cap, w.H), -3.0, dtype=torch.bfloat16, device="cuda")
        h = ep.ep_layout(idx, w.E, w.R, *o)
    s.synchronize()
    statuses = []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ep.ep_layout(idx, w.E, w.R, *o, handle=h)
        for call in (lambda: ep.ep_dispatch(h, x, ep.EP_DTYPE_BF16, small, cap - 1),
                     lambda: ep.ep_layout(idx, w.E, w.R, *o),
                     lambda: ep.ep_handle_query(h)):
            try:
                call()
                statuses.append(ep.EP_OK)
            except ep.EPError as e:
                statuses.append(e.status)
        ep.ep_dispatch(h, x, ep.EP_DTYPE_BF16, full, cap)
    assert statuses == [ep.EP_ERR_INVALID_ARG] * 3
    with torch.cuda.stream(s):
        full.fill_(-3.0)
        g.replay()
    s.synchronize()
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    n = int(ref["expert_offsets"][-1])
    r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
    np.testing.assert_array_equal(_u16(full[:n]), r_x)
    assert ep.ep_handle_query(h)[0] == n
    del g
    h.destroy()


@pytest.mark.parametrize("kind", ["bf16", "e4m3", "e5m2", "passthrough"])
def test_overlapped_dispatch_ragged_shapes(ep, kind):
    """Overlapped dispatch (programmatic dependent of the layout, with the L2
    prefetch of x) on a ragged token count and a row that is not a whole
    number of work items: the prefetch window is clamped to x and every
    kernel variant gives the oracle's bytes."""
    H = 4104 if kind == "bf16" else 4224
    w = _workload(5001, H, 64, 6, 4, routing="zipf", drop_p=0.05)
    inp = gi.make(w, 55, with_y=False)
    ref = oracle.layout(inp.topk_idx, w.E, w.R)
    n = int(ref["expert_offsets"][-1])
    nb = H // 128
    h = _layout_dev(ep, inp)
    idx = _dev(inp.topk_idx)
    o = [torch.empty(w.E, dtype=torch.int32, device="cuda"), torch.empty(w.R, dtype=torch.int32, device="cuda"),
         torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda"), torch.empty(w.E + 1, dtype=torch.int32, device="cuda")]
    if kind == "passthrough":
        codes = np.zeros((w.T, H), np.uint8)
        scales = np.zeros((w.T, nb), np.float32)
        for t in range(w.T):
            codes[t], scales[t] = oracle.quant_row_e4m3(inp.x[t])
        x, xs = _dev(codes), _dev(scales)
    else:
        x, xs = _dev(inp.x.view(np.int16)), None
    bf16 = kind == "bf16"
    cap = w.T * w.K
    recv = torch.full((cap, H), SENT16 if bf16 else SENT8, dtype=torch.int16 if bf16 else torch.uint8,
                      device="cuda")
    sc = None if bf16 else torch.full((cap, nb), -1.0, dtype=torch.float32, device="cuda")
    fmt = {"bf16": ep.EP_DTYPE_BF16, "e4m3": ep.EP_DTYPE_FP8_E4M3, "e5m2": ep.EP_DTYPE_FP8_E5M2,
           "passthrough": ep.EP_DTYPE_FP8_E4M3}[kind]
    for _ in range(2):
        ep.ep_layout(idx, w.E, w.R, *o, handle=h)
        ep.ep_dispatch_ex(h, x, recv, cap, out_dtype=fmt,
                          in_dtype=ep.EP_DTYPE_FP8_E4M3 if kind == "passthrough" else ep.EP_DTYPE_BF16,
                          x_scales=xs, recv_scales=sc, H=H, overlap_layout=True)
    torch.cuda.synchronize()
    got = recv.cpu().numpy()
    if bf16:
        r_x, _, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
        np.testing.assert_array_equal(got[:n].view(np.uint16), r_x)
        assert (got[n:] == SENT16).all()
        h.destroy()
        return
    if kind == "passthrough":
        r_q = oracle.dispatch_rows(codes, ref["row_of_slot"], n)
        r_s = oracle.dispatch_rows(scales, ref["row_of_slot"], n)
    elif kind == "e5m2":
        r_q, r_s = oracle.dispatch_e5m2(inp.x, ref["row_of_slot"], n)
    else:
        r_q, r_s, _, _ = oracle.dispatch_e4m3(inp.x, ref["row_of_slot"], n)
    np.testing.assert_array_equal(got[:n], r_q)
    assert (got[n:] == SENT8).all()
    np.testing.assert_array_equal(sc.cpu().numpy()[:n].view(np.uint32), r_s.view(np.uint32))
    h.destroy()


def test_two_host_threads_with_their_own_handles(ep):
    """Handles used from two host threads at once (one handle per thread,
    one stream each), alternating shapes so the shared launch-state cache
    takes new entries while the other thread launches."""
    import threading
    cases = [gi.make("decode", 60 + i, with_y=False) for i in range(2)] + \
            [gi.make("skewed", 62 + i, T=3000, with_y=False) for i in range(2)]
    refs = [oracle.layout(c.topk_idx, c.w.E, c.w.R) for c in cases]
    errors = []

    def worker(order):
        try:
            s = torch.cuda.Stream()
            h = None
            for rep in range(6):
                for ci in order:
                    c, ref = cases[ci], refs[ci]
                    w = c.w
                    with torch.cuda.stream(s):
                        idx, x = _dev(c.topk_idx), _dev(c.x.view(np.int16), torch.bfloat16)
                        o = [torch.empty(w.E, dtype=torch.int32, device="cuda"),
                             torch.empty(w.R, dtype=torch.int32, device="cuda"),
                             torch.empty(w.T, w.R, dtype=torch.uint8, device="cuda"),
                             torch.empty(w.E + 1, dtype=torch.int32, device="cuda")]
                        recv = torch.empty(w.T * w.K, w.H, dtype=torch.bfloat16, device="cuda")
                        h = ep.ep_layout(idx, w.E, w.R, *o, handle=h, stream=s)
                        ep.ep_dispatch(h, x, ep.EP_DTYPE_BF16, recv, w.T * w.K, stream=s)
                    s.synchronize()
                    n = int(ref["expert_offsets"][-1])
                    if not np.array_equal(o[3].cpu().numpy(), ref["expert_offsets"]):
                        errors.append(("offsets", ci))
                    r_x, _, _ = oracle.dispatch_bf16(c.x, ref["row_of_slot"], n)
                    if not np.array_equal(_u16(recv[:n]), r_x):
                        errors.append(("rows", ci))
            h.destroy()
        except Exception as e:   # surfaced below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(o,)) for o in ([0, 2, 1, 3], [3, 1, 2, 0])]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert errors == []


# ------------------------------------------------------------------ randomised configurations

def _random_config(seed):
    """A seeded random shape inside the API's limits, with its options."""
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 64]))
    E = R * int(rng.integers(1, max(2, 512 // R) + 1))
    K = int(rng.integers(1, min(32, E) + 1))
    T = int(rng.choice([0, 1, 7, int(rng.integers(2, 3000))]))
    H = int(rng.choice([8, 136, 256, 1024, 1288, 2048, 3072]))
    w = _workload(T, H, E, K, R, routing=str(rng.choice(["uniform", "zipf"])),
                  drop_p=float(rng.choice([0.0, 0.05, 0.5])))
    opts = dict(A=int(rng.choice([1, 1, 2, 8, 64, 128])), mode=int(rng.integers(0, 3)),
                fmt=int(rng.choice([1, 2])), col=bool(rng.integers(0, 2)))
    return w, opts


@pytest.mark.parametrize("seed", range(40))
def test_random_configurations(ep, seed):
    """Random shapes, routings and options through layout, dispatch (bf16, and
    fp8 when H % 128 == 0) and combine, plus the aligned fp8 variant, all
    against the oracle."""
    w, o = _random_config(seed)
    inp = gi.make(w, 2000 + seed)
    fp8 = w.H % 128 == 0
    full_path(ep, inp, fp8=fp8, weights=bool(seed % 4))
    if fp8 and w.T > 0:
        fp8_variant(ep, inp, o["mode"], col_major=o["col"], A=o["A"], fmt=o["fmt"])


def _random_large_config(seed):
    """A seeded random shape toward the API's limits: E up to 4096, K up to 32,
    up to 2^20 slots (so about one in five takes the three-kernel layout
    path), H shrunk so the receive rows stay within 256 MB."""
    rng = np.random.default_rng(90000 + seed)
    R = int(rng.choice([1, 2, 4, 8, 16, 32, 64]))
    E = R * int(rng.integers(1, 4096 // R + 1))
    K = int(rng.integers(1, min(32, E) + 1))
    T = int(np.exp(rng.uniform(0, np.log(max(2, (1 << 20) // K)))))
    h_max = max(8, min(7168, (256 << 20) // max(1, 2 * T * K) // 8 * 8))
    H = int(rng.choice([h for h in [8, 64, 128, 264, 1024, 2048, 4096, 7168] if h <= h_max] or [8]))
    w = _workload(T, H, E, K, R, routing=str(rng.choice(["uniform", "zipf"])),
                  drop_p=float(rng.choice([0.0, 0.02, 0.3])))
    opts = dict(A=int(rng.choice([1, 8, 128])), mode=int(rng.integers(0, 3)), fmt=int(rng.choice([1, 2])),
                col=bool(rng.integers(0, 2)))
    return w, opts


@pytest.mark.parametrize("seed", range(12))
def test_random_large_configurations(ep, seed):
    """Random large shapes through layout, dispatch (bf16, and fp8 when
    H % 128 == 0), combine and an fp8 variant, against the oracle."""
    w, o = _random_large_config(seed)
    inp = gi.make(w, 3000 + seed)
    fp8 = w.H % 128 == 0
    full_path(ep, inp, fp8=fp8, weights=bool(seed % 3))
    if fp8 and w.T > 0:
        fp8_variant(ep, inp, o["mode"], col_major=o["col"], A=o["A"], fmt=o["fmt"])
    torch.cuda.empty_cache()


def test_empty_inputs_with_optional_outputs(ep):
    """Empty arrays arrive as null pointers: T = 0 with weights requested, and
    a dispatch backward whose receive side has no rows (every slot dropped),
    are valid calls that write what they must and nothing else."""
    # T = 0, recv_weights requested, weights tensor empty
    idx0 = np.zeros((0, 4), np.int64)
    run0 = Run(ep, idx0, 8, 2)
    recv = torch.full((GUARD, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    rw = torch.full((GUARD,), 5.0, dtype=torch.float32, device="cuda")
    ep.ep_dispatch(run0.h, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), ep.EP_DTYPE_BF16, recv, GUARD,
                   recv_weights=rw, topk_weights=torch.empty(0, 4, dtype=torch.float32, device="cuda"))
    rm = torch.empty(0, 8, dtype=torch.uint8, device="cuda")
    ep.ep_topk_to_routing_map(torch.empty(0, 4, dtype=torch.int64, device="cuda"), 8, rm,
                              topk_weights=torch.empty(0, 4, dtype=torch.float32, device="cuda"),
                              probs=torch.empty(0, 8, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert (recv == 3.0).all() and (rw == 5.0).all()
    run0.h.destroy()
    # T > 0, every slot dropped: no receive rows, weight gradients all 0
    T, K = 50, 3
    idx = np.full((T, K), -1, np.int64)
    run = Run(ep, idx, 8, 2)
    gx = torch.full((T, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    gtw = torch.full((T, K), 9.0, dtype=torch.float32, device="cuda")
    ep.ep_dispatch_backward(run.h, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), gx,
                            grad_recv_weights=torch.empty(0, dtype=torch.float32, device="cuda"),
                            grad_topk_weights=gtw)
    torch.cuda.synchronize()
    assert (gx == 0).all() and (gtw == 0).all()
    run.h.destroy()


@pytest.mark.parametrize("seed", range(30))
def test_random_configurations_other_paths(ep, seed):
    """Random shapes through the aligned, backward, strided (capacity drawn
    at random, sometimes too small) and non-expand paths against the oracle."""
    w, o = _random_config(100 + seed)
    inp = gi.make(w, 3000 + seed)
    rng = np.random.default_rng(4000 + seed)
    full_path_aligned(ep, inp, o["A"], fp8=(w.H % 128 == 0))
    backward_path(ep, inp, A=o["A"], weights=bool(seed % 3))
    strided_path(ep, inp, cap=int(rng.integers(1, max(2, w.T + 2))))
    nonexpand_path(ep, inp)


@pytest.mark.parametrize("seed", range(30))
def test_random_overlapped_dispatch(ep, seed):
    """Random shapes and alignments with the dispatch launched as the layout's
    programmatic dependent (x loaded and prefetched during the layout, pad rows
    zeroed by the dispatch grid): bf16, and fp8 in a random format and scale
    mode when H % 128 == 0, against the oracle, pad rows included."""
    w, o = _random_config(200 + seed)
    if w.T == 0:
        w = _workload(1 + 37 * seed, w.H, w.E, w.K, w.R, routing=w.routing, drop_p=w.drop_p)
    inp = gi.make(w, 5000 + seed, with_y=False)
    T, K, E, R, H, A = w.T, w.K, w.E, w.R, w.H, o["A"]
    ref = oracle.layout_aligned(inp.topk_idx, E, R, A)
    n = int(ref["expert_offsets"][-1])
    cap = T * K + E * (A - 1)
    idx, x = _dev(inp.topk_idx), _dev(inp.x.view(np.int16))
    h = _layout_dev(ep, inp, A)
    outs = [torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(R, dtype=torch.int32, device="cuda"),
            torch.empty(T, R, dtype=torch.uint8, device="cuda"), torch.empty(E + 1, dtype=torch.int32, device="cuda")]
    src = torch.full((cap,), -5, dtype=torch.int32, device="cuda")
    # bf16
    recv = torch.full((cap, H), SENT16, dtype=torch.int16, device="cuda")
    ep.ep_layout_aligned(idx, E, R, A, *outs, handle=h)
    ep.ep_dispatch_ex(h, x, recv, cap, out_dtype=ep.EP_DTYPE_BF16, recv_src_token=src, H=H, overlap_layout=True)
    torch.cuda.synchronize()
    r_x, r_src, _ = oracle.dispatch_bf16(inp.x, ref["row_of_slot"], n)
    r_src = r_src.copy()
    oracle.fill_pad_rows(ref, r_x, src=r_src)
    got = recv.cpu().numpy()
    np.testing.assert_array_equal(got[:n].view(np.uint16), r_x)
    assert (got[n:] == SENT16).all()
    np.testing.assert_array_equal(src.cpu().numpy()[:n], r_src)
    if H % 128 or n == 0:
        h.destroy()
        return
    # fp8, format / scale mode / scale layout drawn for this seed
    mode, fmt, col = o["mode"], o["fmt"], o["col"]
    ue = mode == ep.EP_SCALE_UE8M0
    nb = H // 128
    ld = cap + 4
    q = torch.full((cap, H), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.full((nb * ld,) if col else (cap, nb), 0xEE if ue else -1.0,
                    dtype=torch.uint8 if ue else torch.float32, device="cuda")
    ep.ep_layout_aligned(idx, E, R, A, *outs, handle=h)
    ep.ep_dispatch_ex(h, x, q, cap, out_dtype=fmt, scale_mode=mode, recv_scales=sc, scales_col_major=col,
                      scales_ld=ld if col else 0, H=H, overlap_layout=True)
    torch.cuda.synchronize()
    if fmt == ep.EP_DTYPE_FP8_E5M2:
        r_q, r_s = oracle.dispatch_e5m2(inp.x, ref["row_of_slot"], n, scale_mode=mode)
    elif mode == ep.EP_SCALE_FP32:
        r_q, r_s, _, _ = oracle.dispatch_e4m3(inp.x, ref["row_of_slot"], n)
    else:
        r_q, r_s = oracle.dispatch_e4m3_pow2(inp.x, ref["row_of_slot"], n, ue8m0=ue)
    oracle.fill_pad_rows(ref, r_q, scales=None if ue else r_s)
    if ue:
        for e in range(E):
            r_s[ref["expert_offsets"][e] + ref["num_tokens_per_expert"][e]:ref["expert_offsets"][e + 1]] = 0
    gq = q.cpu().numpy()
    np.testing.assert_array_equal(gq[:n], r_q)
    assert (gq[n:] == SENT8).all()
    g = sc.cpu().numpy()
    got_s = g.reshape(nb, ld)[:, :n].T if col else g[:n]
    if ue:
        np.testing.assert_array_equal(got_s, r_s)
    else:
        np.testing.assert_array_equal(got_s.view(np.uint32), r_s.view(np.uint32))
    h.destroy()


@pytest.mark.parametrize("seed", range(20))
def test_random_routing_map_conversions(ep, seed):
    """Both conversion directions on random T, E (any value, so both kernel
    forms), K, duplicate experts, dropped slots and buffer offsets."""
    rng = np.random.default_rng(6000 + seed)
    E = int(rng.choice([int(rng.integers(1, 64)), 8 * int(rng.integers(1, 65)), int(rng.integers(1, 4097))]))
    K = int(rng.integers(1, min(32, E) + 1))
    T = int(rng.choice([0, 1, int(rng.integers(2, 2000))]))
    off = int(rng.choice([0, 0, 1, 3]))
    idx = rng.integers(-1, E, (T, K)).astype(np.int64)
    wts = rng.random((T, K)).astype(np.float32)
    r_map, r_probs, _ = oracle.topk_to_routing_map(idx, wts, E)
    mbuf = torch.full((T * E + 16,), SENT8, dtype=torch.uint8, device="cuda")
    pbuf = torch.full((T * E + 8,), -1.0, dtype=torch.float32, device="cuda")
    rm, pr = mbuf[off:off + T * E].view(T, E), pbuf[off:off + T * E].view(T, E)
    ep.ep_topk_to_routing_map(_dev(idx), E, rm, topk_weights=_dev(wts), probs=pr)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(rm.cpu().numpy(), r_map)
    np.testing.assert_array_equal(pr.cpu().numpy().view(np.uint32), r_probs.view(np.uint32))
    assert (mbuf[:off] == SENT8).all() and (mbuf[off + T * E:] == SENT8).all()
    r_idx, r_w, _ = oracle.routing_map_to_topk(r_map, r_probs, K)
    out_i = torch.full((T, K), -9, dtype=torch.int64, device="cuda")
    out_w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    ep.ep_routing_map_to_topk(rm, K, out_i, probs=pr, topk_weights=out_w)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out_i.cpu().numpy(), r_idx)
    np.testing.assert_array_equal(out_w.cpu().numpy().view(np.uint32), r_w.view(np.uint32))


@pytest.mark.parametrize("seed", range(12))
def test_random_fp8_passthrough(ep, seed):
    """fp8 input pass-through on random shapes, formats, scale modes and
    layouts and alignments: codes and scale rows moved unchanged, pad rows
    zeroed."""
    rng = np.random.default_rng(7000 + seed)
    w, o = _random_config(300 + seed)
    H = 128 * int(rng.integers(1, 25))
    w = _workload(max(1, w.T), H, w.E, w.K, w.R, routing=w.routing, drop_p=w.drop_p)
    inp = gi.make(w, 8000 + seed, with_y=False)
    T, K, E, R, A = w.T, w.K, w.E, w.R, o["A"]
    fmt, ue, col = o["fmt"], bool(rng.integers(0, 2)), o["col"]
    nb = H // 128
    codes = rng.integers(0, 256, (T, H)).astype(np.uint8)
    scales = rng.integers(0, 256, (T, nb)).astype(np.uint8) if ue else rng.random((T, nb)).astype(np.float32)
    ref = oracle.layout_aligned(inp.topk_idx, E, R, A)
    n = int(ref["expert_offsets"][-1])
    cap = T * K + E * (A - 1)
    ld = cap + 2
    h = _layout_dev(ep, inp, A)
    q = torch.full((cap, H), SENT8, dtype=torch.uint8, device="cuda")
    sc = torch.full((nb * ld,) if col else (cap, nb), 0xEE if ue else -1.0,
                    dtype=torch.uint8 if ue else torch.float32, device="cuda")
    ep.ep_dispatch_ex(h, _dev(codes), q, cap, in_dtype=fmt, out_dtype=fmt,
                      scale_mode=ep.EP_SCALE_UE8M0 if ue else ep.EP_SCALE_FP32, x_scales=_dev(scales),
                      recv_scales=sc, scales_col_major=col, scales_ld=ld if col else 0, H=H)
    torch.cuda.synchronize()
    r_q = oracle.dispatch_rows(codes, ref["row_of_slot"], n)
    r_s = oracle.dispatch_rows(scales, ref["row_of_slot"], n)
    oracle.fill_pad_rows(ref, r_q, scales=None if ue else r_s)
    if ue:
        for e in range(E):
            r_s[ref["expert_offsets"][e] + ref["num_tokens_per_expert"][e]:ref["expert_offsets"][e + 1]] = 0
    gq = q.cpu().numpy()
    np.testing.assert_array_equal(gq[:n], r_q)
    assert (gq[n:] == SENT8).all()
    g = sc.cpu().numpy()
    got_s = g.reshape(nb, ld)[:, :n].T if col else g[:n]
    np.testing.assert_array_equal(got_s.view(np.uint8) if ue else got_s.view(np.uint32),
                                  r_s.view(np.uint8) if ue else r_s.view(np.uint32))
    h.destroy()
