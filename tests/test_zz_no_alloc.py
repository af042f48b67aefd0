"""The allocation-free layout entry point against the handle-based one.

ep_layout_noalloc serves callers that cannot allocate device memory (all of
it belongs to another allocator, or cudaMalloc's implicit synchronisation is
not allowed where they run); it keeps its scratch in a fixed array inside
the library. This file is named to be collected last, so a run that stops
at the first failure has already run every other test. It passes alone in a
fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from gen import inputs as gi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    import combine_get_dispatch_layout_gb300 as m
    from combine_get_dispatch_layout_gb300.build import build

    build()
    m.lib()
    torch.cuda.set_device(0)
    return m


def _outs(T, K, E, R):
    return dict(num_tokens_per_expert=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
                num_tokens_per_rank=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                is_token_in_rank=torch.full((T, R), 0xA5, dtype=torch.uint8, device="cuda"),
                expert_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
                row_of_slot=torch.full((T, K), -9, dtype=torch.int32, device="cuda"))


def _with_handle(ep, idx, E, R):
    T, K = idx.shape
    o = _outs(T, K, E, R)
    h = ep.ep_layout(idx, E, R, o["num_tokens_per_expert"], o["num_tokens_per_rank"],
                     o["is_token_in_rank"], o["expert_offsets"])
    ep.ep_handle_copy_row_of_slot(h, o["row_of_slot"])
    _, err = ep.ep_handle_query(h)
    h.destroy()
    return {k: v.cpu().numpy() for k, v in o.items()}, err


def _no_alloc(ep, idx, E, R, with_error=True):
    T, K = idx.shape
    o = _outs(T, K, E, R)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ep.ep_layout_noalloc(idx, E, R, o["num_tokens_per_expert"], o["num_tokens_per_rank"],
                         o["is_token_in_rank"], o["expert_offsets"], o["row_of_slot"],
                         device_error=err if with_error else None)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}, int(err.item()) if with_error else None


def _cases():
    prefill = gi.make("prefill", 0, with_y=False)
    skewed = gi.make("skewed", 1, with_y=False)
    rng = np.random.default_rng(7)
    bad = np.argsort(rng.random((300, 16)), axis=1)[:, :4].astype(np.int64)
    bad[3, 2], bad[77, 0] = 16, -5
    large = gi.make(gi.Workload("large", T=40000, H=128, E=64, K=8, R=4, routing="zipf", drop_p=0.05),
                    3, with_y=False)
    # 2^18 slots on one cluster: 16 rounds a warp, the packed instance of the cluster kernel
    packed = gi.make(gi.Workload("packed", T=32768, H=64, E=256, K=8, R=8, drop_p=0.02), 4, with_y=False)
    return [(prefill.topk_idx, 256, 8), (skewed.topk_idx, 64, 4), (bad, 16, 4),
            (large.topk_idx, 64, 4), (gi.make("decode", 2, with_y=False).topk_idx, 256, 8),
            (packed.topk_idx, 256, 8)]


def test_no_alloc_matches_layout_on_consecutive_calls(ep):
    # consecutive calls share the scratch array: each must match the handle path,
    # including after a call that saw invalid ids (its error flag must not leak)
    for idx_np, E, R in _cases():
        idx = torch.from_numpy(idx_np).cuda()
        want, want_err = _with_handle(ep, idx, E, R)
        for _ in range(2):
            got, got_err = _no_alloc(ep, idx, E, R)
            assert got_err == want_err
            for k in want:
                np.testing.assert_array_equal(got[k], want[k], err_msg=k)


def test_no_alloc_rejects_routings_beyond_the_scratch(ep):
    T, K, E, R = 4096, 8, 4096, 1024      # (E + R) * 256 words > 2 MiB
    idx = torch.zeros((T, K), dtype=torch.int64, device="cuda")
    o = _outs(T, K, E, R)
    with pytest.raises(ep.EPError) as e:
        ep.ep_layout_noalloc(idx, E, R, o["num_tokens_per_expert"], o["num_tokens_per_rank"],
                             o["is_token_in_rank"], o["expert_offsets"], o["row_of_slot"])
    assert e.value.status == ep.EP_ERR_CAPACITY


def test_no_alloc_without_error_word_and_with_no_tokens(ep):
    # device_error may be NULL; T = 0 zeroes the counts and offsets, as the handle path does
    idx_np = gi.make("tiny", 3, with_y=False).topk_idx
    idx = torch.from_numpy(idx_np).cuda()
    want, _ = _with_handle(ep, idx, 8, 2)
    got, _ = _no_alloc(ep, idx, 8, 2, with_error=False)
    for k in want:
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    empty = torch.zeros((0, 2), dtype=torch.int64, device="cuda")
    want0, err0 = _with_handle(ep, empty, 8, 2)
    for with_error in (True, False):
        got0, e = _no_alloc(ep, empty, 8, 2, with_error=with_error)
        for k in ("num_tokens_per_expert", "num_tokens_per_rank", "expert_offsets"):
            np.testing.assert_array_equal(got0[k], want0[k], err_msg=k)
        assert not got0["expert_offsets"].any()
        if with_error:
            assert e == err0 == 0
