"""CPU-only checks of the C ABI library: it builds, loads, exports every
symbol include/ep.h declares, rejects bad arguments on the host before any
CUDA call, and the binding fails loudly when the library is missing."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from combine_get_dispatch_layout_gb300.build import build
    import combine_get_dispatch_layout_gb300 as ep

    build()
    return ep.lib()


def declared_symbols():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"EP_API\s+[\w\s\*]+?\b(ep_\w+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 7
    for n in names:
        assert hasattr(L, n), n
    import combine_get_dispatch_layout_gb300 as ep
    assert sorted(ep.EXPORTS) == names


def test_status_strings(L):
    import combine_get_dispatch_layout_gb300 as ep
    assert ep.status_string(0) == "EP_OK"
    assert ep.status_string(3) == "EP_ERR_CAPACITY"
    assert ep.status_string(99) == "EP_ERR_UNKNOWN"


def _layout(L, T=4, K=2, E=8, R=2, null_handle=False, idx=16, outs=(32, 32, 32, 32)):
    h = ctypes.c_void_p(None)
    return L.ep_layout(idx, T, K, E, R, *outs, None, None, None if null_handle else ctypes.byref(h), None)


@pytest.mark.parametrize("kw", [
    dict(null_handle=True),
    dict(E=6, R=4),          # E % R != 0
    dict(K=0), dict(K=33),   # top-k range
    dict(E=0), dict(E=5000), dict(R=2000, E=2000),
    dict(T=-1),
    dict(T=1 << 28, K=8),    # T*K >= 2^31
    dict(idx=None),          # T > 0 needs topk_idx
    dict(idx=12),            # topk_idx not 8-byte aligned
    dict(outs=(None, 32, 32, 32)),
    dict(outs=(32, 32, 32, 34)),
])
def test_layout_rejects_bad_args(L, kw):
    assert _layout(L, **kw) == 1


def test_other_calls_reject_null_handle(L):
    assert L.ep_dispatch(None, 16, 128, 0, None, 16, None, None, None, 10, None) == 1
    assert L.ep_combine(None, 16, 10, 128, None, 16, None) == 1
    assert L.ep_handle_query(None, None, None) == 1
    assert L.ep_handle_copy_row_of_slot(None, 16, None) == 1
    assert L.ep_handle_destroy(None) == 0


def test_binding_fails_loudly_without_library(monkeypatch):
    import combine_get_dispatch_layout_gb300 as ep
    monkeypatch.setattr(ep, "_lib", None)
    monkeypatch.setattr(ep, "_LIB_PATH", os.path.join(ROOT, "does-not-exist.so"))
    with pytest.raises(RuntimeError, match="not built"):
        ep.lib()


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "combine_get_dispatch_layout_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", src), f"{f} mentions the oracle"
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert "combine_get_dispatch_layout_gb300" not in src and "libep" not in src


def _handle_ptr():
    return ctypes.byref(ctypes.c_void_p(None))


@pytest.mark.parametrize("align", [0, -3, 1025])
def test_layout_aligned_rejects_bad_alignment(L, align):
    assert L.ep_layout_aligned(16, 4, 2, 8, 2, align, 32, 32, 32, 32, None, None, _handle_ptr(), None) == 1


def test_layout_aligned_rejects_rows_past_int32(L):
    # T*K = 2^31 - 8 is allowed alone, but T*K + E*(A-1) >= 2^31
    assert L.ep_layout_aligned(16, (1 << 28) - 1, 8, 4096, 1, 1024, 32, 32, 32, 32, None, None, _handle_ptr(),
                               None) == 1


@pytest.mark.parametrize("cap", [0, -1])
def test_layout_strided_rejects_bad_capacity(L, cap):
    assert L.ep_layout_strided(16, 4, 2, 8, 2, cap, 32, 32, 32, 32, None, None, _handle_ptr(), None) == 1


def test_layout_strided_rejects_rows_past_int32(L):
    assert L.ep_layout_strided(16, 4, 2, 4096, 2, 1 << 20, 32, 32, 32, 32, None, None, _handle_ptr(), None) == 1


def test_layout_nonexpand_rejects_bad_args(L):
    assert L.ep_layout_nonexpand(16, 4, 2, 6, 4, 32, 32, 32, 32, None, None, _handle_ptr(), None) == 1  # E % R
    assert L.ep_layout_nonexpand(16, 4, 2, 8, 2, 32, 32, 32, 32, None, None, None, None) == 1           # no handle


def test_new_calls_reject_null_handle(L):
    import combine_get_dispatch_layout_gb300 as ep
    cfg = ep.DispatchConfig()
    assert L.ep_dispatch_ex(None, 16, None, 128, ctypes.byref(cfg), None, 16, None, None, None, 8, None) == 1
    assert L.ep_combine_backward(None, 16, 16, 8, 128, None, 16, 8, None, None) == 1
    assert L.ep_dispatch_backward(None, 16, 8, 128, None, 16, None, None) == 1
    assert L.ep_nonexpand_recv_topk(None, 16, None, 8, 16, None, 8, None) == 1
    assert L.ep_handle_layout_kernels(None) == -1


def test_cluster_query_rejects_bad_routings_without_a_device(L):
    # argument checks come before any device query
    for args in [(-1, 8, 256, 8), (16, 0, 256, 8), (16, 33, 256, 8), (16, 8, 0, 8), (16, 8, 256, 0),
                 (16, 8, 255, 8), (16, 8, 8192, 8), (1 << 30, 8, 256, 8)]:
        assert L.ep_layout_cluster_ctas(*args) == -1, args
    assert L.ep_layout_cluster_ctas(0, 8, 256, 8) == 0      # no tokens: nothing is launched


@pytest.mark.parametrize("args", [
    (16, None, 4, 0, 8),        # K = 0
    (16, None, 4, 33, 8),       # K > 32
    (16, None, 4, 2, 0),        # E = 0
    (16, None, -1, 2, 8),       # T < 0
    (None, None, 4, 2, 8),      # topk_idx missing
    (12, None, 4, 2, 8),        # topk_idx not 8-byte aligned
])
def test_topk_to_routing_map_rejects_bad_args(L, args):
    idx, w, T, K, E = args
    assert L.ep_topk_to_routing_map(idx, w, T, K, E, 64, None, None, None) == 1


def test_topk_to_routing_map_probs_need_weights(L):
    assert L.ep_topk_to_routing_map(16, None, 4, 2, 8, 64, 64, None, None) == 1


@pytest.mark.parametrize("args", [(64, 4, 8, 0), (64, 4, 0, 2), (None, 4, 8, 2), (64, -1, 8, 2)])
def test_routing_map_to_topk_rejects_bad_args(L, args):
    rm, T, E, K = args
    assert L.ep_routing_map_to_topk(rm, None, T, E, K, 16, None, None, None) == 1


def test_dispatch_config_struct_matches_header():
    """The binding's ep_dispatch_config_t mirror has the header's field order and size."""
    import combine_get_dispatch_layout_gb300 as ep
    src = open(os.path.join(ROOT, "include", "ep.h")).read()
    body = src[src.index("typedef struct {", src.index("ep_scale_mode_t;")):src.index("} ep_dispatch_config_t;")]
    fields = re.findall(r"^\s*(?:int|int64_t)\s+(\w+);", body, flags=re.M)
    assert fields == [f for f, _ in ep.DispatchConfig._fields_]
    assert ctypes.sizeof(ep.DispatchConfig) == 32


def test_enum_constants_match_header():
    """Every enumerator the header defines has the same value in the binding."""
    import combine_get_dispatch_layout_gb300 as ep
    src = open(os.path.join(ROOT, "include", "ep.h")).read()
    enums = dict((k, int(v)) for k, v in re.findall(r"^\s*(EP_[A-Z0-9_]+)\s*=\s*(\d+)\s*,?", src, flags=re.M))
    assert {"EP_DTYPE_FP8_E5M2", "EP_SCALE_UE8M0", "EP_ERR_ALLOC"} <= set(enums)
    for name, value in enums.items():
        assert getattr(ep, name) == value, name


def test_binding_refuses_tensors_the_kernels_cannot_index():
    """The binding passes raw addresses: a non-contiguous view or a pageable
    host tensor is refused before any call (empty tensors and raw ints pass)."""
    import torch
    import combine_get_dispatch_layout_gb300 as ep
    base = torch.zeros(8, 16, dtype=torch.int16)
    with pytest.raises(ValueError, match="contiguous"):
        ep._ptr(base[:, :8])
    with pytest.raises(ValueError, match="contiguous"):
        ep._ptr(base.t())
    with pytest.raises(ValueError, match="pinned"):
        ep._ptr(base)
    assert ep._ptr(None) is None
    assert ep._ptr(1234) == 1234
    assert ep._ptr(torch.empty(0, 4)) is not None


def test_binding_refuses_wrong_types_and_short_buffers():
    """Index arrays must be int64 and every tensor must hold the bytes the
    call will touch; the binding raises before any call into the library."""
    import torch
    import combine_get_dispatch_layout_gb300 as ep
    T, K, E, R, H = 4, 2, 8, 2, 256
    idx = torch.zeros(T, K, dtype=torch.int64)
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)
    outs = [i32(E), i32(R), torch.zeros(T, R, dtype=torch.uint8), i32(E + 1)]
    with pytest.raises(ValueError, match="int64"):
        ep.ep_layout(idx.to(torch.int32), E, R, *outs)
    with pytest.raises(ValueError, match="is_token_in_rank"):
        ep.ep_layout(idx, E, R, outs[0], outs[1], torch.zeros(T * R - 1, dtype=torch.uint8), outs[3])
    with pytest.raises(ValueError, match="offsets"):
        ep.ep_layout(idx, E, R, outs[0], outs[1], outs[2], i32(E))
    h = ep.Handle()
    h.T, h.K, h.E = T, K, E                      # a routing shape, no library handle
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="recv_x"):
        ep.ep_dispatch(h, x, ep.EP_DTYPE_BF16, torch.zeros(T * K - 1, H, dtype=torch.bfloat16), T * K)
    with pytest.raises(ValueError, match="recv_scales"):
        ep.ep_dispatch_ex(h, x, torch.zeros(T * K, H, dtype=torch.uint8), T * K,
                          recv_scales=torch.zeros(T * K, H // 128 - 1, dtype=torch.float32))
    with pytest.raises(ValueError, match="topk_weights"):
        ep.ep_dispatch(h, x, ep.EP_DTYPE_BF16, torch.zeros(T * K, H, dtype=torch.bfloat16), T * K,
                       recv_weights=torch.zeros(T * K), topk_weights=torch.zeros(T, K - 1))
    with pytest.raises(ValueError, match="out"):
        ep.ep_combine(h, torch.zeros(T * K, H, dtype=torch.bfloat16), torch.zeros(T - 1, H, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="grad_x"):
        ep.ep_dispatch_backward(h, torch.zeros(T * K, H, dtype=torch.bfloat16),
                                torch.zeros(T - 1, H, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="routing_map"):
        ep.ep_topk_to_routing_map(idx, E, torch.zeros(T, E - 1, dtype=torch.uint8))
    with pytest.raises(ValueError, match="topk_idx"):
        ep.ep_routing_map_to_topk(torch.zeros(T, E, dtype=torch.uint8), K, torch.zeros(T, K, dtype=torch.int32))
    with pytest.raises(ValueError, match="dst"):
        ep.ep_handle_copy_row_of_slot(h, i32(T * K - 1))


def test_header_is_plain_c99_and_links(tmp_path):
    """include/ep.h compiles as strict C99 (no C++ constructs) and a C program
    links against libep.so and calls it (ep_status_string needs no GPU)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    import combine_get_dispatch_layout_gb300 as ep
    ep.lib()                                             # built in-tree
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.join(root, "combine_get_dispatch_layout_gb300")
    src = tmp_path / "use_ep.c"
    src.write_text('#include <string.h>\n#include "ep.h"\n'
                   'int main(void) {\n'
                   '    ep_handle_t h = 0;\n'
                   '    (void)h;\n'
                   '    return strcmp(ep_status_string(EP_OK), ep_status_string(EP_ERR_INVALID_ARG)) == 0;\n'
                   '}\n')
    exe = tmp_path / "use_ep"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(root, "include"),
                    str(src), "-L", libdir, "-lep", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    assert subprocess.run([str(exe)]).returncode == 0
