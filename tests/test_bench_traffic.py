"""bench.py reports a kernel's measured DRAM traffic only while the committed
ncu summary was taken of the same token count and the same kernel source:
the per-launch bytes come from a marker in profiles/, keyed by a hash of the
kernel's source file, and a changed source or another size gives null."""
import hashlib
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "combine_get_dispatch_layout_gb300", "csrc")


def _sha16(name):
    return hashlib.sha256(open(os.path.join(CSRC, name), "rb").read()).hexdigest()[:16]


def test_committed_markers_match_the_current_sources():
    # the summaries in profiles/ were taken at the current kernel sources
    for kernel, T, case in [("combine", 8192, "prefill"), ("dispatch_bf16", 8192, "prefill"),
                            ("combine", 16384, "skewed")]:
        assert isinstance(bench.read_traffic(kernel, T, case), int), (kernel, case)


def test_markers_are_keyed_by_size_source_and_kernel(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    good = _sha16("ep_combine.cu")
    (prof / "dram_traffic_prefill_T4096.md").write_text(
        f"<!-- traffic kernel=combine T=4096 bytes=123456 src_sha256={good} -->\n"
        f"<!-- traffic kernel=dispatch_bf16 T=4096 bytes=999 src_sha256=0000000000000000 -->\n")
    (prof / "dram_traffic_skewed_T64.md").write_text(
        f"<!-- traffic kernel=combine case=skewed T=64 bytes=77 src_sha256={good} -->\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the hash is taken of the real source, which lives under the tree's csrc
    os.makedirs(tmp_path / "combine_get_dispatch_layout_gb300", exist_ok=True)
    os.symlink(CSRC, tmp_path / "combine_get_dispatch_layout_gb300" / "csrc")
    assert bench.read_traffic("combine", 4096) == 123456
    assert bench.read_traffic("dispatch_bf16", 4096) is None      # another source: stale
    assert bench.read_traffic("combine", 2048) is None            # no capture of that size
    assert bench.read_traffic("layout", 4096) is None             # no source mapping
    assert bench.read_traffic("combine", 64, "skewed") == 77
    assert bench.read_traffic("combine", 64) is None              # the prefill case has no such file
