"""Multi-rank aggregation of bench.py on CPU: two gloo ranks, each a replica
with its own step time and bytes; the job time is the slowest rank's and the
bytes are summed (no data exchange between replicas)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, nbytes = bench.aggregate_over_ranks(1.5 + rank, 1000 * (rank + 1))
        out[rank] = (ms, nbytes)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert out[0] == out[1] == (2.5, 3000)


def test_single_process_is_identity():
    import bench
    assert bench.aggregate_over_ranks(3.0, 7) == (3.0, 7)


def test_traffic_marker_needs_matching_size_and_source(tmp_path, monkeypatch):
    """The roofline's measured traffic is reported only for the token count it
    was captured on and while the kernel source is unchanged."""
    import hashlib

    import bench
    csrc = tmp_path / "combine_get_dispatch_layout_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "ep_combine.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "dram_traffic_prefill_T8192.md").write_text(
        f"text\n<!-- traffic kernel=combine T=8192 bytes=1234 src_sha256={sha} -->\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic("combine", 8192) == 1234
    assert bench.read_traffic("combine", 2048) is None
    assert bench.read_traffic("dispatch_bf16", 8192) is None
    src.write_text("// kernel v2\n")
    assert bench.read_traffic("combine", 8192) is None
