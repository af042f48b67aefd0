"""The oracle's e4m3 and e5m2 encoders against the GPU's conversion
instructions (cvt.rn.satfinite.{e4m3x2,e5m2x2}.f32, the ones the fp8
dispatch uses) on every one of the 2^32 fp32 bit patterns.

The device converts a chunk of patterns into shared host memory; worker
processes (started with spawn, see fp8_sweep_worker.py) run the oracle's
sweeps over slices of the chunk and compare them. NaN inputs are outside the
contract and only have to come back as a NaN code."""
import ctypes
import multiprocessing as mp
import os
import subprocess
from multiprocessing import shared_memory

import numpy as np
import pytest
import torch

from fp8_sweep_worker import compare_slice

HERE = os.path.dirname(os.path.abspath(__file__))
CHUNK = 1 << 28


@pytest.fixture(scope="module")
def sweep_lib(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("cvt") / "libfp8_cvt_sweep.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", "-o", so, os.path.join(HERE, "fp8_cvt_sweep.cu")], check=True)
    lib = ctypes.CDLL(so)
    lib.fp8_cvt_sweep.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p]
    lib.fp8_cvt_sweep.restype = ctypes.c_int
    return lib


@pytest.mark.gpu
def test_oracle_encoders_match_the_gpu_on_all_fp32_patterns(sweep_lib):
    import oracle
    oracle.build()
    dev = torch.device("cuda:0")
    q4 = torch.empty(CHUNK, dtype=torch.uint8, device=dev)
    q5 = torch.empty(CHUNK, dtype=torch.uint8, device=dev)
    sh4 = shared_memory.SharedMemory(create=True, size=CHUNK)
    sh5 = shared_memory.SharedMemory(create=True, size=CHUNK)
    workers = max(1, min(16, len(os.sched_getaffinity(0))))
    part = CHUNK // 64
    failures = []
    compared = {"e4m3": 0, "e5m2": 0}
    try:
        h4 = np.ndarray((CHUNK,), np.uint8, buffer=sh4.buf)
        h5 = np.ndarray((CHUNK,), np.uint8, buffer=sh5.buf)
        with mp.get_context("spawn").Pool(workers) as pool:
            for lo in range(0, 1 << 32, CHUNK):
                assert sweep_lib.fp8_cvt_sweep(lo, CHUNK, q4.data_ptr(), q5.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream) == 0
                torch.cuda.synchronize()
                h4[:] = q4.cpu().numpy()
                h5[:] = q5.cpu().numpy()
                jobs = [(sh4.name, sh5.name, off, lo + off, part) for off in range(0, CHUNK, part)]
                for res in pool.map(compare_slice, jobs):
                    for fmt, (n, count, first) in zip(("e4m3", "e5m2"), res):
                        compared[fmt] += n
                        if count:
                            failures.append((fmt, count, first))
        del h4, h5
    finally:
        sh4.close(); sh4.unlink()
        sh5.close(); sh5.unlink()
    assert failures == [], failures[:8]
    assert compared == {"e4m3": 1 << 32, "e5m2": 1 << 32}
