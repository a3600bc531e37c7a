"""The allocation-free entry point, kda_chunk_fwd_static_scratch, for callers
that cannot allocate device memory (not even a workspace): it takes its
scratch from a fixed array inside the library. Called through the C ABI, it
runs the same deterministic kernel as the ordinary entry point, so its
results must equal that entry point's bit for bit, on calls in a row (each
call reuses the array the previous one left behind, including a small call
after a large one). A build of the entry point with a deliberately small
array shows the size limit: a problem that needs more scratch is refused with
KDA_ERR_SCRATCH_TOO_SMALL and nothing runs, while one that fits still
matches. This file is named to be collected last."""
import ctypes
import glob
import os
import subprocess
import tempfile

import pytest
import torch

from kda_chunked_prefill_gb300 import _lib
from kda_chunked_prefill_gb300 import build as kbuild
from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu

SMALL_SCRATCH_BYTES = 1 << 20


def _static_fn(lib):
    f = lib.kda_chunk_fwd_static_scratch
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, f32, f32, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def run_static(inp, lib=None, expect=_lib.KDA_OK):
    f = _static_fn(lib if lib is not None else _lib.load_library(build_if_missing=True))
    d = pu.to_device(inp)
    T, H, D = inp["q"].shape
    N = len(inp["seqlens"])
    o = torch.full((T, H, D), float("nan"), dtype=torch.float32, device="cuda")
    fs = torch.full((N, H, D, D), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    rc = f(_ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["g"]), _ptr(d["beta"]), _ptr(d["cu_seqlens"]),
           N, T, H, D, D, _ptr(d["initial_state"]), inp["scale"], inp["lower_bound"], _ptr(o), _ptr(fs),
           _ptr(status), ctypes.c_void_p(stream.cuda_stream))
    assert rc == expect, _lib.status_string(rc)
    torch.cuda.synchronize()
    if expect != _lib.KDA_OK:
        assert torch.isnan(o).all() and torch.isnan(fs).all(), "a refused call wrote its outputs"
        return None, None
    assert int(status.item()) == _lib.KDA_OK
    return o, fs


def _assert_same(inp, lib=None):
    o_s, f_s = run_static(inp, lib)
    o_w, f_w = pu.run_gpu(inp)
    assert torch.equal(o_s, o_w), "o differs between the static-scratch and the workspace entry points"
    assert torch.equal(f_s, f_w), "final_state differs between the static-scratch and the workspace entry points"


def test_static_scratch_entry_matches_workspace_entry_bitwise():
    small = kin.make_inputs([130, 64, 210], 4, seed=21, state_std=0.02)
    cases = [small, kin.make_workload(kin.workloads()["headline_4x2048_H16"]), small]
    for inp in cases:  # calls in a row on the one array; the last one smaller than the one before
        _assert_same(inp)


def _small_scratch_library(tmp):
    """libkda built with a 1 MiB static scratch array: the other objects of the
    in-tree build, and kda_no_alloc.cu compiled again with the smaller size."""
    kbuild.build()
    objs = [o for o in sorted(glob.glob(os.path.join(kbuild.BUILD_DIR, "*.o")))
            if os.path.basename(o) != "kda_no_alloc.cu.o"]
    obj = os.path.join(tmp, "kda_no_alloc_small.o")
    src = os.path.join(kbuild.CSRC, "kda_no_alloc.cu")
    subprocess.run([kbuild.nvcc(), *kbuild.ARCH, *kbuild.NVCC_FLAGS, f"-DKDA_STATIC_SCRATCH_BYTES={SMALL_SCRATCH_BYTES}u",
                    "-I", kbuild.INCLUDE, "-I", kbuild.CSRC, "-c", src, "-o", obj], check=True, capture_output=True)
    so = os.path.join(tmp, "libkda_small_scratch.so")
    subprocess.run([kbuild.nvcc(), *kbuild.ARCH, "-shared", "-o", so, *objs, obj, "-lcudart"], check=True,
                   capture_output=True)
    return ctypes.CDLL(so)


def test_static_scratch_size_limit():
    lib = _lib.load_library(build_if_missing=True)
    need_small = lib.kda_chunk_fwd_workspace_size(1, 2)
    need_big = lib.kda_chunk_fwd_workspace_size(4, 16)
    assert 0 < need_small <= SMALL_SCRATCH_BYTES < need_big
    with tempfile.TemporaryDirectory() as tmp:
        small_lib = _small_scratch_library(tmp)
        run_static(kin.make_workload(kin.workloads()["headline_4x2048_H16"]), small_lib,
                   expect=_lib.KDA_ERR_SCRATCH_TOO_SMALL)
        _assert_same(kin.make_inputs([200], 2, seed=5, state_std=0.02), small_lib)
