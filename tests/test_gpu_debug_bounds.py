"""A library compiled with -DKDA_DEBUG_BOUNDS checks, before each global-memory
access of the prefill kernel, that its index lies inside the buffer (token rows
against the token count, heads, state rows, ring slots); a failed check would
record KDA_ERR_BOUNDS and skip the access. Run over workloads with ragged
tails, a one-token sequence, several sequences, long chains and an initial
state, it must report no failed check and give the same outputs, bit for bit,
as the ordinary build (the checks change no arithmetic)."""
import concurrent.futures as cf
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


@pytest.fixture(scope="module")
def bounds_lib():
    kbuild.build()
    with tempfile.TemporaryDirectory() as tmp:
        def compile_one(src):
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            subprocess.run([kbuild.nvcc(), *kbuild.ARCH, *kbuild.NVCC_FLAGS, "-DKDA_DEBUG_BOUNDS", "-I", kbuild.INCLUDE,
                            "-I", kbuild.CSRC, "-c", src, "-o", obj], check=True, capture_output=True)
            return obj
        with cf.ThreadPoolExecutor(max_workers=8) as ex:
            objs = list(ex.map(compile_one, sorted(glob.glob(os.path.join(kbuild.CSRC, "*.cu")))))
        so = os.path.join(tmp, "libkda_bounds.so")
        subprocess.run([kbuild.nvcc(), *kbuild.ARCH, "-shared", "-o", so, *objs, "-lcudart"], check=True,
                       capture_output=True)
        lib = ctypes.CDLL(so)
        yield lib


def _run(lib, inp):
    f = lib.kda_chunk_fwd
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, f32, f32, vp, vp, vp, vp, ctypes.c_size_t, vp]
    f.restype = ctypes.c_int
    lib.kda_chunk_fwd_workspace_size.argtypes = [i32, i32]
    lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_size_t
    d = pu.to_device(inp)
    T, H, D = inp["q"].shape
    N = len(inp["seqlens"])
    o = torch.full((T, H, D), float("nan"), dtype=torch.float32, device="cuda")
    fs = torch.full((N, H, D, D), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = lib.kda_chunk_fwd_workspace_size(N, H)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = f(P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), P(d["cu_seqlens"]), N, T, H, D, D,
           P(d["initial_state"]), inp["scale"], inp["lower_bound"], P(o), P(fs), P(status), P(ws), wsb,
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.KDA_OK, _lib.status_string(rc)
    torch.cuda.synchronize()
    return o, fs, int(status.item())


@pytest.mark.parametrize("case", ["ragged", "tiny", "headline"])
def test_bounds_checked_build_reports_nothing_and_matches(bounds_lib, case):
    if case == "ragged":
        inp = kin.make_inputs([130, 1, 64, 210, 63], 4, seed=31, state_std=0.02)
    else:
        inp = kin.make_workload(kin.workloads()["tiny_T256_H2" if case == "tiny" else "headline_4x2048_H16"])
    o_b, f_b, st = _run(bounds_lib, inp)
    assert st == _lib.KDA_OK, f"status {st}: {_lib.status_string(st)}"
    o_n, f_n = pu.run_gpu(inp)
    assert torch.equal(o_b, o_n) and torch.equal(f_b, f_n)
