"""kda_chunk_fwd_host: the forward on host-resident inputs and outputs. With the
default grouping and page-locked buffers the device addresses in place, one
launch reads and writes the host buffers directly; with an explicit grouping
(or pageable memory) the copies of each group of sequences overlap the
computation of its neighbours. The kernel's arithmetic per (sequence, head)
chain does not depend on which other chains share the launch or where the
buffers live, so every form must reproduce the device call bit for bit."""
import pytest
import torch

import kda_chunked_prefill_gb300 as kda
from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu


def _host_call(inp, groups, pinned=True, with_final=True, alias=False):
    T, H, _ = inp["q"].shape
    N = len(inp["seqlens"])
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    h = {key: (None if inp[key] is None else pin(inp[key].contiguous()))
         for key in ("q", "k", "v", "g", "beta", "initial_state")}
    o = pin(torch.empty(T, H, 128, dtype=torch.float32))
    if alias:
        fs = h["initial_state"]
    else:
        fs = pin(torch.empty(N, H, 128, 128, dtype=torch.float32)) if with_final else None
    nbytes = kda.host_buffer_size(inp["cu_seqlens"], H, h["initial_state"] is not None, fs is not None, groups)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    stream = torch.cuda.current_stream()
    kda.kda_chunk_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], inp["cu_seqlens"], h["initial_state"],
                           inp["scale"], inp["lower_bound"], o, fs, buf, status=status, groups=groups,
                           stream=stream, h2d_stream=s_in, d2h_stream=s_out)
    stream.synchronize()
    assert int(status.item()) == 0
    return o, fs


@pytest.mark.parametrize("groups", [0, 1, 2, 3, 16])
def test_host_call_equals_device_call_bitwise(groups):
    inp = kin.make_inputs([700, 64, 1, 333, 0, 129, 1000], 3, seed=31, state_std=0.02)
    o_d, fs_d = pu.run_gpu(inp)
    o_h, fs_h = _host_call(inp, groups)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(fs_h, fs_d.cpu())


def test_host_call_on_the_headline_workload_matches_oracle():
    inp = kin.make_workload(kin.workloads()["headline_4x2048_H16"])
    o, fs = _host_call(inp, 0)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(o.numpy(), ref_o, "o")
    pu.assert_parity(fs.numpy(), ref_s, "final_state")


def test_host_call_groups_of_empty_sequences_and_aliasing():
    """A group holding only empty sequences passes their states through; the
    final states may overwrite the initial ones in place."""
    inp = kin.make_inputs([0, 0, 150, 0], 2, seed=32, state_std=0.02)
    o_d, fs_d = pu.run_gpu(inp)
    o_h, fs_h = _host_call(inp, 4, alias=True)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(fs_h, fs_d.cpu())


def test_host_call_with_pageable_memory_and_no_final_state():
    inp = kin.make_inputs([300, 200], 2, seed=33)
    o_d, _ = pu.run_gpu(inp)
    o_h, fs_h = _host_call(inp, 2, pinned=False, with_final=False)
    assert fs_h is None and torch.equal(o_h, o_d.cpu())


def test_host_call_in_place_with_empty_sequences_and_aliasing():
    """The in-place form (default grouping, pinned buffers): empty sequences pass
    their states through and the final states overwrite the initial ones."""
    inp = kin.make_inputs([0, 0, 150, 0, 64], 2, seed=34, state_std=0.02)
    o_d, fs_d = pu.run_gpu(inp)
    o_h, fs_h = _host_call(inp, 0, alias=True)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(fs_h, fs_d.cpu())
