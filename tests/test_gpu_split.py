"""GPU parity of kda_chunk_fwd_split, the split-sequence scan: long sequences
cut into segments whose entry states come from composing each segment's affine
state map (the chunk recurrence of the TPU report's §6.2 is affine in S), then
run as sequences of their own. Checked against the fp64 oracle (the token
recurrence over the whole sequences) at the parity bar, with forced segment
lengths on small cases (several segments, ragged last segments, unsplit and
empty sequences beside split ones), against the plain call, and on the long
few-head workload with the planned segment length."""
import numpy as np
import pytest
import torch

import kda_chunked_prefill_gb300 as kda
from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu


def _run_split(inp, segment_chunks, output_final_state=True):
    d = pu.to_device(inp)
    o, fs = kda.chunk_fwd_split(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                cu_seqlens_host=inp["cu_seqlens"], initial_state=d["initial_state"],
                                scale=inp["scale"], lower_bound=inp["lower_bound"],
                                output_final_state=output_final_state, check=True, segment_chunks=segment_chunks)
    torch.cuda.synchronize()
    return o.cpu().numpy(), (None if fs is None else fs.cpu().numpy())


CASES = {
    # name: (seqlens, H, initial state std, segment length in chunks)
    "four_segments_ragged_tail": ([700, 130, 64], 3, 0.02, 3),
    "eight_segments": ([1000], 2, 0.02, 2),
    "empty_and_short_beside_split": ([0, 640, 0, 65, 1], 2, 0.02, 2),
    "no_initial_state": ([900, 200], 2, None, 4),
    "one_chunk_segments": ([400, 63], 2, 0.02, 1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_split_matches_oracle(name):
    lens, H, s0, L = CASES[name]
    inp = kin.make_inputs(lens, H, seed=700 + sum(lens), state_std=s0)
    o, fs = _run_split(inp, L)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(o, ref_o, "o")
    pu.assert_parity(fs, ref_s, "final_state")


def test_split_without_final_state_writes_the_same_o():
    inp = kin.make_inputs([700, 130], 3, seed=11, state_std=0.02)
    o1, _ = _run_split(inp, 3, output_final_state=False)
    o2, _ = _run_split(inp, 3)
    assert np.array_equal(o1, o2)


def test_split_agrees_with_the_plain_call():
    """Same inputs through the plain call and the split call (16 segments): the
    two differ only by the fp32 combine's rounding, far inside the bar."""
    inp = kin.make_inputs([8192, 300], 4, seed=12, state_std=0.02)
    o_s, fs_s = _run_split(inp, 8)
    o_p, fs_p = pu.run_gpu(inp, check=True)
    for a, b in ((o_s, o_p.cpu().numpy()), (fs_s, fs_p.cpu().numpy())):
        e = pu.errors(a, b)
        assert e["rel_l2"] < 2e-3 and e["max_abs"] < 2e-2 * e["rms_ref"], e


def test_split_long_few_head_workload_planned():
    """1 x 65536 tokens, H = 4, with the planned segment length (the benchmark's
    launch configuration for this workload), against the oracle on all heads."""
    wl = kin.workloads()["long_1x65536_H4"]
    inp = kin.make_workload(wl)
    L = kda.split_plan(inp["cu_seqlens"], wl.num_heads)
    assert L > 0
    o, fs = _run_split(inp, 0)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(o, ref_o, "o")
    pu.assert_parity(fs, ref_s, "final_state")
