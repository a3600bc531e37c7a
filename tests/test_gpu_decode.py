"""GPU parity of the decode / recurrent step (kda_decode_fwd) against the fp64
oracle, and its agreement with the chunked prefill on the same tokens.

The decode step is the token recurrence itself, so the oracle pins it
directly; the tolerance is the stated bar (relative L2 <= 1e-2 and max-abs <=
3e-2 * RMS, o and final_state separately) although the step runs in fp32.
"""
import numpy as np
import pytest
import torch

import kda_chunked_prefill_gb300 as kda
from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu


def run_decode(inp, num_seqs, in_place=False):
    d = pu.to_device(inp)
    state = d["initial_state"]
    if in_place and state is None:
        state = torch.zeros(num_seqs, inp["q"].shape[1], 128, 128, device="cuda")
    o, fs = kda.decode_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], num_seqs, state, scale=inp["scale"],
                           lower_bound=inp["lower_bound"], in_place=in_place, check=True)
    torch.cuda.synchronize()
    return o, fs


@pytest.mark.parametrize("N,Tn,H,state", [(1, 1, 2, True), (7, 1, 16, True), (64, 1, 16, False),
                                          (5, 3, 4, True), (3, 64, 2, True), (256, 1, 16, True)])
def test_decode_matches_the_oracle(N, Tn, H, state):
    inp = kin.make_inputs([Tn] * N, H, seed=100 + N + Tn, state_std=0.02 if state else None)
    o, fs = run_decode(inp, N)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(o.cpu().numpy(), ref_o, "o")
    pu.assert_parity(fs.cpu().numpy(), ref_s, "final_state")
    assert pu.errors(o.cpu().numpy(), ref_o)["rel_l2"] < 1e-4  # fp32 throughout


def test_decode_in_place_state_update():
    inp = kin.make_inputs([2] * 9, 4, seed=3, state_std=0.02)
    ref_o, ref_s = pu.run_oracle(inp)
    o, fs = run_decode(inp, 9, in_place=True)
    pu.assert_parity(o.cpu().numpy(), ref_o, "o")
    pu.assert_parity(fs.cpu().numpy(), ref_s, "final_state (in place)")


def test_decode_agrees_with_the_chunked_prefill():
    inp = kin.make_inputs([5] * 12, 8, seed=11, state_std=0.02)
    o_dec, s_dec = run_decode(inp, 12)
    o_pre, s_pre = pu.run_gpu(inp)
    pu.assert_parity(o_dec.cpu().numpy(), o_pre.cpu().numpy().astype(np.float64), "o decode vs prefill")
    pu.assert_parity(s_dec.cpu().numpy(), s_pre.cpu().numpy().astype(np.float64), "state decode vs prefill")


def test_prefill_then_decode_continues_the_sequence():
    """Prefill the first 200 tokens of each sequence, then decode the next 2
    from its final state: the result is the oracle on all 202 tokens."""
    H, N, L, Tn = 4, 3, 200, 2
    full = kin.make_inputs([L + Tn] * N, H, seed=21, state_std=0.02)
    ref_o, ref_s = pu.run_oracle(full)
    rows_pre = np.concatenate([np.arange(n * (L + Tn), n * (L + Tn) + L) for n in range(N)])
    rows_dec = np.concatenate([np.arange(n * (L + Tn) + L, (n + 1) * (L + Tn)) for n in range(N)])
    pre = dict(full)
    for key in ("q", "k", "v", "g", "beta"):
        pre[key] = full[key][rows_pre]
    pre["cu_seqlens"] = torch.arange(0, N * L + 1, L, dtype=torch.int32)
    _, state = pu.run_gpu(pre)
    dec = {key: full[key][rows_dec].cuda() for key in ("q", "k", "v", "g", "beta")}
    o, fs = kda.decode_fwd(dec["q"], dec["k"], dec["v"], dec["g"], dec["beta"], N, state, scale=full["scale"],
                           lower_bound=full["lower_bound"], check=True)
    torch.cuda.synchronize()
    pu.assert_parity(o.cpu().numpy(), ref_o[rows_dec], "o of the decoded tokens")
    pu.assert_parity(fs.cpu().numpy(), ref_s, "final_state after decoding")


def test_zero_tokens_pass_the_state_through():
    H, N = 2, 3
    s0 = torch.randn(N, H, 128, 128, device="cuda") * 0.02
    empty = torch.empty(0, H, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(0, H, 128, device="cuda")
    fs = torch.empty_like(s0)
    kda.kda_decode_fwd(empty, empty, empty, empty.float(), torch.empty(0, H, device="cuda"), N, s0, 0.088, -5.0,
                       o, fs)
    torch.cuda.synchronize()
    assert torch.equal(fs, s0)


def test_decode_reports_gates_out_of_range():
    inp = kin.make_inputs([1] * 4, 2, seed=5)
    inp["g"][2, 1, 7] = -7.0  # below lower_bound = -5
    with pytest.raises(kda.KdaError) as e:
        run_decode(inp, 4)
    assert e.value.code == kda.KDA_ERR_GATE_RANGE
