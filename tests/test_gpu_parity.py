"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element, at the stated tolerance (relative L2
<= 1e-2 and max-abs <= 3e-2 * RMS of the reference, for o and final_state
separately). Small cases span several chunks and ragged tails; the
full-size workloads run in the launch configuration the benchmark times and
are compared on all heads (headline, cached prefix) or on a sample of heads
the oracle computes one chain at a time (batch sweep, wide).
"""
import numpy as np
import pytest
import torch

from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu


def check_case(inp, heads=None):
    o, fs = pu.run_gpu(inp)
    ref_o, ref_s = pu.run_oracle(inp, heads=heads)
    sel = slice(None) if heads is None else list(heads)
    eo = pu.assert_parity(o[:, sel].float().cpu().numpy(), ref_o, "o")
    es = pu.assert_parity(fs[:, sel].cpu().numpy(), ref_s, "final_state")
    return eo, es


SMALL = {
    # name: (seqlens, H, with initial state, sigma_g)
    "one_chunk_T64": ([64], 2, False, 1.0),
    "page_lens_130_64_210": ([130, 64, 210], 4, True, 1.0),
    "below_subblock_T5": ([5], 2, True, 1.0),
    "exactly_subblock_T16": ([16], 1, False, 1.0),
    "single_token": ([1], 3, True, 1.0),
    "empty_and_ragged": ([0, 70, 0, 1, 64, 0, 129], 2, True, 1.0),
    "many_short": ([7, 33, 17, 64, 1, 100, 15, 48], 2, True, 1.0),
    "strong_decay_sigma2": ([300, 190], 3, True, 2.0),
    "aligned_multi_chunk": ([64, 128, 192, 256], 2, False, 1.0),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_cases(name):
    lens, H, state, sg = SMALL[name]
    inp = kin.make_inputs(lens, H, seed=100 + len(name), sigma_g=sg,
                          state_std=0.02 if state else None)
    check_case(inp)


def test_unequal_lengths_schedules():
    """Sequences of unequal length go to consumers by the longest-first table
    (up to 1024 chains) or, beyond that, by the plain stride order; both must
    cover every chain exactly once. Lengths include empty and one-token
    sequences; every head is checked against the oracle."""
    rng = np.random.default_rng(7)
    # 16 sequences of ~3000 tokens, H = 4: 64 chains, long enough for the table
    # to pay for itself; 70 short sequences, H = 16: 1120 chains (stride order)
    for n_seq, H, lo, hi in ((16, 4, 500, 5000), (70, 16, 0, 200)):
        lens = [int(x) for x in rng.integers(lo, hi, size=n_seq)]
        lens[3], lens[5] = 0, 1
        lens[7] = 7000  # one long sequence
        inp = kin.make_inputs(lens, H, seed=300 + n_seq, state_std=0.02)
        check_case(inp)


def test_tiny_workload():
    check_case(kin.make_workload(kin.workloads()["tiny_T256_H2"]))


def test_headline_workload_all_heads():
    check_case(kin.make_workload(kin.workloads()["headline_4x2048_H16"]))


def test_cached_prefix_workload_all_heads():
    check_case(kin.make_workload(kin.workloads()["cached_prefix_B16_H16"]))


def test_cached_prefix_every_sequence_on_its_own():
    """The parity bar applied to each sequence's o and final_state separately
    (each against its own RMS), not only to the whole tensors; the worst
    values are written as JSON to the file KDA_PARITY_REPORT names, if set."""
    import json
    import os
    inp = kin.make_workload(kin.workloads()["cached_prefix_B16_H16"])
    o, fs = pu.run_gpu(inp)
    ref_o, ref_s = pu.run_oracle(inp)
    o = o.float().cpu().numpy()
    fs = fs.cpu().numpy()
    cu = inp["cu_seqlens"].numpy()
    worst = {"o_rel_l2": 0.0, "o_maxabs_over_rms": 0.0, "S_rel_l2": 0.0, "S_maxabs_over_rms": 0.0}
    for n in range(len(cu) - 1):
        a, b = int(cu[n]), int(cu[n + 1])
        eo = pu.assert_parity(o[a:b], ref_o[a:b], f"o of sequence {n} ({b - a} tokens)")
        es = pu.assert_parity(fs[n], ref_s[n], f"final_state of sequence {n}")
        worst["o_rel_l2"] = max(worst["o_rel_l2"], eo["rel_l2"])
        worst["o_maxabs_over_rms"] = max(worst["o_maxabs_over_rms"], eo["max_abs"] / eo["rms_ref"])
        worst["S_rel_l2"] = max(worst["S_rel_l2"], es["rel_l2"])
        worst["S_maxabs_over_rms"] = max(worst["S_maxabs_over_rms"], es["max_abs"] / es["rms_ref"])
    report = os.environ.get("KDA_PARITY_REPORT")
    if report:
        with open(report, "w") as f:
            json.dump({"workload": "cached_prefix_B16_H16", "worst_over_sequences": worst}, f, indent=1)


@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 32, 64])
def test_batch_sweep_workload_all_heads(b):
    """B = 64 is 1024 chains, the largest count the longest-first schedule table takes."""
    inp = kin.make_workload(kin.workloads()[f"sweep_B{b}_H16"])
    o, fs = pu.run_gpu(inp)
    pu.assert_parity_by_head_groups(inp, o, fs, group=16)


@pytest.mark.parametrize("name", ["wide_3x8192_H96", "wide_1x16384_H96"])
def test_wide_workload_all_heads(name):
    inp = kin.make_workload(kin.workloads()[name])
    o, fs = pu.run_gpu(inp)
    pu.assert_parity_by_head_groups(inp, o, fs, group=16)


def test_zero_state_tensor_equals_null_state():
    inp = kin.make_inputs([100, 37], 2, seed=7)
    o1, f1 = pu.run_gpu(inp)
    inp2 = dict(inp)
    inp2["initial_state"] = torch.zeros(2, 2, 128, 128)
    o2, f2 = pu.run_gpu(inp2)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_final_state_in_place_over_initial_state():
    from kda_chunked_prefill_gb300 import kda_chunk_fwd
    inp = kin.make_inputs([90, 200], 2, seed=8, state_std=0.02)
    d = pu.to_device(inp)
    o_ref, f_ref = pu.run_gpu(inp)
    st = d["initial_state"].clone()
    o = torch.empty(d["v"].shape, dtype=torch.float32, device=d["v"].device)
    kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], st, inp["scale"],
                  inp["lower_bound"], o, st)  # default workspace
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(st, f_ref)


def test_final_state_not_requested():
    inp = kin.make_inputs([77], 2, seed=9)
    o1, _ = pu.run_gpu(inp)
    o2, f2 = pu.run_gpu(inp, output_final_state=False)
    assert f2 is None and torch.equal(o1, o2)


def test_deterministic_bitwise():
    inp = kin.make_workload(kin.workloads()["cached_prefix_B16_H16"])
    o1, f1 = pu.run_gpu(inp)
    o2, f2 = pu.run_gpu(inp)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_beta_one_self_query_reads_back_value():
    """beta = 1, q = k (unit rows): the oracle's closed form o_t = scale * v_t
    must hold on the GPU too, through the whole chunked solve."""
    inp = kin.make_inputs([200, 64], 2, seed=10, state_std=0.02)
    inp["q"] = inp["k"].clone()
    inp["beta"] = torch.ones_like(inp["beta"])
    o, _ = pu.run_gpu(inp)
    pu.assert_parity(o.float().cpu().numpy(), inp["scale"] * kin.to_f64(inp["v"]), "o vs scale*v")


def test_padding_does_not_change_valid_tokens():
    """A sequence followed by another one gives the same outputs as alone."""
    a = kin.make_inputs([70], 2, seed=11, state_std=0.02)
    b = kin.make_inputs([70, 50], 2, seed=11, state_std=0.02)
    for key in ("q", "k", "v", "g", "beta"):
        b[key][:70] = a[key]
    b["initial_state"][:1] = a["initial_state"]
    oa, fa = pu.run_gpu(a)
    ob, fb = pu.run_gpu(b)
    assert torch.equal(oa, ob[:70]) and torch.equal(fa[0], fb[0])


def test_gate_out_of_range_sets_device_status():
    from kda_chunked_prefill_gb300 import KDA_ERR_GATE_RANGE, KdaError
    inp = kin.make_inputs([80], 1, seed=12)
    inp["g"][40, 0, 3] = 0.5
    with pytest.raises(KdaError) as ei:
        pu.run_gpu(inp)
    assert ei.value.code == KDA_ERR_GATE_RANGE


def test_bad_cu_seqlens_sets_device_status_and_skips():
    from kda_chunked_prefill_gb300 import KDA_ERR_BAD_SEQLENS, KdaError
    inp = kin.make_inputs([40, 40], 1, seed=13)
    inp["cu_seqlens"] = torch.tensor([0, 60, 50], dtype=torch.int32)  # decreasing, ends short
    with pytest.raises(KdaError) as ei:
        pu.run_gpu(inp)
    assert ei.value.code == KDA_ERR_BAD_SEQLENS


def test_host_rejects_bad_arguments_without_launch():
    from kda_chunked_prefill_gb300 import KDA_ERR_INVALID_ARG, KdaError, kda_chunk_fwd
    inp = kin.make_inputs([10], 1, seed=14)
    d = pu.to_device(inp)
    o = torch.empty(d["v"].shape, dtype=torch.float32, device=d["v"].device)
    with pytest.raises(KdaError) as ei:
        kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], None, 0.1, -20.0, o, None)
    assert ei.value.code == KDA_ERR_INVALID_ARG


def test_nonblocking_on_side_stream():
    inp = kin.make_inputs([300], 2, seed=15, state_std=0.02)
    o_ref, f_ref = pu.run_gpu(inp)
    from kda_chunked_prefill_gb300 import chunk_fwd
    d = pu.to_device(inp)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, f = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                         scale=inp["scale"], stream=s)
    s.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(f, f_ref)


def test_value_beyond_fp16_operand_range_sets_device_status():
    from kda_chunked_prefill_gb300 import KDA_ERR_VALUE_RANGE, KdaError
    inp = kin.make_inputs([50], 1, seed=16)
    inp["v"][20, 0, 5] = 1.0e6
    inp["beta"][20, 0] = 1.0
    with pytest.raises(KdaError) as ei:
        pu.run_gpu(inp)
    assert ei.value.code == KDA_ERR_VALUE_RANGE


def test_inverse_beyond_fp16_range_sets_device_status():
    # three equal long keys with beta = 1 and g = 0: L has entries a = |k|^2 = 900 (inside the fp16 range)
    # while T = (I + L)^-1 has a^2 - a ~ 8e5 in row 2, column 0, beyond it
    from kda_chunked_prefill_gb300 import KDA_ERR_VALUE_RANGE, KdaError
    inp = kin.make_inputs([50], 1, seed=17)
    inp["k"][0:3, 0, :] = (30.0 / 128 ** 0.5)
    inp["g"][0:3, 0, :] = 0.0
    inp["beta"][0:3, 0] = 1.0
    with pytest.raises(KdaError) as ei:
        pu.run_gpu(inp)
    assert ei.value.code == KDA_ERR_VALUE_RANGE
