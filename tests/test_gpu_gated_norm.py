"""GPU parity of kda_chunk_fwd_gated_norm: the gated RMSNorm of the output
fused into the kernel's output store (the strided o-norm entry of the Kimi K3
PP16 prefill notes' flag table, read as o / sqrt(mean(o^2) + eps) * weight *
sigmoid(gate) over one head's value channels) against the fp64 oracle (the
token recurrence, then the restated norm), and against the plain entry point's
output normalised by the oracle's norm."""
import numpy as np
import pytest
import torch

from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu


def _run(inp, nrm, norm=True):
    from kda_chunked_prefill_gb300 import chunk_fwd
    dev = torch.device("cuda")
    d = pu.to_device(inp)
    kw = dict(norm_gate=nrm["gate"].to(dev), norm_weight=nrm["weight"].to(dev), norm_eps=nrm["eps"]) if norm else {}
    o, fs = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                      scale=inp["scale"], lower_bound=inp["lower_bound"], check=True, **kw)
    torch.cuda.synchronize()
    return o.cpu().numpy(), fs.cpu().numpy()


def _norm_ref(o, nrm):
    from oracle import norm
    return norm.gated_rmsnorm(o, kin.to_f64(nrm["gate"]), kin.to_f64(nrm["weight"]), nrm["eps"])


CASES = {
    "page_lens_130_64_210": ([130, 64, 210], 4, 0.02),
    "empty_and_ragged": ([0, 70, 0, 1, 64, 0, 129], 2, 0.02),
    "single_token": ([1], 3, None),
    "multi_chunk_300_190": ([300, 190], 3, 0.02),
}


@pytest.mark.parametrize("name", list(CASES))
def test_gated_norm_matches_oracle(name):
    lens, H, s0 = CASES[name]
    inp = kin.make_inputs(lens, H, seed=500 + sum(lens), state_std=s0)
    nrm = kin.make_norm_inputs(sum(lens), H, seed=600 + sum(lens))
    y, fs = _run(inp, nrm)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(y, _norm_ref(ref_o, nrm), "normed o")
    pu.assert_parity(fs, ref_s, "final_state")


def test_gated_norm_headline_all_heads():
    """4 x 2048 tokens, H = 16, in the launch configuration the benchmark times."""
    inp = kin.make_workload(kin.workloads()["headline_4x2048_H16"])
    nrm = kin.make_norm_inputs(inp["q"].shape[0], inp["q"].shape[1], seed=7)
    y, fs = _run(inp, nrm)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(y, _norm_ref(ref_o, nrm), "normed o")
    pu.assert_parity(fs, ref_s, "final_state")


def test_gated_norm_is_the_plain_output_normalised():
    """The fused call equals the plain call's output put through the oracle's
    norm (the pre-norm rows are the same fp32 values; the kernel's sigmoid runs
    on the packed fp16 hardware tanh, about 1e-3 absolute error), far inside the parity
    bar, and leaves the final state bit-identical."""
    inp = kin.make_inputs([1000, 333, 64], 4, seed=91, state_std=0.02)
    nrm = kin.make_norm_inputs(1397, 4, seed=92)
    y, fs = _run(inp, nrm)
    o_plain, fs_plain = _run(inp, nrm, norm=False)
    ref = _norm_ref(o_plain, nrm)
    e = pu.errors(y, ref)
    assert e["rel_l2"] < 2e-3 and e["max_abs"] < 1e-2 * e["rms_ref"], e
    assert np.array_equal(fs, fs_plain)
