"""GPU parity of kda_chunk_fwd_raw_gates: the raw gate and beta projections
activated inside the kernel (g = lower_bound * sigmoid(e^A_log (g_raw +
dt_bias)), beta = sigmoid(beta_raw): the library's stated reading of the
gate activation the TPU report fuses in §6.1) against the fp64 oracle run on
the same projections activated in fp64, and against the activated-input entry
point fed the same activation computed on the host."""
import numpy as np
import pytest
import torch

from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu


def raw_case(lens, H, seed, with_params):
    """Inputs whose g and beta are raw projections: g_raw ~ N(0, 1) per channel,
    beta_raw ~ N(0, 1), with (optionally) per-head A_log and dt_bias."""
    inp = kin.make_inputs(lens, H, seed=seed, state_std=0.02)
    rng = np.random.default_rng(seed + 1)
    T = inp["q"].shape[0]
    inp["g"] = torch.from_numpy(rng.normal(size=(T, H, 128)).astype(np.float32))
    inp["beta"] = torch.from_numpy(rng.normal(size=(T, H)).astype(np.float32))
    A = torch.from_numpy(rng.normal(scale=0.5, size=(H,)).astype(np.float32)) if with_params else None
    dt = torch.from_numpy(rng.normal(scale=0.5, size=(H, 128)).astype(np.float32)) if with_params else None
    return inp, A, dt


def activated_for_oracle(inp, A, dt):
    from oracle import gates
    out = dict(inp)
    out["g"] = torch.from_numpy(gates.activate_gate(inp["g"].double().numpy(), inp["lower_bound"],
                                                    None if A is None else A.double().numpy(),
                                                    None if dt is None else dt.double().numpy()))
    out["beta"] = torch.from_numpy(gates.activate_beta(inp["beta"].double().numpy()))
    return out


@pytest.mark.parametrize("lens,H,with_params", [
    ([130, 64, 210], 4, True),
    ([0, 70, 1, 5, 129], 2, False),
    ([300, 190], 3, True),
])
def test_raw_gates_match_oracle(lens, H, with_params):
    from kda_chunked_prefill_gb300 import chunk_fwd
    inp, A, dt = raw_case(lens, H, 400 + sum(lens), with_params)
    dev = torch.device("cuda")
    d = {k2: (v2.to(dev) if torch.is_tensor(v2) else v2) for k2, v2 in inp.items()}
    o, fs = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                      scale=inp["scale"], lower_bound=inp["lower_bound"], check=True, raw_gates=True,
                      A_log=None if A is None else A.to(dev), dt_bias=None if dt is None else dt.to(dev))
    ref_o, ref_s = pu.run_oracle(activated_for_oracle(inp, A, dt))
    pu.assert_parity(o.float().cpu().numpy(), ref_o, "o")
    pu.assert_parity(fs.cpu().numpy(), ref_s, "final_state")


def test_raw_gates_agree_with_host_activation():
    """The in-kernel activation and an fp32 host activation feed the same
    chunked forward: the outputs agree far inside the parity bar."""
    from kda_chunked_prefill_gb300 import chunk_fwd
    inp, A, dt = raw_case([1000, 333, 64], 4, 77, True)
    dev = torch.device("cuda")
    d = {k2: (v2.to(dev) if torch.is_tensor(v2) else v2) for k2, v2 in inp.items()}
    Ad, dtd = A.to(dev), dt.to(dev)
    o_raw, s_raw = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                             scale=inp["scale"], lower_bound=inp["lower_bound"], check=True, raw_gates=True,
                             A_log=Ad, dt_bias=dtd)
    g_act = inp["lower_bound"] * torch.sigmoid(torch.exp(Ad)[None, :, None] * (d["g"] + dtd[None]))
    b_act = torch.sigmoid(d["beta"])
    o_act, s_act = chunk_fwd(d["q"], d["k"], d["v"], g_act.contiguous(), b_act.contiguous(), d["cu_seqlens"],
                             d["initial_state"], scale=inp["scale"], lower_bound=inp["lower_bound"], check=True)
    for a, b in ((o_raw, o_act), (s_raw, s_act)):
        rel = (torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b)).item()
        assert rel < 1e-4, rel
