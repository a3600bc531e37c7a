"""Both placements of the WY product X = T [beta v | beta k e^G] against the
oracle: in the producer CTAs (they send u and w) and in the consumer CTAs
(they receive T, beta v and beta k e^G and form v_new = T (beta v - beta k e^G S)
on the tensor cores). A launch picks one from its schedule; the debug flags
force each, so that both are checked on every shape here, whichever the
launch would pick.
(Report "在 TPU 上加速 Kimi K3 KDA", §4: the WY representation u = T beta v,
w = T beta k e^G; §13: the token recurrence is the reference.)
"""
import pytest

import kda_chunked_prefill_gb300 as kda
from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu

CASES = [
    ([256], 2, None),                  # one chain of four chunks
    ([130, 64, 210, 1], 4, 0.02),      # ragged tails, a one-token sequence, initial states
    ([2048] * 4, 16, None),            # the equal-length batch (64 chains of 32 chunks)
    (None, 16, 0.02),                  # 12 lognormal lengths (unequal chains, scheduled by table)
]


@pytest.mark.parametrize("flags", [kda.KDA_DEBUG_WY_PRODUCER, kda.KDA_DEBUG_WY_CONSUMER],
                         ids=["producer", "consumer"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_wy_placement_matches_the_oracle(flags, case):
    seqlens, H, s0 = CASES[case]
    if seqlens is None:
        import numpy as np
        seqlens = kin._lognormal_lengths(np.random.default_rng(11), 12)
    inp = kin.make_inputs(seqlens, H, seed=40 + case, state_std=s0)
    o, fs = pu.run_gpu(inp, debug_flags=flags)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(o.cpu().numpy(), ref_o, f"o (flags {flags})")
    pu.assert_parity(fs.cpu().numpy(), ref_s, f"final_state (flags {flags})")



def test_plan_on_this_device():
    # num_sms = 0 asks the current device; on it, the plan is the one for its SM count
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for shape in ((4, 8192, 16), (1, 16384, 96), (16, 12091, 16), (1, 65536, 4)):
        assert kda.chunk_fwd_plan(*shape) == kda.chunk_fwd_plan(*shape, num_sms=sms)
