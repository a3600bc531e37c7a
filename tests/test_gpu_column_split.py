"""Consumers as CTA pairs, each CTA taking half of a chain's 128 value
columns, against the oracle. Column j of v_new, o and the state depends on
column j of the state alone (report "在 TPU 上加速 Kimi K3 KDA", §6.2: the
recurrence v_new = u - w S, o = q_hat S + Aqk v_new, S <- Diag(e^G) S + kg^T
v_new), so the halves run without exchanging anything. A launch with few
chains picks the split itself; the debug flags force either layout here.
(§13 of the same report: the token recurrence is the reference.)
"""
import numpy as np
import pytest

import kda_chunked_prefill_gb300 as kda
from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu

CASES = [
    ([256], 2, None),                   # one chain of four chunks
    ([130, 64, 210, 1], 4, 0.02),       # ragged tails, a one-token sequence, initial states
    ([2048] * 2, 16, None),             # 32 chains: 64 consumer CTAs when split
    ([700, 333, 1024], 8, 0.02),        # unequal lengths, scheduled by table
    (None, 2, 0.02),                    # 12 lognormal lengths
]


@pytest.mark.parametrize("flags", [kda.KDA_DEBUG_SPLIT_COLUMNS, kda.KDA_DEBUG_WHOLE_COLUMNS],
                         ids=["split", "whole"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_column_layout_matches_the_oracle(flags, case):
    seqlens, H, s0 = CASES[case]
    if seqlens is None:
        seqlens = kin._lognormal_lengths(np.random.default_rng(13), 12)
    inp = kin.make_inputs(seqlens, H, seed=60 + case, state_std=s0)
    o, fs = pu.run_gpu(inp, debug_flags=flags)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(o.cpu().numpy(), ref_o, f"o (flags {flags})")
    pu.assert_parity(fs.cpu().numpy(), ref_s, f"final_state (flags {flags})")


def test_split_layout_is_bitwise_deterministic():
    inp = kin.make_inputs([900, 77, 1500], 4, seed=66, state_std=0.02)
    o1, f1 = pu.run_gpu(inp, debug_flags=kda.KDA_DEBUG_SPLIT_COLUMNS)
    o2, f2 = pu.run_gpu(inp, debug_flags=kda.KDA_DEBUG_SPLIT_COLUMNS)
    assert bool((o1 == o2).all()) and bool((f1 == f2).all())
