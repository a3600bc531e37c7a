"""Failure detection, tested without a GPU fault.

Every wait inside the kernel is bounded. With KDA_DEBUG_WITHHOLD_READY the
producers compute their chunks but never publish them, so the consumers wait
on flags that nothing sets; the waits run out (after 2^14 polls in this mode),
the device reports KDA_ERR_TIMEOUT in the status word, every CTA leaves, and
the same context then runs a normal call that meets the parity bar.
"""
import time

import pytest
import torch

import kda_chunked_prefill_gb300 as kda
from kda_chunked_prefill_gb300 import inputs as kin

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seqlens,H", [([256], 2), ([130, 64, 210], 4), ([2048] * 4, 16)])
def test_withheld_chunks_time_out_and_the_context_stays_usable(seqlens, H):
    inp = kin.make_inputs(seqlens, H, seed=7, state_std=0.02)
    d = pu.to_device(inp)
    T, _, D = inp["q"].shape
    N = len(seqlens)
    o = torch.empty(T, H, D, dtype=torch.float32, device="cuda")
    fs = torch.empty(N, H, D, D, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                      inp["scale"], inp["lower_bound"], o, fs, status,
                      debug_flags=kda.KDA_DEBUG_WITHHOLD_READY)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(status.item()) == kda.KDA_ERR_TIMEOUT
    assert elapsed < 20.0, f"the timed-out launch took {elapsed:.1f} s"

    # the context is intact: a normal call on the same inputs meets the bar
    o2, fs2 = pu.run_gpu(inp)
    ref_o, ref_s = pu.run_oracle(inp)
    pu.assert_parity(o2.cpu().numpy(), ref_o, "o after a timed-out launch")
    pu.assert_parity(fs2.cpu().numpy(), ref_s, "final_state after a timed-out launch")
