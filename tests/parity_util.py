"""Helpers for the GPU-vs-oracle parity tests (test code only).

Tolerance (the stated parity bar): for each of o and final_state separately,
relative L2 error <= 1e-2 and max-abs error <= 3e-2 * RMS(reference).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kda_chunked_prefill_gb300 import inputs as kin

REL_L2 = 1e-2
MAX_ABS_RMS = 3e-2


def errors(got: np.ndarray, ref: np.ndarray) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    nref = float(np.linalg.norm(ref))
    return {
        "rel_l2": float(np.linalg.norm(diff)) / nref if nref > 0 else float(np.linalg.norm(diff)),
        "max_abs": float(np.max(np.abs(diff))) if diff.size else 0.0,
        "rms_ref": rms,
        "finite": bool(np.all(np.isfinite(got))),
    }


def assert_parity(got, ref, what: str):
    e = errors(got, ref)
    assert e["finite"], f"{what}: non-finite values"
    if e["rms_ref"] == 0.0:
        assert e["max_abs"] <= 1e-6, f"{what}: {e}"
        return e
    assert e["rel_l2"] <= REL_L2, f"{what}: rel L2 {e['rel_l2']:.3e} > {REL_L2} ({e})"
    assert e["max_abs"] <= MAX_ABS_RMS * e["rms_ref"], \
        f"{what}: max abs {e['max_abs']:.3e} > {MAX_ABS_RMS} * RMS {e['rms_ref']:.3e} ({e})"
    return e


def to_device(inp: dict, device="cuda"):
    out = {}
    for key in ("q", "k", "v", "g", "beta", "cu_seqlens", "initial_state"):
        x = inp[key]
        out[key] = None if x is None else x.to(device).contiguous()
    return out


def run_gpu(inp: dict, device="cuda", check=True, output_final_state=True):
    from kda_chunked_prefill_gb300 import chunk_fwd
    d = to_device(inp, device)
    o, fs = chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                      scale=inp["scale"], lower_bound=inp["lower_bound"],
                      output_final_state=output_final_state, check=check)
    torch.cuda.synchronize()
    return o, fs


def run_oracle(inp: dict, heads=None, num_threads: int = 0):
    """Oracle on all heads, or on the given head subset (chains are independent)."""
    sel = slice(None) if heads is None else list(heads)
    s0 = inp["initial_state"]
    return oracle.kda_recurrence(
        kin.to_f64(inp["q"][:, sel]), kin.to_f64(inp["k"][:, sel]), kin.to_f64(inp["v"][:, sel]),
        kin.to_f64(inp["g"][:, sel]), kin.to_f64(inp["beta"][:, sel]),
        inp["cu_seqlens"].numpy().astype(np.int64),
        None if s0 is None else kin.to_f64(s0[:, sel]), inp["scale"], num_threads=num_threads)
