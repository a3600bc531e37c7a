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


def assert_parity_by_head_groups(inp: dict, o, fs, group: int = 16):
    """The parity bar over the whole o and final_state tensors, with the oracle
    run on groups of heads at a time (chains are independent) so that its fp64
    copies stay small: the error norms, the maximum and the reference RMS are
    accumulated over the groups, then judged as for the whole tensors."""
    H = inp["q"].shape[1]
    acc = {"o": [0.0, 0.0, 0.0, 0, True], "final_state": [0.0, 0.0, 0.0, 0, True]}  # sum d^2, sum r^2, max|d|, n, finite
    o = o.float().cpu()
    fs = fs.cpu()
    for h0 in range(0, H, group):
        heads = list(range(h0, min(H, h0 + group)))
        ref_o, ref_s = run_oracle(inp, heads=heads)
        for name, got, ref in (("o", o[:, heads].numpy(), ref_o), ("final_state", fs[:, heads].numpy(), ref_s)):
            got = np.asarray(got, dtype=np.float64)
            d = got - ref
            a = acc[name]
            a[0] += float(np.sum(d * d))
            a[1] += float(np.sum(ref * ref))
            a[2] = max(a[2], float(np.max(np.abs(d))) if d.size else 0.0)
            a[3] += ref.size
            a[4] = a[4] and bool(np.all(np.isfinite(got)))
    out = {}
    for name, (sd, sr, mx, n, fin) in acc.items():
        assert fin, f"{name}: non-finite values"
        rms = (sr / n) ** 0.5 if n else 0.0
        rel = (sd ** 0.5) / (sr ** 0.5) if sr > 0 else sd ** 0.5
        e = {"rel_l2": rel, "max_abs": mx, "rms_ref": rms, "finite": fin}
        if rms == 0.0:
            assert mx <= 1e-6, f"{name}: {e}"
        else:
            assert rel <= REL_L2, f"{name}: rel L2 {rel:.3e} > {REL_L2} ({e})"
            assert mx <= MAX_ABS_RMS * rms, f"{name}: max abs {mx:.3e} > {MAX_ABS_RMS} * RMS {rms:.3e} ({e})"
        out[name] = e
    return out


def to_device(inp: dict, device="cuda"):
    out = {}
    for key in ("q", "k", "v", "g", "beta", "cu_seqlens", "initial_state"):
        x = inp[key]
        out[key] = None if x is None else x.to(device).contiguous()
    return out


GUARD = 4096  # fp32 elements of NaN kept before and after each output buffer


def _guarded(shape, device):
    """A NaN-filled buffer with GUARD elements on both sides of a contiguous
    view of `shape` (16-byte aligned): the view is the output, the bands are
    canaries that no kernel may write."""
    n = int(np.prod(shape))
    flat = torch.full((n + 2 * GUARD,), float("nan"), dtype=torch.float32, device=device)
    return flat, flat[GUARD:GUARD + n].view(*shape)


def check_guard(flat, what: str):
    assert bool(torch.isnan(flat[:GUARD]).all()) and bool(torch.isnan(flat[-GUARD:]).all()), \
        f"{what}: a kernel wrote into the guard band around the output"


def run_gpu(inp: dict, device="cuda", check=True, output_final_state=True, debug_flags: int = 0):
    """kda_chunk_fwd (kda_chunk_fwd_debug with nonzero ``debug_flags``) through
    the C ABI into outputs surrounded by NaN guard bands, which are checked to
    be untouched afterwards."""
    from kda_chunked_prefill_gb300 import _lib
    d = to_device(inp, device)
    T, H, D = inp["q"].shape
    N = inp["cu_seqlens"].shape[0] - 1
    o_flat, o = _guarded((T, H, D), device)
    fs_flat, fs = _guarded((N, H, D, D), device) if output_final_state else (None, None)
    status = torch.zeros(1, dtype=torch.int32, device=device) if check else None
    _lib.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                       inp["scale"], inp["lower_bound"], o, fs, status, debug_flags=debug_flags)
    torch.cuda.synchronize()
    if check:
        code = int(status.item())
        if code != _lib.KDA_OK:
            raise _lib.KdaError(code, "kda_chunk_fwd (device)")
    check_guard(o_flat, "o")
    if fs_flat is not None:
        check_guard(fs_flat, "final_state")
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
