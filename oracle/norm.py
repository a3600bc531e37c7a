"""Gated RMSNorm of the attention output — TEST INFRASTRUCTURE ONLY (part of the oracle).

The Kimi K3 PP16 prefill deployment notes (KDA flag table, the strided o-norm
entry) fuse ``FusedRMSNormGated`` on the KDA output into one kernel with the
copy its reshape forced; the page names the operation without writing it out.
The reading restated here (and in the library's header) is, per token t and
head h, over the head's value channels c = 0..V-1:

    y[t, h, c] = o[t, h, c] / sqrt(mean_c(o[t, h, :]^2) + eps) * weight[c] * sigmoid(gate[t, h, c])

in fp64: an RMS normalisation over the value channels of one head, a learned
per-channel weight shared by the heads, and a sigmoid output gate (the same
logistic function as the page's fused beta activation). Parity of this reading
is unpinned by the pages (they print no value of it); ``tests/test_oracle_pins.py``
pins the restatement to the closed forms of the RMS and logistic functions.
"""
from __future__ import annotations

import numpy as np

from .gates import sigmoid


def gated_rmsnorm(o, gate, weight, eps: float):
    """y [T, H, V] from o [T, H, V], gate [T, H, V] and weight [V] (see the
    module docstring for the reading); eps > 0 keeps an all-zero row finite."""
    o = np.asarray(o, dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64).reshape(-1)
    if o.shape != gate.shape or o.shape[-1] != weight.shape[0]:
        raise ValueError(f"shapes: o {o.shape}, gate {gate.shape}, weight {weight.shape}")
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return o / np.sqrt(ms + float(eps)) * weight * sigmoid(gate)
