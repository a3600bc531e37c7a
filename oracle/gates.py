"""Gate and beta activations — TEST INFRASTRUCTURE ONLY (part of the oracle).

"在 TPU 上加速 Kimi K3 KDA" §6.1 moves ``activate_gate(g, A_log[head],
dt_bias[head])`` into the intra-chunk kernel, ahead of the chunk prefix sum,
and the Kimi K3 PP16 prefill notes' flag table fuses the beta sigmoid; neither
page defines the gate activation. The reading restated here (and in the
library's header) is

    g    = lower_bound * sigmoid(exp(A_log[h]) * (g_raw + dt_bias[h, c]))
    beta = sigmoid(beta_raw)

in fp64, which keeps lower_bound <= g <= 0 and, with A_log = dt_bias = 0, is
the ``lower_bound * sigmoid(x)`` form the synthetic workloads draw g from.
Parity of this reading is unpinned by the pages (they print no value of it);
``tests/test_oracle_pins.py`` pins the restatement to the closed forms of the
logistic function.
"""
from __future__ import annotations

import numpy as np


def sigmoid(x):
    """The logistic function 1 / (1 + e^-x) in fp64, evaluated without overflow."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def activate_gate(g_raw, lower_bound: float, A_log=None, dt_bias=None):
    """g [T, H, K] from the raw gate projection g_raw [T, H, K] (see the module
    docstring for the reading); A_log [H] and dt_bias [H, K] default to zeros."""
    g_raw = np.asarray(g_raw, dtype=np.float64)
    T, H, K = g_raw.shape
    a = np.zeros(H) if A_log is None else np.asarray(A_log, dtype=np.float64).reshape(H)
    b = np.zeros((H, K)) if dt_bias is None else np.asarray(dt_bias, dtype=np.float64).reshape(H, K)
    return float(lower_bound) * sigmoid(np.exp(a)[None, :, None] * (g_raw + b[None]))


def activate_beta(beta_raw):
    """beta [T, H] = sigmoid(beta_raw)."""
    return sigmoid(beta_raw)
