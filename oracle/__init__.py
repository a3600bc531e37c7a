"""KDA oracle — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path
(``kda_chunked_prefill_gb300``) and imports nothing from it; the two meet
only in the seeded input generators, which hold none of the method's
arithmetic.

Contents
--------
``kda_recurrence``  the oracle proper: the token-by-token fp64 recurrence of
                    Kimi Delta Attention, compiled from ``kda_oracle.c`` and
                    run on host threads over (sequence, head) chains.
``gates``           the gate and beta activations of the raw-gate entry point
                    (a stated reading: the pages name the gate activation
                    without defining it).
``norm``            the gated RMSNorm of the output for the fused-norm entry
                    point (a stated reading: the pages name the operation
                    without writing it out).
``chunked``         a second, independent fp64 formulation — the chunked
                    algebra of the TPU report (§4 strip GEMMs with sub-block
                    midpoints, the Neumann factor chain, the WY form and the
                    §6.2 chunk recurrence) — used only to pin the recurrence.

Every public function cites the passage it follows. The pins live in
``tests/test_oracle_pins.py`` (run with ``-m "not gpu"``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``liboracle.so`` beside it (gcc, -O2, no
    fast-math: the oracle keeps IEEE fp64 semantics)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64),
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, dp, ctypes.c_double, dp, dp,
                                           ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            lib.kda_oracle_fwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x, shape=None):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if a is not None else None


def kda_recurrence(q, k, v, g, beta, cu_seqlens, initial_state=None, scale=None,
                   num_threads: int = 0, return_threads: bool = False):
    """Token-by-token fp64 KDA forward over varlen-packed sequences.

    Follows "在 TPU 上加速 Kimi K3 KDA" (junyi.dev tpu-kda report) §1–§2 for
    the recurrence and §13 for its use as the naive reference:
    ``S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T``,
    ``o_t = scale * S_t^T q_t``; the state restarts per sequence (§6.5).

    Arguments are array-likes convertible to float64 (callers upcast bf16
    inputs exactly before the call). Shapes: q, k, g ``[T,H,K]``; v ``[T,H,V]``;
    beta ``[T,H]``; cu_seqlens ``[N+1]``; initial_state ``[N,H,K,V]`` or None.
    Returns ``(o [T,H,V], final_state [N,H,K,V])`` in float64 (and the thread
    count used when ``return_threads``).
    """
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    q = _f64(q)
    T, H, K = q.shape
    v = _f64(v)
    V = v.shape[2]
    k = _f64(k, (T, H, K))
    g = _f64(g, (T, H, K))
    beta = _f64(beta, (T, H))
    if v.shape != (T, H, V):
        raise ValueError("v must be [T,H,V]")
    if N < 0 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, be nondecreasing and end at T")
    s0 = None if initial_state is None else _f64(initial_state, (N, H, K, V))
    if scale is None:
        scale = K ** -0.5
    o = np.zeros((T, H, V), dtype=np.float64)
    sT = np.zeros((N, H, K, V), dtype=np.float64)
    used = ctypes.c_int(0)
    rc = _load().kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                N, H, K, V, _ptr(s0), float(scale), _ptr(o), _ptr(sT),
                                int(num_threads), ctypes.byref(used))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_fwd failed with code {rc}")
    if return_threads:
        return o, sT, used.value
    return o, sT
