"""ctypes binding of ``libkda.so`` (C ABI in ``include/kda.h``).

Argument marshalling only: tensors are checked for dtype, device, shape and
contiguity and turned into raw pointers; every step of the computation runs
in the library's CUDA kernels. There is no fallback: if the library is
missing or fails to load, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_GATE_RANGE = 4
KDA_ERR_BAD_SEQLENS = 5
KDA_ERR_TIMEOUT = 6
KDA_ERR_VALUE_RANGE = 7
KDA_ERR_SCRATCH_TOO_SMALL = 8
KDA_ERR_BOUNDS = 9
KDA_DEBUG_WITHHOLD_READY = 1
KDA_DEBUG_WY_PRODUCER = 2  # the producer CTAs form the WY product
KDA_DEBUG_WY_CONSUMER = 4  # the consumer CTAs form it
KDA_DEBUG_SPLIT_COLUMNS = 8  # a chain's value columns over two consumer CTAs
KDA_DEBUG_WHOLE_COLUMNS = 16  # one consumer CTA per chain's columns

HEAD_DIM = 128
EXPORTED = ("kda_chunk_fwd", "kda_chunk_fwd_workspace_size", "kda_chunk_fwd_static_scratch",
            "kda_chunk_fwd_debug", "kda_chunk_fwd_raw_gates", "kda_chunk_fwd_gated_norm", "kda_chunk_fwd_split",
            "kda_chunk_fwd_split_plan", "kda_chunk_fwd_split_workspace_size", "kda_chunk_fwd_host", "kda_chunk_fwd_plan",
            "kda_chunk_fwd_host_buffer_size", "kda_decode_fwd",
            "kda_chunk_fwd_launches",
            "kda_status_string", "kda_version")
DECODE_MAX_TOKENS = 64

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} (code {code})")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load ``libkda.so``; raises ``OSError`` if it is absent (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"{path} not found: build it with kda_chunked_prefill_gb300.build.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.kda_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, f32, f32,
                                      vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.kda_chunk_fwd.restype = ctypes.c_int
        lib.kda_chunk_fwd_debug.argtypes = lib.kda_chunk_fwd.argtypes + [ctypes.c_uint32]
        lib.kda_chunk_fwd_debug.restype = ctypes.c_int
        lib.kda_chunk_fwd_raw_gates.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, f32, f32,
                                                vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.kda_chunk_fwd_raw_gates.restype = ctypes.c_int
        lib.kda_chunk_fwd_gated_norm.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, f32, f32,
                                                 vp, vp, f32, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.kda_chunk_fwd_gated_norm.restype = ctypes.c_int
        lib.kda_chunk_fwd_split.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, f32, f32, i32,
                                            vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.kda_chunk_fwd_split.restype = ctypes.c_int
        lib.kda_chunk_fwd_split_plan.argtypes = [vp, i32, i32, i32]
        lib.kda_chunk_fwd_split_plan.restype = ctypes.c_int32
        lib.kda_chunk_fwd_plan.argtypes = [i32, i64, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                           ctypes.POINTER(i32)]
        lib.kda_chunk_fwd_plan.restype = ctypes.c_int
        lib.kda_chunk_fwd_split_workspace_size.argtypes = [vp, i32, i32, i32]
        lib.kda_chunk_fwd_split_workspace_size.restype = ctypes.c_size_t
        lib.kda_chunk_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, f32, f32, vp, vp, vp,
                                           vp, ctypes.c_size_t, i32, vp, vp, vp]
        lib.kda_chunk_fwd_host.restype = ctypes.c_int
        lib.kda_chunk_fwd_host_buffer_size.argtypes = [vp, i32, i32, i32, i32, i32]
        lib.kda_chunk_fwd_host_buffer_size.restype = ctypes.c_size_t
        lib.kda_decode_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, f32, f32, vp, vp, vp, vp]
        lib.kda_decode_fwd.restype = ctypes.c_int
        lib.kda_chunk_fwd_workspace_size.argtypes = [i32, i32]
        lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_size_t
        lib.kda_chunk_fwd_launches.argtypes = [i32, i64, i32]
        lib.kda_chunk_fwd_launches.restype = i32
        lib.kda_status_string.argtypes = [i32]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_version.argtypes = []
        lib.kda_version.restype = i32
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().kda_status_string(int(code)).decode()


def version() -> int:
    return int(load_library().kda_version())


def workspace_size(num_seqs: int, num_heads: int) -> int:
    """Workspace bytes ``kda_chunk_fwd`` needs on the current CUDA device."""
    return int(load_library().kda_chunk_fwd_workspace_size(int(num_seqs), int(num_heads)))


_ws_cache = {}


def workspace_for(num_seqs: int, num_heads: int, device) -> torch.Tensor:
    """A cached workspace buffer for calls on ``device``'s current stream.
    Calls that may overlap on the GPU need buffers of their own."""
    need = workspace_size(num_seqs, num_heads)
    key = torch.device(device)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < need:
        buf = torch.empty(max(need, 1), dtype=torch.uint8, device=key)
        _ws_cache[key] = buf
    return buf


def chunk_fwd_launches(num_seqs: int, total_tokens: int, num_heads: int) -> int:
    return int(load_library().kda_chunk_fwd_launches(int(num_seqs), int(total_tokens), int(num_heads)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def kda_chunk_fwd(q, k, v, g, beta, cu_seqlens, initial_state, scale: float, lower_bound: float,
                  o, final_state, status=None, stream=None, workspace=None, debug_flags: int = 0,
                  raw_gates: bool = False, A_log=None, dt_bias=None, norm_gate=None, norm_weight=None,
                  norm_eps: float = 1e-5) -> int:
    """Call the C entry point ``kda_chunk_fwd`` with caller-allocated outputs.

    q, k, v: bf16 [T,H,128]; o: fp32 [T,H,128]; g: fp32 [T,H,128]; beta: fp32 [T,H];
    cu_seqlens: int32 [N+1]; initial_state / final_state: fp32 [N,H,128,128]
    or None; status: int32 [1] or None; workspace: uint8 tensor of at least
    ``workspace_size(N, H)`` bytes (default: a cached per-device buffer). All on
    one CUDA device. ``stream`` is a ``torch.cuda.Stream`` (default: the current
    stream). Raises ``KdaError`` on a host-side error; returns ``KDA_OK`` once
    the work is queued. A nonzero ``debug_flags`` calls ``kda_chunk_fwd_debug``
    (failure-detection testing; see include/kda.h). ``raw_gates=True`` calls
    ``kda_chunk_fwd_raw_gates``: ``g`` and ``beta`` are then the raw gate and
    beta projections, activated inside the kernel with the optional per-head
    ``A_log`` (fp32 [H]) and ``dt_bias`` (fp32 [H,128]). Given ``norm_gate``
    (bf16 [T,H,128]) and ``norm_weight`` (fp32 [128]), ``kda_chunk_fwd_gated_norm``
    writes ``o`` as the gated RMSNorm of the output (``norm_eps`` inside the root).
    """
    T, H, D = q.shape
    N = cu_seqlens.shape[0] - 1
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    _check(q, "q", torch.bfloat16, (T, H, D), dev)
    _check(k, "k", torch.bfloat16, (T, H, D), dev)
    _check(v, "v", torch.bfloat16, (T, H, v.shape[2]), dev)
    _check(g, "g", torch.float32, (T, H, D), dev)
    _check(beta, "beta", torch.float32, (T, H), dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    _check(o, "o", torch.float32, tuple(v.shape), dev)
    if initial_state is not None:
        _check(initial_state, "initial_state", torch.float32, (N, H, D, v.shape[2]), dev)
    if final_state is not None:
        _check(final_state, "final_state", torch.float32, (N, H, D, v.shape[2]), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    if not raw_gates and (A_log is not None or dt_bias is not None):
        raise ValueError("A_log and dt_bias apply only with raw_gates=True")
    if A_log is not None:
        _check(A_log, "A_log", torch.float32, (H,), dev)
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", torch.float32, (H, D), dev)
    norm = norm_gate is not None or norm_weight is not None
    if norm:
        if norm_gate is None or norm_weight is None:
            raise ValueError("norm_gate and norm_weight go together")
        _check(norm_gate, "norm_gate", torch.bfloat16, tuple(v.shape), dev)
        _check(norm_weight, "norm_weight", torch.float32, (v.shape[2],), dev)
        if raw_gates or debug_flags:
            raise ValueError("the gated norm combines with neither raw_gates nor debug_flags")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = workspace_for(N, H, dev)
    if workspace.device != dev or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, D, v.shape[2],
            _ptr(initial_state), float(scale), float(lower_bound), _ptr(o), _ptr(final_state),
            _ptr(status), _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    lib = load_library()
    if norm:
        rc = lib.kda_chunk_fwd_gated_norm(*args[:14], _ptr(norm_gate), _ptr(norm_weight), float(norm_eps), *args[14:])
        what = "kda_chunk_fwd_gated_norm"
    elif raw_gates:
        if debug_flags:
            raise ValueError("debug_flags and raw_gates cannot be combined")
        rc = lib.kda_chunk_fwd_raw_gates(*args[:5], _ptr(A_log), _ptr(dt_bias), *args[5:])
        what = "kda_chunk_fwd_raw_gates"
    else:
        rc = lib.kda_chunk_fwd_debug(*args, int(debug_flags)) if debug_flags else lib.kda_chunk_fwd(*args)
        what = "kda_chunk_fwd"
    if rc != KDA_OK:
        raise KdaError(rc, what)
    return rc


def chunk_fwd(q, k, v, g, beta, cu_seqlens, initial_state=None, scale: Optional[float] = None,
              lower_bound: float = -5.0, output_final_state: bool = True, check: bool = False,
              stream=None, raw_gates: bool = False, A_log=None, dt_bias=None, norm_gate=None,
              norm_weight=None, norm_eps: float = 1e-5):
    """Allocate ``o`` (and ``final_state``) and run ``kda_chunk_fwd``.

    Returns ``(o, final_state)``; ``final_state`` is None when not requested.
    With ``check=True`` the device status word is read back (a synchronising
    copy) and a device-detected error raises ``KdaError``. ``raw_gates``,
    ``A_log``, ``dt_bias`` and the gated-norm arguments are passed to
    ``kda_chunk_fwd``.
    """
    T, H, D = q.shape
    N = cu_seqlens.shape[0] - 1
    if scale is None:
        scale = D ** -0.5
    o = torch.empty((T, H, v.shape[2]), dtype=torch.float32, device=q.device)
    fs = (torch.empty((N, H, D, v.shape[2]), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    status = torch.zeros(1, dtype=torch.int32, device=q.device) if check else None
    kda_chunk_fwd(q, k, v, g, beta, cu_seqlens, initial_state, scale, lower_bound, o, fs, status, stream,
                  raw_gates=raw_gates, A_log=A_log, dt_bias=dt_bias, norm_gate=norm_gate,
                  norm_weight=norm_weight, norm_eps=norm_eps)
    if check:
        code = int(status.item())
        if code != KDA_OK:
            raise KdaError(code, "kda_chunk_fwd (device)")
    return o, fs


def _host_cu(cu_seqlens_host):
    cu = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).cpu().contiguous()
    return cu, ctypes.c_void_p(cu.data_ptr())


def split_plan(cu_seqlens_host, num_heads: int, num_sms: int = 0) -> int:
    """Segment length (in 64-token chunks) ``kda_chunk_fwd_split`` would pick
    for these sequence lengths (0: no split). ``num_sms`` 0 = the current device."""
    cu, ptr = _host_cu(cu_seqlens_host)
    return int(load_library().kda_chunk_fwd_split_plan(ptr, cu.numel() - 1, int(num_heads), int(num_sms)))


def chunk_fwd_plan(num_seqs: int, total_tokens: int, num_heads: int, num_sms: int = 0,
                   plain_device_o: bool = True) -> Tuple[int, bool, bool]:
    """``kda_chunk_fwd_plan``: (consumers, whether the consumers form the WY
    product, whether each consumer is two CTAs with half the value columns each)
    for a call of this shape. ``num_sms`` 0 = the current device."""
    c, w, sp = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    rc = load_library().kda_chunk_fwd_plan(int(num_seqs), int(total_tokens), int(num_heads), int(num_sms),
                                           1 if plain_device_o else 0, ctypes.byref(c), ctypes.byref(w),
                                           ctypes.byref(sp))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_plan")
    return int(c.value), bool(w.value), bool(sp.value)


def split_workspace_size(cu_seqlens_host, num_heads: int, segment_chunks: int = 0) -> int:
    cu, ptr = _host_cu(cu_seqlens_host)
    return int(load_library().kda_chunk_fwd_split_workspace_size(ptr, cu.numel() - 1, int(num_heads),
                                                                  int(segment_chunks)))


def kda_chunk_fwd_split(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, initial_state, scale: float,
                        lower_bound: float, o, final_state, status=None, stream=None, segment_chunks: int = 0,
                        workspace=None) -> int:
    """Call ``kda_chunk_fwd_split`` (the split-sequence scan; see include/kda.h).
    Arguments as ``kda_chunk_fwd`` plus ``cu_seqlens_host`` (the same offsets on
    the host: a CPU tensor, array or list) and ``segment_chunks`` (0: planned).
    ``workspace`` defaults to a fresh uint8 tensor of the needed size."""
    T, H, D = q.shape
    dev = q.device
    cu, cu_ptr = _host_cu(cu_seqlens_host)
    N = cu.numel() - 1
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    _check(q, "q", torch.bfloat16, (T, H, D), dev)
    _check(k, "k", torch.bfloat16, (T, H, D), dev)
    _check(v, "v", torch.bfloat16, (T, H, v.shape[2]), dev)
    _check(g, "g", torch.float32, (T, H, D), dev)
    _check(beta, "beta", torch.float32, (T, H), dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,), dev)
    _check(o, "o", torch.float32, tuple(v.shape), dev)
    for t, name in ((initial_state, "initial_state"), (final_state, "final_state")):
        if t is not None:
            _check(t, name, torch.float32, (N, H, D, v.shape[2]), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    lib = load_library()
    if workspace is None:
        nbytes = lib.kda_chunk_fwd_split_workspace_size(cu_ptr, N, H, int(segment_chunks))
        if nbytes == 0:
            raise KdaError(KDA_ERR_INVALID_ARG, "kda_chunk_fwd_split_workspace_size")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if workspace.device != dev or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = lib.kda_chunk_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), cu_ptr, N, T, H,
                                 D, v.shape[2], _ptr(initial_state), float(scale), float(lower_bound),
                                 int(segment_chunks), _ptr(o), _ptr(final_state), _ptr(status), _ptr(workspace),
                                 workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_split")
    return rc


def chunk_fwd_split(q, k, v, g, beta, cu_seqlens, cu_seqlens_host=None, initial_state=None,
                    scale: Optional[float] = None, lower_bound: float = -5.0, output_final_state: bool = True,
                    check: bool = False, stream=None, segment_chunks: int = 0):
    """Allocate ``o`` (and ``final_state``) and run ``kda_chunk_fwd_split``.
    ``cu_seqlens_host`` defaults to a copy of ``cu_seqlens`` (a synchronising
    device-to-host read)."""
    T, H, D = q.shape
    if cu_seqlens_host is None:
        cu_seqlens_host = cu_seqlens.cpu()
    N = cu_seqlens.shape[0] - 1
    if scale is None:
        scale = D ** -0.5
    o = torch.empty((T, H, v.shape[2]), dtype=torch.float32, device=q.device)
    fs = (torch.empty((N, H, D, v.shape[2]), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    status = torch.zeros(1, dtype=torch.int32, device=q.device) if check else None
    kda_chunk_fwd_split(q, k, v, g, beta, cu_seqlens, cu_seqlens_host, initial_state, scale, lower_bound, o, fs,
                        status, stream, segment_chunks=segment_chunks)
    if check:
        code = int(status.item())
        if code != KDA_OK:
            raise KdaError(code, "kda_chunk_fwd_split (device)")
    return o, fs


def host_buffer_size(cu_seqlens_host, num_heads: int, with_initial_state: bool, with_final_state: bool = True,
                     groups: int = 0) -> int:
    cu, ptr = _host_cu(cu_seqlens_host)
    return int(load_library().kda_chunk_fwd_host_buffer_size(ptr, cu.numel() - 1, int(num_heads),
                                                              int(bool(with_initial_state)),
                                                              int(bool(with_final_state)), int(groups)))


def kda_chunk_fwd_host(q, k, v, g, beta, cu_seqlens_host, initial_state, scale: float, lower_bound: float, o,
                       final_state, device_buffer, status=None, groups: int = 0, stream=None, h2d_stream=None,
                       d2h_stream=None) -> int:
    """Call ``kda_chunk_fwd_host``: q .. beta, initial_state, o and final_state
    are CPU tensors (layouts as ``kda_chunk_fwd``), ``device_buffer`` a CUDA uint8
    tensor of ``host_buffer_size(...)`` bytes. With ``groups=0`` and page-locked
    tensors (``pin_memory()``) the kernel reads and writes them in place; else
    the copies of groups of sequences overlap the computation. The results are
    in ``o`` / ``final_state`` once ``stream`` is synchronised."""
    T, H, D = q.shape
    cu, cu_ptr = _host_cu(cu_seqlens_host)
    N = cu.numel() - 1
    cpu = torch.device("cpu")
    _check(q, "q", torch.bfloat16, (T, H, D), cpu)
    _check(k, "k", torch.bfloat16, (T, H, D), cpu)
    _check(v, "v", torch.bfloat16, (T, H, v.shape[2]), cpu)
    _check(g, "g", torch.float32, (T, H, D), cpu)
    _check(beta, "beta", torch.float32, (T, H), cpu)
    _check(o, "o", torch.float32, tuple(v.shape), cpu)
    for t, name in ((initial_state, "initial_state"), (final_state, "final_state")):
        if t is not None:
            _check(t, name, torch.float32, (N, H, D, v.shape[2]), cpu)
    dev = device_buffer.device
    if dev.type != "cuda" or device_buffer.dtype != torch.uint8 or not device_buffer.is_contiguous():
        raise ValueError("device_buffer must be a contiguous CUDA uint8 tensor")
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sp = lambda s_: None if s_ is None else ctypes.c_void_p(s_.cuda_stream)
    rc = load_library().kda_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), cu_ptr, N, T, H, D,
                                           v.shape[2], _ptr(initial_state), float(scale), float(lower_bound), _ptr(o),
                                           _ptr(final_state), _ptr(status), _ptr(device_buffer), device_buffer.numel(),
                                           int(groups), sp(stream), sp(h2d_stream), sp(d2h_stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_host")
    return rc


def kda_decode_fwd(q, k, v, g, beta, num_seqs: int, initial_state, scale: float, lower_bound: float,
                   o, final_state, status=None, stream=None) -> int:
    """Call the C entry point ``kda_decode_fwd`` with caller-allocated outputs.

    q, k, v: bf16 [N*Tn, H, 128] (sequence n's Tn tokens at rows n*Tn..); g:
    fp32 [N*Tn, H, 128]; beta: fp32 [N*Tn, H]; o: fp32 [N*Tn, H, 128];
    initial_state / final_state: fp32 [N, H, 128, 128] or None (they may be
    the same tensor). Raises ``KdaError`` on a host-side error.
    """
    T, H, D = q.shape
    N = int(num_seqs)
    if N < 0 or (N == 0 and T != 0) or (N > 0 and T % N != 0):
        raise ValueError("q must hold the same number of tokens for every sequence")
    Tn = T // N if N > 0 else 0
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    _check(q, "q", torch.bfloat16, (T, H, D), dev)
    _check(k, "k", torch.bfloat16, (T, H, D), dev)
    _check(v, "v", torch.bfloat16, (T, H, v.shape[2]), dev)
    _check(g, "g", torch.float32, (T, H, D), dev)
    _check(beta, "beta", torch.float32, (T, H), dev)
    _check(o, "o", torch.float32, tuple(v.shape), dev)
    if initial_state is not None:
        _check(initial_state, "initial_state", torch.float32, (N, H, D, v.shape[2]), dev)
    if final_state is not None:
        _check(final_state, "final_state", torch.float32, (N, H, D, v.shape[2]), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = load_library().kda_decode_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), N, Tn, H, D, v.shape[2], _ptr(initial_state),
        float(scale), float(lower_bound), _ptr(o), _ptr(final_state), _ptr(status), ctypes.c_void_p(stream.cuda_stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_fwd")
    return rc


def decode_fwd(q, k, v, g, beta, num_seqs: int, state=None, scale: Optional[float] = None,
               lower_bound: float = -5.0, in_place: bool = False, check: bool = False, stream=None):
    """Run ``kda_decode_fwd``; returns ``(o, final_state)``. With ``in_place``
    the given ``state`` tensor is updated and returned as ``final_state``."""
    T, H, D = q.shape
    N = int(num_seqs)
    if scale is None:
        scale = D ** -0.5
    o = torch.empty((T, H, v.shape[2]), dtype=torch.float32, device=q.device)
    if in_place:
        if state is None:
            raise ValueError("in_place needs a state tensor")
        fs = state
    else:
        fs = torch.empty((N, H, D, v.shape[2]), dtype=torch.float32, device=q.device)
    status = torch.zeros(1, dtype=torch.int32, device=q.device) if check else None
    kda_decode_fwd(q, k, v, g, beta, N, state, scale, lower_bound, o, fs, status, stream)
    if check:
        code = int(status.item())
        if code != KDA_OK:
            raise KdaError(code, "kda_decode_fwd (device)")
    return o, fs
