"""Kimi Delta Attention (KDA) on GB300: Python binding of libkda.so.

The binding only marshals arguments: it checks tensor shapes, dtypes and
devices, allocates outputs with PyTorch, and passes raw device pointers and the
current CUDA stream to the C ABI declared in ``include/kda.h``.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.  If
``libkda.so`` is missing or fails to load, every call raises.

    out, final_state = chunk_fwd(q, k, v, g, beta, init_state, cu_seqlens, chunk=64)
    out = decode_step(q, k, v, g, beta, state)          # state updated in place
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["chunk_fwd", "decode_step", "checkpoint_offsets", "prologue", "chunk_transition", "transition_apply", "chunk_fwd_kcp", "debug_wait_timeout", "workspace_size", "algorithm", "KDAError", "lib_path", "load"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libkda.so"
_lock = threading.Lock()
_lib = None
_lib_debug = None

KDA_F32, KDA_BF16 = 0, 1
_DTYPES = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().kda_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


class _Dims(ctypes.Structure):
    _fields_ = [("n_seqs", ctypes.c_int), ("total_tokens", ctypes.c_longlong),
                ("heads", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
                ("dtype", ctypes.c_int)]


def lib_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


def load():
    """Load libkda.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} not found: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


def load_debug_bounds():
    """The KDA_DEBUG_BOUNDS build of the library (libkda_debug.so, built on
    first use): every prefill and decode call given a dev_status first checks
    g in [-5, 0] and beta in [0, 1] on the device (KDA_ERR_RANGE).  Same
    entry points as ``load()``."""
    global _lib_debug
    with _lock:
        if _lib_debug is None:
            from . import build as _build
            _lib_debug = _declare(ctypes.CDLL(_build.build(debug_bounds=True)))
    return _lib_debug


def _declare(lib):
    """Argument and result types of every entry point of kda.h."""
    vp, ip, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    dp = ctypes.POINTER(_Dims)
    lib.kda_chunk_fwd_workspace_size.argtypes = [dp, ip]
    lib.kda_chunk_fwd_workspace_size.restype = sz
    lib.kda_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ip, dp, vp, sz, vp,
                                  vp]
    lib.kda_chunk_fwd.restype = ip
    lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, dp, vp, vp]
    lib.kda_decode_step.restype = ip
    lib.kda_status_string.argtypes = [ip]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_version.restype = ip
    lib.kda_chunk_fwd_checkpoints.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ip, dp,
                                              vp, sz, vp, vp, vp, vp, ip]
    lib.kda_chunk_fwd_checkpoints.restype = ip
    fl = ctypes.c_float
    lib.kda_chunk_fwd_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, fl, vp, vp,
                                        ip, dp, vp, sz, vp, vp]
    lib.kda_chunk_fwd_gated.restype = ip
    lib.kda_decode_step_gated.argtypes = [vp, vp, vp, vp, vp, vp, vp, fl, vp, vp, dp, vp,
                                          vp]
    lib.kda_decode_step_gated.restype = ip
    ll = ctypes.c_longlong
    lib.kda_chunk_transition_workspace_size.argtypes = [dp]
    lib.kda_chunk_transition_workspace_size.restype = sz
    lib.kda_chunk_transition.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ip, dp, vp, sz,
                                         vp, vp]
    lib.kda_chunk_transition.restype = ip
    lib.kda_transition_apply.argtypes = [vp, vp, vp, vp, ll, ip, ip, vp]
    lib.kda_transition_apply.restype = ip
    lib.kda_debug_wait_timeout.argtypes = [vp, ctypes.c_uint, vp]
    lib.kda_debug_wait_timeout.restype = ip
    lib.kda_chunk_fwd_kcp_workspace_size.argtypes = [dp, ip]
    lib.kda_chunk_fwd_kcp_workspace_size.restype = sz
    lib.kda_chunk_fwd_kcp.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ip, dp, vp, sz, vp,
                                      vp]
    lib.kda_chunk_fwd_kcp.restype = ip
    lib.kda_prologue.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, dp, vp]
    lib.kda_prologue.restype = ip
    lib.kda_chunk_fwd_algorithm.argtypes = [dp, ip]
    lib.kda_chunk_fwd_algorithm.restype = ip
    lib.kda_chunk_fwd_launch_count.argtypes = [dp, ip, sz, ip]
    lib.kda_chunk_fwd_launch_count.restype = ip
    lib.kda_debug_chunk_fwd_withhold.argtypes = [ip, vp, vp, vp, vp, vp, vp, vp, vp, dp, vp, sz,
                                                 vp, vp]
    lib.kda_debug_chunk_fwd_withhold.restype = ip
    lib.kda_check_inputs.argtypes = [vp, vp, dp, vp, vp]
    lib.kda_check_inputs.restype = ip
    lib.kda_debug_bounds_build.restype = ip
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_input(name, t, shape, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(n_seqs, total_tokens, heads, dk, dv, dtype):
    return _Dims(int(n_seqs), int(total_tokens), int(heads), int(dk), int(dv), _DTYPES[dtype])


def workspace_size(n_seqs, total_tokens, heads, dk, dv, dtype=torch.bfloat16, chunk=64) -> int:
    d = _dims(n_seqs, total_tokens, heads, dk, dv, dtype)
    return int(load().kda_chunk_fwd_workspace_size(ctypes.byref(d), int(chunk)))


def algorithm(n_seqs, total_tokens, heads, dk, dv, dtype=torch.bfloat16, chunk=64) -> str:
    """Name of the kernel kda_chunk_fwd dispatches to for these sizes."""
    d = _dims(n_seqs, total_tokens, heads, dk, dv, dtype)
    rc = int(load().kda_chunk_fwd_algorithm(ctypes.byref(d), int(chunk)))
    if rc < 0:
        raise KDAError(rc, "kda_chunk_fwd_algorithm")
    return {0: "recurrent", 1: "tcgen05", 2: "tcgen05_split"}[rc]


def launch_count(n_seqs, total_tokens, heads, dk, dv, dtype=torch.bfloat16, chunk=64,
                 workspace_bytes=None, varlen=False) -> int:
    """Kernels one kda_chunk_fwd call launches for these sizes (the workspace
    ``workspace_size`` gives unless workspace_bytes is passed; varlen: with
    cu_seqlens), on the current CUDA device."""
    d = _dims(n_seqs, total_tokens, heads, dk, dv, dtype)
    lib = load()
    if workspace_bytes is None:
        workspace_bytes = int(lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), int(chunk)))
    rc = int(lib.kda_chunk_fwd_launch_count(ctypes.byref(d), int(chunk), int(workspace_bytes),
                                            int(bool(varlen))))
    if rc < 0:
        raise KDAError(rc, "kda_chunk_fwd_launch_count")
    return rc


def checkpoint_offsets(lengths, interval: int) -> list:
    """Checkpoint row offsets for host-side sequence lengths: sequence n owns
    floor(len_n / interval) rows starting at offsets[n]."""
    offs = [0]
    for n in lengths:
        offs.append(offs[-1] + int(n) // int(interval))
    return offs


def chunk_fwd(q, k, v, g, beta, init_state=None, cu_seqlens=None, chunk: int = 64, *,
              n_seqs: int | None = None, out=None, final_state=None,
              output_final_state: bool = True, workspace=None, dev_status=None, stream=None,
              ckpt_interval: int = 0, ckpt_offsets=None, checkpoints=None, gate=None):
    """Chunkwise KDA prefill over packed sequences (``kda_chunk_fwd``).

    q, k, g: [T, H, dk]; v: [T, H, dv]; beta: [T, H] (fp32 or bf16, one dtype,
    on one CUDA device).  init_state: [N, H, dk, dv] fp32 or None (zeros).
    cu_seqlens: int32 [N+1] on the device, or None for ``n_seqs`` (default 1)
    equal-length sequences.  Returns (out [T, H, dv], final_state or None).

    With ckpt_interval > 0 (a multiple of 64) it calls
    ``kda_chunk_fwd_checkpoints`` and returns (out, final_state, checkpoints):
    the state after every ckpt_interval tokens of each sequence, rows laid out
    by ckpt_offsets (int32 [N+1] on the device; computed from cu_seqlens when
    not given, which reads the lengths back to the host).

    With gate = (z, norm_weight, eps) it calls ``kda_chunk_fwd_gated``: out is
    RMSNorm(o) * norm_weight * sigmoid(z) per (token, head) row (z [T, H, dv]
    in the inputs' dtype, norm_weight fp32 [dv]).
    """
    lib = load()
    if q.dim() != 3:
        raise ValueError("q must be [T, H, dk]")
    T, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if dt not in _DTYPES:
        raise TypeError(f"unsupported dtype {dt}")
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("g", g, (T, H, dk)),
                         ("v", v, (T, H, dv)), ("beta", beta, (T, H))):
        _check_input(name, t, shp, dt, dev)
    if cu_seqlens is not None:
        _check_input("cu_seqlens", cu_seqlens, (cu_seqlens.numel(),), torch.int32, dev)
        N = cu_seqlens.numel() - 1
    else:
        N = 1 if n_seqs is None else int(n_seqs)
    if init_state is not None:
        _check_input("init_state", init_state, (N, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=dt, device=dev)
    else:
        _check_input("out", out, (T, H, dv), dt, dev)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    elif final_state is not None:
        _check_input("final_state", final_state, (N, H, dk, dv), torch.float32, dev)
    d = _dims(N, T, H, dk, dv, dt)
    need = int(lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), int(chunk)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if gate is not None:
        if ckpt_interval:
            raise ValueError("checkpoints and the output gate are separate calls")
        z, nw, eps = gate
        _check_input("gate", z, (T, H, dv), dt, dev)
        _check_input("norm_weight", nw, (dv,), torch.float32, dev)
        with torch.cuda.device(dev):
            rc = lib.kda_chunk_fwd_gated(
                _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                _ptr(cu_seqlens), _ptr(z), _ptr(nw), float(eps), _ptr(out), _ptr(final_state),
                int(chunk), ctypes.byref(d), _ptr(workspace), ws_bytes, _ptr(dev_status),
                _stream_handle(stream))
        if rc != 0:
            raise KDAError(rc, "kda_chunk_fwd_gated")
        return out, final_state
    if ckpt_interval:
        if ckpt_offsets is None:
            lens = ([T // N] * N if cu_seqlens is None
                    else (cu_seqlens[1:] - cu_seqlens[:-1]).tolist())
            ckpt_offsets = torch.tensor(checkpoint_offsets(lens, ckpt_interval),
                                        dtype=torch.int32, device=dev)
        _check_input("ckpt_offsets", ckpt_offsets, (N + 1,), torch.int32, dev)
        if checkpoints is None:
            n_ck = int(ckpt_offsets[-1].item())
            checkpoints = torch.empty((max(n_ck, 1), H, dk, dv), dtype=torch.float32, device=dev)
        with torch.cuda.device(dev):
            rc = lib.kda_chunk_fwd_checkpoints(
                _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                _ptr(cu_seqlens), _ptr(out), _ptr(final_state), int(chunk), ctypes.byref(d),
                _ptr(workspace), ws_bytes, _ptr(dev_status), _stream_handle(stream),
                _ptr(checkpoints), _ptr(ckpt_offsets), int(ckpt_interval))
        if rc != 0:
            raise KDAError(rc, "kda_chunk_fwd_checkpoints")
        return out, final_state, checkpoints
    with torch.cuda.device(dev):
        rc = lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                               _ptr(cu_seqlens), _ptr(out), _ptr(final_state), int(chunk),
                               ctypes.byref(d), _ptr(workspace), ws_bytes, _ptr(dev_status),
                               _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_chunk_fwd")
    return out, final_state


def decode_step(q, k, v, g, beta, state, *, out=None, dev_status=None, stream=None, gate=None):
    """One KDA decode step (``kda_decode_step``): q, k, g [N, H, dk], v [N, H, dv],
    beta [N, H]; state [N, H, dk, dv] fp32 is updated in place.  Returns out.
    gate = (z [N, H, dv], norm_weight fp32 [dv], eps) applies the output
    epilogue (``kda_decode_step_gated``)."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if dt not in _DTYPES:
        raise TypeError(f"unsupported dtype {dt}")
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("g", g, (N, H, dk)),
                         ("v", v, (N, H, dv)), ("beta", beta, (N, H))):
        _check_input(name, t, shp, dt, dev)
    _check_input("state", state, (N, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((N, H, dv), dtype=dt, device=dev)
    else:
        _check_input("out", out, (N, H, dv), dt, dev)
    d = _dims(N, N, H, dk, dv, dt)
    if gate is not None:
        z, nw, eps = gate
        _check_input("gate", z, (N, H, dv), dt, dev)
        _check_input("norm_weight", nw, (dv,), torch.float32, dev)
        with torch.cuda.device(dev):
            rc = lib.kda_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                           _ptr(z), _ptr(nw), float(eps), _ptr(state), _ptr(out),
                                           ctypes.byref(d), _ptr(dev_status),
                                           _stream_handle(stream))
        if rc != 0:
            raise KDAError(rc, "kda_decode_step_gated")
        return out
    with torch.cuda.device(dev):
        rc = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                 _ptr(out), ctypes.byref(d), _ptr(dev_status),
                                 _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_decode_step")
    return out


def chunk_transition(q, k, v, g, beta, cu_seqlens=None, *, n_seqs: int | None = None,
                     workspace=None, dev_status=None, stream=None):
    """Segment transitions (``kda_chunk_transition``): for each (sequence, head)
    of the packed input, (M [N, H, dk, dk], H [N, H, dk, dv]) with
    S_end = M S_0 + H."""
    lib = load()
    T, Hh, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (n_seqs or 1)
    for name, t, shp in (("q", q, (T, Hh, dk)), ("k", k, (T, Hh, dk)), ("g", g, (T, Hh, dk)),
                         ("v", v, (T, Hh, dv)), ("beta", beta, (T, Hh))):
        _check_input(name, t, shp, dt, dev)
    d = _dims(N, T, Hh, dk, dv, dt)
    M = torch.empty((N, Hh, dk, dk), dtype=torch.float32, device=dev)
    Hs = torch.empty((N, Hh, dk, dv), dtype=torch.float32, device=dev)
    need = int(lib.kda_chunk_transition_workspace_size(ctypes.byref(d)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib.kda_chunk_transition(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                      _ptr(cu_seqlens), _ptr(M), _ptr(Hs), 64, ctypes.byref(d),
                                      _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                      _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_chunk_transition")
    return M, Hs


def check_inputs(g, beta, dev_status, *, stream=None, lib=None):
    """Range precondition of the inputs (``kda_check_inputs``): sets the device
    int dev_status to KDA_ERR_RANGE if any g [T, H, dk] lies outside [-5, 0] or
    any beta [T, H] outside [0, 1] (NaN included), unless it is non-zero
    already.  Asynchronous; read dev_status after synchronising."""
    lib = lib or load()
    T, H, dk = g.shape
    dev, dt = g.device, g.dtype
    _check_input("beta", beta, (T, H), dt, dev)
    _check_input("dev_status", dev_status, (1,), torch.int32, dev)
    d = _dims(1, T, H, dk, dk, dt)
    with torch.cuda.device(dev):
        rc = lib.kda_check_inputs(_ptr(g), _ptr(beta), ctypes.byref(d), _ptr(dev_status),
                                  _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_check_inputs")


def debug_chunk_fwd_withhold(which: int, q, k, v, g, beta, init_state, dev_status, *,
                             stream=None):
    """Failure-detection self-test of the prefill kernels
    (``kda_debug_chunk_fwd_withhold``): one copy is never issued (which = 1:
    the split state kernel's first record; 2: the split preparation kernel's
    first raw tiles; 3: the fused kernel's first raw tiles), so a production
    kernel's bounded wait expires and it reports KDA_ERR_TIMEOUT through
    dev_status.  One sequence; returns the (meaningless) outputs."""
    lib = load()
    T, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    out = torch.empty((T, H, dv), dtype=dt, device=dev)
    fin = torch.empty((1, H, dk, dv), dtype=torch.float32, device=dev)
    d = _dims(1, T, H, dk, dv, dt)
    need = int(lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), 64))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib.kda_debug_chunk_fwd_withhold(int(which), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                              _ptr(beta), _ptr(init_state), _ptr(out), _ptr(fin),
                                              ctypes.byref(d), _ptr(ws), need, _ptr(dev_status),
                                              _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_debug_chunk_fwd_withhold")
    return out, fin


def debug_wait_timeout(dev_status, timeout_us: int, *, stream=None):
    """``kda_debug_wait_timeout``: a kernel whose bounded wait cannot succeed
    stores KDA_ERR_TIMEOUT (-4) into the device int ``dev_status`` after
    ``timeout_us`` microseconds and returns (failure-detection self-test)."""
    lib = load()
    with torch.cuda.device(dev_status.device):
        rc = lib.kda_debug_wait_timeout(_ptr(dev_status), int(timeout_us), _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_debug_wait_timeout")


def transition_apply(M, H, S, *, out=None, stream=None):
    """``kda_transition_apply``: out = M S + H per (…, dk, dv) pair (H may be None)."""
    lib = load()
    dk, dv = S.shape[-2], S.shape[-1]
    pairs = S.numel() // (dk * dv)
    if out is None:
        out = torch.empty_like(S)
    with torch.cuda.device(S.device):
        rc = lib.kda_transition_apply(_ptr(M), _ptr(H), _ptr(S), _ptr(out), pairs, dk, dv,
                                      _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_transition_apply")
    return out


def chunk_fwd_kcp(q, k, v, g, beta, init_state=None, *, n_seqs: int = 1, segments: int = 4,
                  out=None, final_state=None, workspace=None, dev_status=None, stream=None):
    """Single-GPU KCP prefill (``kda_chunk_fwd_kcp``) of n_seqs equal-length
    sequences, each cut into `segments` segments.  Returns (out, final_state)."""
    lib = load()
    T, Hh, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if out is None:
        out = torch.empty((T, Hh, dv), dtype=dt, device=dev)
    if final_state is None:
        final_state = torch.empty((n_seqs, Hh, dk, dv), dtype=torch.float32, device=dev)
    d = _dims(n_seqs, T, Hh, dk, dv, dt)
    need = int(lib.kda_chunk_fwd_kcp_workspace_size(ctypes.byref(d), int(segments)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib.kda_chunk_fwd_kcp(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   _ptr(init_state), _ptr(out), _ptr(final_state), int(segments),
                                   ctypes.byref(d), _ptr(workspace), workspace.numel(),
                                   _ptr(dev_status), _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_chunk_fwd_kcp")
    return out, final_state


def prologue(q_pre, k_pre, z, conv_q, conv_k, a_log, cu_seqlens=None, *, n_seqs: int = 1,
             q=None, k=None, g=None, stream=None):
    """``kda_prologue``: (q, k, g) from the pre-activations ([T, H, dk], one
    dtype), the 4-tap convolution kernels conv_q, conv_k (fp32 [H, dk, 4]) and
    a_log (fp32 [H])."""
    lib = load()
    T, Hh, dk = q_pre.shape
    dev, dt = q_pre.device, q_pre.dtype
    for name, t in (("q_pre", q_pre), ("k_pre", k_pre), ("z", z)):
        _check_input(name, t, (T, Hh, dk), dt, dev)
    _check_input("conv_q", conv_q, (Hh, dk, 4), torch.float32, dev)
    _check_input("conv_k", conv_k, (Hh, dk, 4), torch.float32, dev)
    _check_input("a_log", a_log, (Hh,), torch.float32, dev)
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else n_seqs
    q = torch.empty_like(q_pre) if q is None else q
    k = torch.empty_like(q_pre) if k is None else k
    g = torch.empty_like(q_pre) if g is None else g
    d = _dims(N, T, Hh, dk, dk, dt)
    with torch.cuda.device(dev):
        rc = lib.kda_prologue(_ptr(q_pre), _ptr(k_pre), _ptr(z), _ptr(conv_q), _ptr(conv_k),
                              _ptr(a_log), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(g),
                              ctypes.byref(d), _stream_handle(stream))
    if rc != 0:
        raise KDAError(rc, "kda_prologue")
    return q, k, g
