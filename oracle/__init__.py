"""fp64 CPU oracle for Kimi Delta Attention (KDA).

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the CUDA library never
imports, links or runs anything here, and this package shares no code with it.

``prefill``/``decode`` wrap the C recurrence in ``kda_oracle.c`` (token by
token, fp64).  ``chunk_form`` is a plain fp64 NumPy statement of the chunkwise
parallel form the paper review names ("Kimi Linear's chunkwise parallel form",
section "Kimi Delta Attention (KDA)"), kept only to pin that algebra against
the recurrence.
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

F32, BF16, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain C, no GPU)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC",
           "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, dp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
            lib.kda_oracle_prefill.argtypes = [vp, vp, vp, vp, vp, ip, dp, dp, ip, ip, ip, ip,
                                               dp, dp, ip]
            lib.kda_oracle_prefill.restype = ip
            lib.kda_oracle_prefill_ckpt.argtypes = [vp, vp, vp, vp, vp, ip, dp, dp, ip, ip, ip,
                                                    ip, dp, dp, dp, dp, ctypes.c_longlong, ip]
            lib.kda_oracle_prefill_ckpt.restype = ip
            lib.kda_oracle_decode.argtypes = [vp, vp, vp, vp, vp, ip, dp, ip, ip, ip, ip, dp, ip]
            lib.kda_oracle_decode.restype = ip
            lib.kda_oracle_default_threads.restype = ip
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().kda_oracle_default_threads())


def _as_host(x, name):
    """Return (contiguous numpy array, dtype code) holding exactly x's bytes."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                x = x.cpu()
            x = x.contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float64:
                return x.numpy(), F64
            raise TypeError(f"{name}: unsupported dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"{name}: unsupported dtype {a.dtype}")


def _state_f64(s, shape):
    if s is None:
        return None
    try:
        import torch
        if isinstance(s, torch.Tensor):
            s = s.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    s = np.ascontiguousarray(s, dtype=np.float64)
    if s.shape != shape:
        raise ValueError(f"state shape {s.shape} != {shape}")
    return s


def checkpoint_offsets(cu_seqlens, interval: int):
    """Row offsets of each sequence's checkpoints: sequence n owns
    floor(len_n / interval) rows starting at offsets[n]."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    counts = (cu[1:] - cu[:-1]) // int(interval)
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


def output_gate(o, z, weight, eps):
    """KDA output epilogue, in fp64: head-wise RMSNorm of the output, then the
    full-rank gate ("[Paper Review] Kimi K3: Open Frontier Intelligence",
    section "Kimi Delta Attention (KDA)", paragraph "Full-rank gate"; its
    formula was lost from the page, the reading is y = RMSNorm(o) * w * sigmoid(z)).

    o, z: [..., dv] (z is the gate pre-activation of the same tokens and
    heads); weight: [dv], the RMSNorm scale; eps: added to the mean square.
    For every row: y = o / sqrt(mean(o^2) + eps) * weight * sigmoid(z).
    """
    o = np.asarray(o, dtype=np.float64)
    z = _f64(z)
    w = _f64(weight)
    if z.shape != o.shape or w.shape != o.shape[-1:]:
        raise ValueError("output_gate: shape mismatch")
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return o / np.sqrt(ms + float(eps)) * w * (1.0 / (1.0 + np.exp(-z)))


G_MIN = -5.0
CONV_LEN = 4


def prologue(q_pre, k_pre, z, conv_q, conv_k, a_log, cu_seqlens=None, eps: float = 1e-6):
    """KDA's input prologue, in fp64 ("[Paper Review] Kimi K3: Open Frontier
    Intelligence", section "Kimi Delta Attention (KDA)": query and key pass
    through a short convolution, then Swish, and are L2-normalised; the
    log-decay is the scaled sigmoid g = g_min sigmoid(exp(A_h) z), g_min = -5;
    the page lost both formulas, these are their plain readings).

    q_pre, k_pre, z: [T, H, dk] pre-activations (z is the decay logit);
    conv_q, conv_k: [H, dk, 4] depthwise causal kernels, tap 3 on the current
    token (out_t = sum_i w[i] x_{t-3+i}, zero before each sequence's start);
    a_log: [H] the per-head log-scale A_h.  Returns q, k, g ([T, H, dk] fp64).
    """
    xq, xk, zz = _f64(q_pre), _f64(k_pre), _f64(z)
    wq, wk, al = _f64(conv_q), _f64(conv_k), _f64(a_log)
    T, H, dk = xq.shape
    cu = (np.array([0, T]) if cu_seqlens is None
          else np.asarray(_f64(cu_seqlens), dtype=np.int64))

    def branch(x, w):
        y = np.zeros_like(x)
        for n in range(len(cu) - 1):
            t0, t1 = int(cu[n]), int(cu[n + 1])
            for t in range(t0, t1):
                for i in range(CONV_LEN):
                    src = t - (CONV_LEN - 1) + i
                    if src >= t0:
                        y[t] += w[:, :, i] * x[src]
        y = y / (1.0 + np.exp(-y))                    # Swish: y sigmoid(y)
        return y / np.sqrt(np.sum(y * y, axis=-1, keepdims=True) + eps)

    g = G_MIN / (1.0 + np.exp(-(np.exp(al)[None, :, None] * zz)))
    return branch(xq, wq), branch(xk, wk), g


def prefill(q, k, v, g, beta, init_state=None, cu_seqlens=None, threads: int = 0,
            ckpt_interval: int = 0, gate=None):
    """Token-by-token fp64 KDA over packed sequences.

    q, k, g: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; init_state: [N, H, dk, dv]
    or None (zeros); cu_seqlens: [N+1] offsets or None (one sequence).
    Returns (out [T, H, dv] fp64, final_state [N, H, dk, dv] fp64), plus the
    checkpoints [n_ckpt, H, dk, dv] (state after every ckpt_interval tokens of
    each sequence, rows laid out by checkpoint_offsets) when ckpt_interval > 0.
    gate = (z [T, H, dv], weight [dv], eps): out is output_gate(o, z, weight, eps).
    """
    arrs = [_as_host(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"))]
    codes = {c for _, c in arrs}
    if len(codes) != 1:
        raise TypeError("q, k, v, g, beta must share one dtype")
    (qa, dt), (ka, _), (va, _), (ga, _), (ba, _) = arrs
    T, H, dk = qa.shape
    dv = va.shape[2]
    if ka.shape != (T, H, dk) or ga.shape != (T, H, dk) or va.shape != (T, H, dv) or ba.shape != (T, H):
        raise ValueError("shape mismatch among q, k, v, g, beta")
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        try:
            import torch
            if isinstance(cu_seqlens, torch.Tensor):
                cu_seqlens = cu_seqlens.detach().cpu().numpy()
        except ImportError:  # pragma: no cover
            pass
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    if cu[0] != 0 or cu[-1] != T:
        raise ValueError("cu_seqlens must start at 0 and end at T")
    s0 = _state_f64(init_state, (N, H, dk, dv))
    out = np.zeros((T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64)
    ck = offs = None
    if ckpt_interval:
        offs = checkpoint_offsets(cu, ckpt_interval)
        ck = np.zeros((int(offs[-1]), H, dk, dv), dtype=np.float64)
    rc = _load().kda_oracle_prefill_ckpt(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, ga.ctypes.data, ba.ctypes.data, dt,
        None if s0 is None else s0.ctypes.data, cu.ctypes.data, N, H, dk, dv,
        out.ctypes.data, fin.ctypes.data, None if ck is None else ck.ctypes.data,
        None if offs is None else offs.ctypes.data, int(ckpt_interval), int(threads))
    if rc < 0:
        raise RuntimeError(f"kda_oracle_prefill failed ({rc})")
    prefill.last_threads = rc
    if gate is not None:
        out = output_gate(out, *gate)
    if ckpt_interval:
        return out, fin, ck
    return out, fin


prefill.last_threads = 0


def decode(q, k, v, g, beta, state, threads: int = 0, gate=None):
    """One fp64 decode step for N sequences; q, k, g: [N, H, dk], v: [N, H, dv],
    beta: [N, H], state: [N, H, dk, dv].  Returns (out [N, H, dv], new_state);
    gate = (z [N, H, dv], weight [dv], eps) applies output_gate to out."""
    arrs = [_as_host(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"))]
    (qa, dt), (ka, _), (va, _), (ga, _), (ba, _) = arrs
    N, H, dk = qa.shape
    dv = va.shape[2]
    st = _state_f64(state, (N, H, dk, dv)).copy()
    out = np.zeros((N, H, dv), dtype=np.float64)
    rc = _load().kda_oracle_decode(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, ga.ctypes.data,
                                   ba.ctypes.data, dt, st.ctypes.data, N, H, dk, dv,
                                   out.ctypes.data, int(threads))
    if rc < 0:
        raise RuntimeError(f"kda_oracle_decode failed ({rc})")
    if gate is not None:
        out = output_gate(out, *gate)
    return out, st


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def chunk_form(q, k, v, g, beta, init_state=None, cu_seqlens=None, chunk: int = 64):
    """The chunkwise parallel form, in fp64 NumPy, written from the recurrence.

    Within one chunk of C tokens of one (sequence, head), with S0 the state
    entering the chunk and G the inclusive cumulative sum of g along the chunk:
        Kt = k*exp(G), Qt = q*exp(G), Kh = k*exp(-G), Kb = k*exp(G_C - G)
        A  = strictly_lower(diag(beta) Kt Kh^T);   Tinv = (I + A)^-1
        U  = Tinv diag(beta) (V - Kt S0)
        O  = Qt S0 + lower_incl(Qt Kh^T) U
        S_C = Diag(exp(G_C)) S0 + Kb^T U
    A chunk never crosses a sequence boundary; the last chunk may be short.
    fp64 holds exp(+-5*C) for the chunk sizes used here.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, T] if cu_seqlens is None else _f64(cu_seqlens), dtype=np.int64)
    N = len(cu) - 1
    s0 = np.zeros((N, H, dk, dv)) if init_state is None else _f64(init_state)
    out = np.zeros((T, H, dv))
    fin = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = s0[n, h].copy()
            for c0 in range(cu[n], cu[n + 1], chunk):
                c1 = min(c0 + chunk, cu[n + 1])
                C = c1 - c0
                kc, qc, vc = k[c0:c1, h], q[c0:c1, h], v[c0:c1, h]
                bc = beta[c0:c1, h]
                G = np.cumsum(g[c0:c1, h], axis=0)
                Kt, Qt = kc * np.exp(G), qc * np.exp(G)
                Kh = kc * np.exp(-G)
                Kb = kc * np.exp(G[-1] - G)
                A = np.tril(bc[:, None] * (Kt @ Kh.T), -1)
                Tinv = np.linalg.inv(np.eye(C) + A)
                U = Tinv @ (bc[:, None] * (vc - Kt @ S))
                out[c0:c1, h] = Qt @ S + np.tril(Qt @ Kh.T) @ U
                S = np.exp(G[-1])[:, None] * S + Kb.T @ U
            fin[n, h] = S
    return out, fin
