"""Seeded synthetic KDA inputs, shared by the tests, the oracle checks and the benchmark.

This module draws random numbers and shapes them into the input recipe; it
holds none of the recurrence's arithmetic and imports neither the CUDA library
nor the oracle.

Recipe (per workload; all draws from one seeded ``torch.Generator`` on the
target device, in the fixed order q, k, v, a, beta, initial state):
  * q, k ~ N(0, 1), then L2-normalised per (token, head) -- the paper review
    ("Kimi Delta Attention (KDA)") states q and k are L2-normalised;
  * v ~ N(0, 1);
  * g = g_min * sigmoid(a) with g_min = -5 and a ~ N(0, 1) per channel
    (a ~ U(-8, 8) for the saturating million-token workload), the
    lower-bounded scaled-sigmoid decay of the same section with the per-head
    log-scale A_h at its initial value 0;
  * beta = sigmoid(N(0, 1)) per (token, head);
  * initial states ~ N(0, 0.02) (standard deviation 0.02) or zeros.
Values are made in fp32 and then rounded (round-to-nearest-even) to the
workload's dtype; the oracle reads those rounded bytes.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

G_MIN = -5.0
SLAB_TOKENS = 1 << 16  # draws are made slab by slab to bound temporary memory


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    heads: int
    dk: int
    dv: int
    dtype: str                      # "f32" or "bf16" (q, k, v, g, beta, out)
    n_seqs: int = 1
    seq_len: int = 0                # tokens per sequence when all are equal
    varlen: tuple | None = None     # (lo, hi) inclusive uniform lengths
    init_state: bool = True         # N(0, 0.02) when True, zeros when False
    chunk: int = 64
    a_dist: str = "normal"          # "normal": N(0,1); "uniform8": U(-8, 8)
    decode_steps: int = 0           # > 0 for the decode workload

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    w.name: w for w in (
        Workload("prefill_T256_H1_d64_f32", heads=1, dk=64, dv=64, dtype="f32",
                 seq_len=256, init_state=False),
        Workload("prefill_T8192_H96_d128_bf16", heads=96, dk=128, dv=128, dtype="bf16",
                 seq_len=8192, init_state=True),
        Workload("varlen_32seq_H96_d128_bf16", heads=96, dk=128, dv=128, dtype="bf16",
                 n_seqs=32, varlen=(512, 16384), init_state=False),
        Workload("decode_256seq_H96_d128_64steps", heads=96, dk=128, dv=128, dtype="bf16",
                 n_seqs=256, seq_len=1, init_state=True, decode_steps=64),
        Workload("prefill_T1M_H32_d128_bf16", heads=32, dk=128, dv=128, dtype="bf16",
                 seq_len=1 << 20, init_state=True, a_dist="uniform8"),
    )
}


def seq_lengths(w: Workload, seed: int = 0) -> list[int]:
    """Per-sequence lengths: equal, or uniform in [lo, hi] from a seeded NumPy PCG64."""
    if w.varlen is None:
        return [w.seq_len] * w.n_seqs
    lo, hi = w.varlen
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=w.n_seqs)]


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def _fill(out: torch.Tensor, gen: torch.Generator, make):
    """Fill `out` ([T, ...]) slab by slab with make(fp32 standard normal slab)."""
    T = out.shape[0]
    for t0 in range(0, T, SLAB_TOKENS):
        t1 = min(T, t0 + SLAB_TOKENS)
        shape = (t1 - t0,) + tuple(out.shape[1:])
        out[t0:t1] = make(shape)


def _normal(gen, device):
    return lambda shape: torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def draw_token_tensors(T: int, H: int, dk: int, dv: int, dtype, gen, device, a_dist="normal"):
    """q, k, v, g, beta for T tokens x H heads, drawn in the recipe's order."""
    normal = _normal(gen, device)

    def unit(shape):
        x = normal(shape)
        return x / x.norm(dim=-1, keepdim=True)

    def gate(shape):
        if a_dist == "uniform8":
            a = torch.rand(shape, generator=gen, device=device, dtype=torch.float32) * 16.0 - 8.0
        else:
            a = normal(shape)
        return G_MIN * torch.sigmoid(a)

    q = torch.empty((T, H, dk), dtype=dtype, device=device)
    k = torch.empty_like(q)
    v = torch.empty((T, H, dv), dtype=dtype, device=device)
    g = torch.empty_like(q)
    beta = torch.empty((T, H), dtype=dtype, device=device)
    _fill(q, gen, unit)
    _fill(k, gen, unit)
    _fill(v, gen, normal)
    _fill(g, gen, gate)
    _fill(beta, gen, lambda s: torch.sigmoid(normal(s)))
    return q, k, v, g, beta


def draw_states(N: int, H: int, dk: int, dv: int, gen, device, std=0.02):
    s = torch.empty((N, H, dk, dv), dtype=torch.float32, device=device)
    for n in range(N):  # one sequence at a time bounds the fp32 temporaries
        s[n] = torch.randn((H, dk, dv), generator=gen, device=device) * std
    return s


def make_prefill(w: Workload, seed: int = 0, device="cpu", lengths=None, heads=None,
                 seq_len=None):
    """Inputs for one prefill call.  `lengths`, `heads`, `seq_len` override the
    workload's sizes (used for reduced parity cases).  Returns a dict with
    q, k, v, g, beta, init_state (or None), cu_seqlens (int32, same device)."""
    H = heads or w.heads
    if lengths is None:
        if seq_len is not None:
            lengths = [seq_len] * w.n_seqs
        else:
            lengths = seq_lengths(w, seed)
    T = int(sum(lengths))
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q, k, v, g, beta = draw_token_tensors(T, H, w.dk, w.dv, w.torch_dtype, gen, device, w.a_dist)
    init = draw_states(len(lengths), H, w.dk, w.dv, gen, device) if w.init_state else None
    cu = cu_from_lengths(lengths).to(device)
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=init, cu_seqlens=cu)


def make_decode_state(w: Workload, seed: int = 0, device="cpu", n_seqs=None, heads=None):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return draw_states(n_seqs or w.n_seqs, heads or w.heads, w.dk, w.dv, gen, device)


def make_decode_tokens(w: Workload, step: int, seed: int = 0, device="cpu", n_seqs=None,
                       heads=None):
    """q, k, v, g, beta ([N, H, d] / [N, H]) for decode step `step`."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + 1 + step)
    return draw_token_tensors(n_seqs or w.n_seqs, heads or w.heads, w.dk, w.dv, w.torch_dtype,
                              gen, device, w.a_dist)


def make_output_gate(T: int, H: int, dv: int, dtype, seed: int = 0, device="cpu"):
    """Synthetic inputs of the output epilogue: the gate pre-activation
    z ~ N(0, 1) ([T, H, dv], the layer's dtype; stands in for the full-rank
    projection of the hidden state), the RMSNorm scale w = 1 + 0.1 N(0, 1)
    (fp32 [dv]) and eps = 1e-6.  Drawn after everything else, from their own
    generator, so the other inputs of a workload do not change."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + 999_983)
    normal = _normal(gen, device)
    z = normal((T, H, dv)).to(dtype)
    w = 1.0 + 0.1 * normal((dv,))
    return z, w.float(), 1e-6


def make_prologue_inputs(T: int, H: int, dk: int, dtype, seed: int = 0, device="cpu"):
    """Synthetic prologue inputs: q_pre, k_pre ~ N(0, 1) and the decay logit
    z ~ N(0, 1) ([T, H, dk], dtype), 4-tap kernels ~ N(0, 1/4) (fp32
    [H, dk, 4]) and A_h ~ N(0, 0.25) (fp32 [H]; the page initialises A_h at 0,
    a spread exercises its scaling)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + 777_767)
    normal = _normal(gen, device)
    q_pre = normal((T, H, dk)).to(dtype)
    k_pre = normal((T, H, dk)).to(dtype)
    z = normal((T, H, dk)).to(dtype)
    conv_q = 0.5 * normal((H, dk, 4))
    conv_k = 0.5 * normal((H, dk, 4))
    a_log = 0.5 * normal((H,))
    return q_pre, k_pre, z, conv_q, conv_k, a_log
