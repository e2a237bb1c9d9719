"""Parity at the method's edge cases, on every path, against the fp64 oracle.

The decay bound of "[Paper Review] Kimi K3: Open Frontier Intelligence",
section "Kimi Delta Attention (KDA)" (g >= g_min = -5, so a 16-token tile's
log-decay stays above -80 and its reciprocal below e^80) is the whole reason
the chunked tensor-core form is safe, so the extremes are tested directly:

  * every g = -5.0 exactly, over whole 16-token tiles and whole 64-token
    chunks (the in-tile factors reach e^80), and mixed with undecayed tiles;
  * g = 0 everywhere (no decay: the longest memory, where the bf16 operand
    copy of the state is used for the most chunks);
  * g in [-0.05, 0] over sequences of one or two chunks and of 1000+ tokens;
  * beta = 0 with g = 0: the state passes through every chunk unchanged, so
    the final state equals the initial one bit for bit on every path;
  * orthonormal keys (signed basis vectors, exact in bf16) with beta = 1 and
    g = 0 from a zero state: the output recalls the value written under the
    queried key.

Each is run on the split and fused tensor-core forms, the fp32 CUDA-core
recurrence, prefix-cache checkpoints, the gated output, and decode; every
assertion message carries the case's maximum error.
"""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close, assert_close_gated, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = inputs.WORKLOADS


@pytest.fixture(params=["split", "fused"])
def tc_path(request, monkeypatch):
    monkeypatch.setenv("KDA_CHUNK_PATH", request.param)
    return request.param


def _set_g(d, kind, seed=0):
    """Replaces d["g"] by one of the edge-case decays (same shape and dtype)."""
    g = d["g"]
    T = g.shape[0]
    if kind == "min":                      # g = g_min everywhere
        d["g"] = torch.full_like(g, -5.0)
    elif kind == "zero":
        d["g"] = torch.zeros_like(g)
    elif kind == "slow":                   # g in [-0.05, 0]
        gen = torch.Generator(device=DEV).manual_seed(900 + seed)
        d["g"] = (-0.05 * torch.rand(g.shape, generator=gen, device=DEV)).to(g.dtype)
    elif kind == "min_tiles":
        # Alternating 16-token tiles at g_min and at g = 0, offset by 8 tokens
        # so some chunks start mid-pattern: e^80 factors next to long memory.
        t = torch.arange(T, device=DEV)
        on = ((t + 8) // 16) % 2 == 0
        d["g"] = torch.where(on[:, None, None], torch.full_like(g, -5.0), torch.zeros_like(g))
    elif kind == "min_chunks":
        # Whole 64-token chunks at g_min, every other chunk undecayed.
        t = torch.arange(T, device=DEV)
        on = (t // 64) % 2 == 0
        d["g"] = torch.where(on[:, None, None], torch.full_like(g, -5.0), torch.zeros_like(g))
    else:
        raise ValueError(kind)
    return d


def _inputs(kind, lengths, heads=2, dtype="bf16", d_head=128, seed=0, init=True):
    w = inputs.Workload("edge", heads=heads, dk=d_head, dv=d_head, dtype=dtype,
                        init_state=init)
    d = inputs.make_prefill(w, seed=100 + seed, device=DEV, lengths=lengths)
    return _set_g(d, kind, seed)


def _x(d):
    return [d[n] for n in ("q", "k", "v", "g", "beta")]


def _check(out, fin, d, tag, what):
    ro, rf = oracle.prefill(*_x(d), d["init_state"], d["cu_seqlens"])
    e_out = assert_close(out, ro, tag, f"{what} out")
    e_fin = assert_close(fin, rf, tag, f"{what} final_state")
    return e_out, e_fin


DECAYS = ["min", "min_tiles", "min_chunks", "zero", "slow"]


@pytest.mark.parametrize("kind", DECAYS)
def test_tensor_core_forms_at_decay_extremes(kind, tc_path):
    # Lengths: a ragged tail, one and two whole chunks, a long sequence.
    lengths = [70, 64, 128, 1100]
    d = _inputs(kind, lengths, heads=2, seed=1)
    out, fin = kda.chunk_fwd(*_x(d), d["init_state"], d["cu_seqlens"], chunk=64)
    torch.cuda.synchronize()
    e = _check(out, fin, d, "bf16", f"{tc_path} g={kind}")
    print(f"{tc_path} g={kind}: max |err| out {e[0]:.3e} final {e[1]:.3e}")


@pytest.mark.parametrize("kind", DECAYS)
def test_fp32_recurrence_at_decay_extremes(kind):
    d = _inputs(kind, [70, 1, 300], heads=2, dtype="f32", seed=2)
    out, fin = kda.chunk_fwd(*_x(d), d["init_state"], d["cu_seqlens"], chunk=64)
    torch.cuda.synchronize()
    e = _check(out, fin, d, "f32", f"fp32 g={kind}")
    print(f"fp32 g={kind}: normwise rel err out {e[0]:.3e} final {e[1]:.3e}")


@pytest.mark.parametrize("kind", ["min", "min_tiles", "zero", "slow"])
def test_checkpoints_at_decay_extremes(kind, tc_path):
    lengths = [700, 64, 1030]
    d = _inputs(kind, lengths, heads=2, seed=3)
    out, fin, ck = kda.chunk_fwd(*_x(d), d["init_state"], d["cu_seqlens"], chunk=64,
                                 ckpt_interval=128)
    torch.cuda.synchronize()
    ro, rf, rck = oracle.prefill(*_x(d), d["init_state"], d["cu_seqlens"], ckpt_interval=128)
    assert_close(out, ro, "bf16", f"ckpt {tc_path} g={kind} out")
    assert_close(fin, rf, "bf16", f"ckpt {tc_path} g={kind} final_state")
    e = assert_close(ck, rck, "bf16", f"ckpt {tc_path} g={kind} checkpoints")
    print(f"checkpoints {tc_path} g={kind}: max |err| {e:.3e}")


@pytest.mark.parametrize("kind", ["min", "zero", "slow"])
def test_gated_output_at_decay_extremes(kind, tc_path):
    lengths = [200, 1000]
    d = _inputs(kind, lengths, heads=2, seed=4)
    T = sum(lengths)
    gate = inputs.make_output_gate(T, 2, 128, torch.bfloat16, seed=4, device=DEV)
    out, fin = kda.chunk_fwd(*_x(d), d["init_state"], d["cu_seqlens"], chunk=64, gate=gate)
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(*_x(d), d["init_state"], d["cu_seqlens"])
    e = assert_close_gated(out, ro, gate, "bf16", f"gated {tc_path} g={kind} out")
    assert_close(fin, rf, "bf16", f"gated {tc_path} g={kind} final_state")
    print(f"gated {tc_path} g={kind}: max |err| {e:.3e}")


@pytest.mark.parametrize("kind", ["min", "zero", "slow"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_chain_at_decay_extremes(kind, dtype):
    N, H, steps = 6, 3, 40
    gen = torch.Generator(device=DEV).manual_seed(5)
    state = inputs.draw_states(N, H, 128, 128, gen, DEV)
    ref = state.cpu().double().numpy()
    tag = "bf16" if dtype == torch.bfloat16 else "f32"
    worst = 0.0
    for s in range(steps):
        tg = torch.Generator(device=DEV).manual_seed(5000 + s)
        q, k, v, g, beta = inputs.draw_token_tensors(N, H, 128, 128, dtype, tg, DEV)
        g = {"min": torch.full_like(g, -5.0), "zero": torch.zeros_like(g),
             "slow": (-0.05 * torch.rand(g.shape, generator=tg, device=DEV)).to(dtype)}[kind]
        out = kda.decode_step(q, k, v, g, beta, state)
        ro, ref = oracle.decode(q, k, v, g, beta, ref)
        if s % 8 == 7:
            torch.cuda.synchronize()
            worst = max(worst, assert_close(out, ro, tag, f"decode g={kind} step {s} out"))
    torch.cuda.synchronize()
    e = assert_close(state, ref, tag, f"decode g={kind} final state")
    print(f"decode {tag} g={kind}: out {worst:.3e} state {e:.3e}")


# ------------------------------------------------- beta = 0, g = 0: pass-through

def _passthrough_inputs(dtype, lengths, seed):
    d = _inputs("zero", lengths, heads=3, dtype=dtype, seed=seed)
    d["beta"] = torch.zeros_like(d["beta"])
    return d


@pytest.mark.parametrize("path", ["split", "fused", "fp32"])
def test_beta0_g0_state_passes_through(path, monkeypatch):
    """No erase, no write, no decay: every chunk maps the state to itself, so
    the final state is the initial one bit for bit, and o_t = S_0^T q_t."""
    if path == "fp32":
        d = _passthrough_inputs("f32", [70, 300, 1], 6)
        tag = "f32"
    else:
        monkeypatch.setenv("KDA_CHUNK_PATH", path)
        d = _passthrough_inputs("bf16", [70, 300, 1, 129], 6)
        tag = "bf16"
    out, fin = kda.chunk_fwd(*_x(d), d["init_state"], d["cu_seqlens"], chunk=64)
    torch.cuda.synchronize()
    assert torch.equal(fin, d["init_state"]), (
        f"{path}: final state moved by {(fin - d['init_state']).abs().max().item():.3e}")
    e = _check(out, fin, d, tag, f"{path} beta=0 g=0")
    # o_t = S_0^T q_t for the token's own sequence (closed form, no oracle).
    cu = d["cu_seqlens"].tolist()
    s0 = to64(d["init_state"])
    q = to64(d["q"])
    ref = np.zeros_like(to64(out))
    for n in range(len(cu) - 1):
        for t in range(cu[n], cu[n + 1]):
            ref[t] = np.einsum("hkv,hk->hv", s0[n], q[t])
    assert_close(out, ref, tag, f"{path} beta=0 g=0 out vs S0^T q")
    print(f"{path} beta=0 g=0: out err {e[0]:.3e}")


def test_beta0_g0_decode_passes_through():
    N, H = 4, 3
    gen = torch.Generator(device=DEV).manual_seed(8)
    state = inputs.draw_states(N, H, 128, 128, gen, DEV)
    s0 = state.clone()
    for s in range(5):
        q, k, v, g, beta = inputs.draw_token_tensors(N, H, 128, 128, torch.bfloat16, gen, DEV)
        out = kda.decode_step(q, k, v, torch.zeros_like(g), torch.zeros_like(beta), state)
    torch.cuda.synchronize()
    assert torch.equal(state, s0)


# --------------------------------------- orthonormal keys, beta = 1, g = 0: recall

def _recall_inputs(dtype, T, lag, seed):
    """Keys k_t = +-e_{pi(t)} (a signed permutation of the basis, repeated every
    128 tokens, so each key slot is overwritten once per cycle), beta = 1,
    g = 0, zero initial state, and queries q_t = k_{t - lag} (t >= lag): with
    orthonormal keys the write of token t replaces S^T k_t by v_t exactly, so
    o_t = v_{t - lag} whenever that key was not overwritten in between."""
    w = inputs.Workload("recall", heads=2, dk=128, dv=128, dtype=dtype, init_state=False)
    d = inputs.make_prefill(w, seed=200 + seed, device=DEV, lengths=[T])
    H = 2
    gen = torch.Generator().manual_seed(300 + seed)
    k = torch.zeros((T, H, 128), dtype=torch.float32)
    for h in range(H):
        perm = torch.randperm(128, generator=gen)
        sign = torch.where(torch.rand(128, generator=gen) < 0.5, -1.0, 1.0)
        for t in range(T):
            i = int(perm[t % 128])
            k[t, h, i] = sign[i]
    q = torch.zeros_like(k)
    q[lag:] = k[:T - lag]
    dt = d["q"].dtype
    d["k"] = k.to(DEV, dt)
    d["q"] = q.to(DEV, dt)
    d["g"] = torch.zeros_like(d["g"])
    d["beta"] = torch.ones_like(d["beta"])
    return d


@pytest.mark.parametrize("path", ["split", "fused", "fp32"])
def test_orthonormal_key_recall(path, monkeypatch):
    T, lag = 300, 5
    if path == "fp32":
        d = _recall_inputs("f32", T, lag, 9)
        tag = "f32"
    else:
        monkeypatch.setenv("KDA_CHUNK_PATH", path)
        d = _recall_inputs("bf16", T, lag, 9)
        tag = "bf16"
    out, fin = kda.chunk_fwd(*_x(d), None, d["cu_seqlens"], chunk=64)
    torch.cuda.synchronize()
    e = _check(out, fin, d, tag, f"{path} recall")
    # Recall: o_t = v_{t - lag} for t >= lag (keys repeat only after 128 tokens).
    got = to64(out)[lag:]
    want = to64(d["v"])[:T - lag]
    assert_close(got, want, tag, f"{path} recall o_t = v_(t-lag)")
    # Before any key is queried (t < lag) the query is zero, so is the output.
    assert float(np.abs(to64(out)[:lag]).max()) == 0.0
    print(f"{path} recall: oracle err {e[0]:.3e}, recall err {np.abs(got - want).max():.3e}")


def test_orthonormal_key_recall_decode():
    """The same recall through decode steps: write 40 pairs, then query each."""
    H = 2
    gen = torch.Generator().manual_seed(10)
    state = torch.zeros((1, H, 128, 128), dtype=torch.float32, device=DEV)
    perm = torch.randperm(128, generator=gen)[:40]
    vals = torch.randn((40, H, 128), generator=gen).to(torch.bfloat16)
    zeros_g = torch.zeros((1, H, 128), dtype=torch.bfloat16, device=DEV)
    ones_b = torch.ones((1, H), dtype=torch.bfloat16, device=DEV)
    for i in range(40):
        k = torch.zeros((1, H, 128), dtype=torch.bfloat16, device=DEV)
        k[0, :, perm[i]] = 1.0
        kda.decode_step(k, k, vals[i:i + 1].to(DEV), zeros_g, ones_b, state)
    # Reading with beta = 0 and a zero value leaves the state as it is.
    for i in range(40):
        q = torch.zeros((1, H, 128), dtype=torch.bfloat16, device=DEV)
        q[0, :, perm[i]] = 1.0
        o = kda.decode_step(q, q, torch.zeros_like(q), zeros_g, torch.zeros_like(ones_b), state)
        torch.cuda.synchronize()
        assert torch.equal(o.cpu(), vals[i:i + 1]), f"decode recall of pair {i}"
