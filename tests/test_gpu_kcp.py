"""KCP building blocks on the GPU: segment transitions (kda_chunk_transition),
their application and composition (kda_transition_apply), and the
single-GPU KCP prefill (kda_chunk_fwd_kcp), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = inputs.WORKLOADS


def _oracle_transition(x, cu):
    q, k, v, g, b = x
    N = cu.numel() - 1
    H, dk = q.shape[1], q.shape[2]
    eye = np.broadcast_to(np.eye(dk), (N, H, dk, dk)).copy()
    _, M = oracle.prefill(q, k, torch.zeros_like(v), g, b, eye, cu)
    _, Hs = oracle.prefill(q, k, v, g, b, None, cu)
    return M, Hs


@pytest.mark.parametrize("lengths", [[130, 0, 64, 300], [1000]])
def test_transitions_match_oracle(lengths):
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=51, device=DEV,
                            lengths=lengths, heads=2)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    M, Hs = kda.chunk_transition(*x, d["cu_seqlens"])
    torch.cuda.synchronize()
    rM, rH = _oracle_transition(x, d["cu_seqlens"])
    assert_close(M, rM, "bf16", "M")
    assert_close(Hs, rH, "bf16", "H")
    # An empty segment maps every state to itself.
    for n, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(M[n], torch.eye(128, device=DEV).expand(2, 128, 128))
            assert torch.count_nonzero(Hs[n]) == 0


def test_transition_apply_and_compose():
    gen = torch.Generator(device=DEV)
    gen.manual_seed(52)
    shape = (3, 4, 128, 128)
    M1, M2, H1, H2, S = (torch.randn(shape, generator=gen, device=DEV) * 0.1 for _ in range(5))
    y = kda.transition_apply(M1, H1, S)
    ref = to64(M1) @ to64(S) + to64(H1)
    assert_close(y, ref, "f32", "M S + H")
    # (M2, H2) after (M1, H1) = (M2 M1, M2 H1 + H2), and applying it equals two steps.
    M12 = kda.transition_apply(M2, None, M1)
    H12 = kda.transition_apply(M2, H2, H1)
    two = kda.transition_apply(M2, H2, kda.transition_apply(M1, H1, S))
    one = kda.transition_apply(M12, H12, S)
    torch.cuda.synchronize()
    assert_close(one, to64(two), "f32", "composed map")


@pytest.mark.parametrize("n_seqs,segments", [(1, 3), (1, 4), (2, 3)])
def test_kcp_prefill_matches_oracle(n_seqs, segments):
    T = 2560 * n_seqs
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=53, device=DEV,
                            lengths=[T // n_seqs] * n_seqs, heads=4)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    out, fin = kda.chunk_fwd_kcp(*x, d["init_state"], n_seqs=n_seqs, segments=segments)
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
    assert_close(out, ro, "bf16", "kcp out")
    assert_close(fin, rf, "bf16", "kcp final_state")


def _slow_decay(d, seed):
    """g in [-0.05, 0]: over segments of up to 64 tokens M stays of order one
    (at the generator's decay it falls below 1e-10 and any small M passes)."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    d["g"] = (-0.05 * torch.rand(d["g"].shape, generator=gen, device=DEV)).to(d["g"].dtype)
    return d


def _assert_scaled(got, ref, what):
    """bf16 bound with the absolute floor scaled to the tensor's size:
    |x - ref| <= 2e-2 |ref| + 1e-2 max|ref|."""
    got, ref = to64(got), to64(ref)
    scale = float(np.abs(ref).max())
    # At the generator's decay max|M| falls below 1e-10; at this decay it is
    # of order 0.1 - 1, so the scaled floor is a real bound.
    assert scale > 0.05, f"{what}: max|ref| = {scale:.3e}, the check would be vacuous"
    err = np.abs(got - ref)
    excess = err - (2e-2 * np.abs(ref) + 1e-2 * scale)
    assert excess.max() <= 0, f"{what}: max |err| {err.max():.3e} (max|ref| {scale:.3e})"
    return float(err.max())


@pytest.mark.parametrize("lengths", [[1, 17, 64, 33, 0, 50], [64, 2, 63]])
def test_transitions_at_slow_decay_match_oracle_elementwise(lengths):
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=54, device=DEV,
                            lengths=lengths, heads=2)
    _slow_decay(d, 540)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    M, Hs = kda.chunk_transition(*x, d["cu_seqlens"])
    torch.cuda.synchronize()
    rM, rH = _oracle_transition(x, d["cu_seqlens"])
    for n, L in enumerate(lengths):
        if L == 0:
            continue
        eM = _assert_scaled(M[n], rM[n], f"M of segment {n} ({L} tokens)")
        eH = _assert_scaled(Hs[n], rH[n], f"H of segment {n} ({L} tokens)")
        print(f"segment {n} ({L} tokens): M err {eM:.3e}, H err {eH:.3e}, "
              f"max|M| {np.abs(rM[n]).max():.3f}")
    # A wrong M would move the composed state: M S + H against the oracle's end state.
    s0 = torch.randn((len(lengths), 2, 128, 128), device=DEV) * 0.02
    y = kda.transition_apply(M, Hs, s0)
    _, rf = oracle.prefill(*x, s0, d["cu_seqlens"])
    torch.cuda.synchronize()
    assert_close(y, rf, "bf16", "M S0 + H vs the oracle's end state")


@pytest.mark.parametrize("segments", [3, 8])
def test_kcp_prefill_at_slow_decay_matches_oracle(segments):
    """At slow decay every segment's entry state depends on all earlier ones
    through M, so the composition is exercised."""
    T = 2048
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=55, device=DEV,
                            lengths=[T], heads=3)
    _slow_decay(d, 550)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    out, fin = kda.chunk_fwd_kcp(*x, d["init_state"], n_seqs=1, segments=segments)
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
    eo = assert_close(out, ro, "bf16", "kcp slow-decay out")
    ef = assert_close(fin, rf, "bf16", "kcp slow-decay final_state")
    print(f"kcp {segments} segments, slow decay: out err {eo:.3e}, final err {ef:.3e}")


def test_transitions_full_headline_size_sampled():
    """One 8192-token sequence x 96 heads (the launch configuration the bench's
    transition leg times: 192 state CTAs for the M and H maps, more than the
    SMs hold at once): two heads' maps against the oracle."""
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=56, device=DEV)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    M, Hs = kda.chunk_transition(*x, d["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.isfinite(M).all() and torch.isfinite(Hs).all()
    heads = [7, 90]
    hs = torch.tensor(heads, device=DEV)
    rM, rH = _oracle_transition([t[:, hs] for t in x], d["cu_seqlens"])
    assert_close(M[:, hs], rM, "bf16", "M (8192 tokens)")
    assert_close(Hs[:, hs], rH, "bf16", "H (8192 tokens)")
