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
