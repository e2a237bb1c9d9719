"""Decode step (kda_decode_step) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
WD = inputs.WORKLOADS["decode_256seq_H96_d128_64steps"]


def _tokens(step, n, h, dk, dv, dtype, seed=0):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(1000 + seed * 97 + step)
    return inputs.draw_token_tensors(n, h, dk, dv, dtype, gen, DEV)


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 64),
                                         (torch.float32, 128, 64), (torch.float32, 64, 128),
                                         (torch.bfloat16, 64, 128)])
def test_decode_chain_small(dtype, dk, dv):
    N, H, steps = 5, 3, 4
    gen = torch.Generator(device=DEV)
    gen.manual_seed(7)
    state = inputs.draw_states(N, H, dk, dv, gen, DEV)
    ref_state = state.cpu().double().numpy()
    tag = "f32" if dtype == torch.float32 else "bf16"
    for s in range(steps):
        q, k, v, g, beta = _tokens(s, N, H, dk, dv, dtype)
        out = kda.decode_step(q, k, v, g, beta, state)
        torch.cuda.synchronize()
        ro, ref_state = oracle.decode(q, k, v, g, beta, ref_state)
        assert_close(out, ro, tag, f"decode out step {s}")
        assert_close(state, ref_state, tag, f"decode state step {s}")


def test_decode_full_size_sampled():
    """256 sequences x 96 heads, 64 chained steps in the benchmark's launch
    configuration; a sample of (sequence, head) pairs is followed by the oracle."""
    state = inputs.make_decode_state(WD, seed=0, device=DEV)
    pairs = [(0, 0), (17, 5), (128, 95), (255, 40)]
    ns = torch.tensor([p[0] for p in pairs], device=DEV)
    hs = torch.tensor([p[1] for p in pairs], device=DEV)
    ref_state = state[ns, hs].cpu().double().numpy()[:, None]      # [P, 1, dk, dv]
    for s in range(WD.decode_steps):
        q, k, v, g, beta = inputs.make_decode_tokens(WD, s, seed=0, device=DEV)
        out = kda.decode_step(q, k, v, g, beta, state)
        sel = [x[ns, hs][:, None] for x in (q, k, v, g, beta)]
        ro, ref_state = oracle.decode(*sel, ref_state)
        if s % 16 == 15 or s == 0:
            torch.cuda.synchronize()
            assert_close(out[ns, hs][:, None], ro, "bf16", f"decode full out step {s}")
    torch.cuda.synchronize()
    assert_close(state[ns, hs][:, None], ref_state, "bf16", "decode full final state")


def test_decode_deterministic():
    N, H = 8, 4
    gen = torch.Generator(device=DEV)
    gen.manual_seed(3)
    s1 = inputs.draw_states(N, H, 128, 128, gen, DEV)
    s2 = s1.clone()
    q, k, v, g, beta = _tokens(0, N, H, 128, 128, torch.bfloat16)
    o1 = kda.decode_step(q, k, v, g, beta, s1)
    o2 = kda.decode_step(q, k, v, g, beta, s2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
