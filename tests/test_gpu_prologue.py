"""The input prologue (kda_prologue) against the fp64 oracle, and the whole
path from pre-activations: prologue then chunkwise prefill."""
import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("dtype,tag", [(torch.bfloat16, "bf16"), (torch.float32, "f32")])
@pytest.mark.parametrize("dk", [64, 128])
def test_prologue_matches_oracle(dtype, tag, dk):
    lengths = [0, 1, 2, 3, 5, 130, 64]
    T, H = sum(lengths), 3
    cu = inputs.cu_from_lengths(lengths).to(DEV)
    x = inputs.make_prologue_inputs(T, H, dk, dtype, seed=71, device=DEV)
    q, k, g = kda.prologue(*x, cu)
    torch.cuda.synchronize()
    rq, rk, rg = oracle.prologue(*x, cu)
    assert_close(q, rq, tag, "q")
    assert_close(k, rk, tag, "k")
    assert_close(g, rg, tag, "g")
    assert float(g.float().max()) < 0 and float(g.float().min()) >= -5.0


def test_prologue_equal_length_sequences():
    T, H, dk = 4 * 96, 2, 128
    x = inputs.make_prologue_inputs(T, H, dk, torch.bfloat16, seed=72, device=DEV)
    q, k, g = kda.prologue(*x, None, n_seqs=4)
    cu = torch.tensor([0, 96, 192, 288, 384], dtype=torch.int32)
    rq, rk, rg = oracle.prologue(*x, cu)
    assert_close(q, rq, "bf16", "q")
    assert_close(k, rk, "bf16", "k")
    assert_close(g, rg, "bf16", "g")


def test_projections_to_outputs():
    """Pre-activations -> prologue -> kda_chunk_fwd, against the oracle's
    prologue and recurrence in fp64."""
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    lengths = [700, 64, 3]
    d = inputs.make_prefill(w, seed=73, device=DEV, lengths=lengths, heads=2)
    T = sum(lengths)
    x = inputs.make_prologue_inputs(T, 2, 128, torch.bfloat16, seed=73, device=DEV)
    q, k, g = kda.prologue(*x, d["cu_seqlens"])
    out, fin = kda.chunk_fwd(q, k, d["v"], g, d["beta"], d["init_state"], d["cu_seqlens"])
    torch.cuda.synchronize()
    rq, rk, rg = oracle.prologue(*x, d["cu_seqlens"])
    ro, rf = oracle.prefill(torch.from_numpy(rq), torch.from_numpy(rk),
                            d["v"].cpu().double(), torch.from_numpy(rg),
                            d["beta"].cpu().double(), d["init_state"], d["cu_seqlens"])
    assert_close(out, ro, "bf16", "out")
    assert_close(fin, rf, "bf16", "final_state")


@pytest.mark.parametrize("dk", [64, 128])
def test_prologue_long_varlen_partial_head_block(dk):
    """A long varlen input (sequence starts inside and between token blocks,
    an empty sequence) with a head count that is not a multiple of the
    heads per block."""
    lengths = [4099, 1, 4000, 0, 97]
    T, H = sum(lengths), 10
    cu = inputs.cu_from_lengths(lengths).to(DEV)
    x = inputs.make_prologue_inputs(T, H, dk, torch.bfloat16, seed=74, device=DEV)
    q, k, g = kda.prologue(*x, cu)
    torch.cuda.synchronize()
    rq, rk, rg = oracle.prologue(*x, cu)
    assert_close(q, rq, "bf16", "q")
    assert_close(k, rk, "bf16", "k")
    assert_close(g, rg, "bf16", "g")
