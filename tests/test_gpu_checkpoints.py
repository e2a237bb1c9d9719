"""Prefix-cache checkpoints (kda_chunk_fwd_checkpoints) against the fp64
oracle: the state after every `interval` tokens of each sequence, on the
tensor-core path (bf16, d = 128) and the CUDA-core path (fp32, d = 64)."""
import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _both(d, interval):
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    out, fin, ck = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64,
                                 ckpt_interval=interval)
    torch.cuda.synchronize()
    ro, rf, rck = oracle.prefill(*x, d["init_state"], d["cu_seqlens"], ckpt_interval=interval)
    return (out, fin, ck), (ro, rf, rck)


# Lengths cover: empty, shorter than one interval, exact multiples, a ragged
# tail after full intervals, and a final chunk that is itself partial.
LENGTHS = [0, 63, 64, 512, 700, 1024, 129, 1]


@pytest.fixture(params=["split", "fused"])
def tc_path(request, monkeypatch):
    monkeypatch.setenv("KDA_CHUNK_PATH", request.param)
    return request.param


@pytest.mark.parametrize("interval", [64, 128, 512])
def test_checkpoints_tensor_core_path_bf16(interval, tc_path):
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=21, device=DEV, lengths=LENGTHS, heads=3)
    assert kda.algorithm(len(LENGTHS), sum(LENGTHS), 3, 128, 128).startswith("tcgen05")
    (out, fin, ck), (ro, rf, rck) = _both(d, interval)
    n_ck = sum(n // interval for n in LENGTHS)
    assert rck.shape[0] == n_ck and ck.shape[0] == n_ck
    assert_close(out, ro, "bf16", "out")
    assert_close(fin, rf, "bf16", "final_state")
    assert_close(ck, rck, "bf16", "checkpoints")


def test_checkpoints_cuda_core_path_f32():
    w = inputs.Workload("ck_f32", heads=2, dk=64, dv=64, dtype="f32", init_state=True)
    lengths = [130, 0, 64, 257, 5]
    d = inputs.make_prefill(w, seed=22, device=DEV, lengths=lengths)
    (out, fin, ck), (ro, rf, rck) = _both(d, 64)
    assert ck.shape[0] == sum(n // 64 for n in lengths)
    assert_close(out, ro, "f32", "out")
    assert_close(fin, rf, "f32", "final_state")
    assert_close(ck, rck, "f32", "checkpoints")


def test_checkpoints_leave_outputs_unchanged_and_end_on_final_state():
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    lengths = [512, 300, 1024]
    d = inputs.make_prefill(w, seed=23, device=DEV, lengths=lengths, heads=2)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    out0, fin0 = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64)
    out1, fin1, ck = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64,
                                   ckpt_interval=256)
    torch.cuda.synchronize()
    # Writing checkpoints is a side output: the same kernel, the same results.
    assert torch.equal(out0, out1) and torch.equal(fin0, fin1)
    offs = kda.checkpoint_offsets(lengths, 256)
    assert offs == [0, 2, 3, 7]
    # A sequence whose length is a multiple of the interval ends on its final state.
    assert torch.equal(ck[offs[1] - 1], fin1[0])
    assert torch.equal(ck[offs[3] - 1], fin1[2])


def test_checkpoints_resume_matches_uninterrupted_prefill():
    """Restarting from a checkpoint (the prefix-cache hit) gives the same
    output and final state as running the whole sequence."""
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=24, device=DEV, lengths=[900], heads=2)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    out, fin, ck = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64,
                                 ckpt_interval=512)
    tail = [t[512:].contiguous() for t in x]
    cu = torch.tensor([0, 388], dtype=torch.int32, device=DEV)
    out2, fin2 = kda.chunk_fwd(*tail, ck[0:1].contiguous(), cu, chunk=64)
    torch.cuda.synchronize()
    assert_close(out2, out[512:], "bf16", "resumed out")
    assert_close(fin2, fin, "bf16", "resumed final_state")


def test_checkpoints_front_loaded_windows_match_serial(monkeypatch):
    """96 sequence-head pairs run as front-loaded windows on the split form;
    the checkpoints, outputs and final states equal those of one serial
    window bit for bit, and the oracle's on three heads.  The first sequence
    spans both windows, so the second window's checkpoints continue the
    state the first one carried over."""
    monkeypatch.setenv("KDA_CHUNK_PATH", "split")
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=25, device=DEV, lengths=[5000, 100], heads=48)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]

    def run():
        r = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64, ckpt_interval=128)
        torch.cuda.synchronize()
        return r

    a = run()
    monkeypatch.setenv("KDA_SPLIT_SERIAL", "1")
    b = run()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    heads = [0, 31, 47]
    hs = torch.tensor(heads, device=DEV)
    ro, rf, rck = oracle.prefill(*[t[:, hs] for t in x], d["init_state"][:, hs],
                                 d["cu_seqlens"], ckpt_interval=128)
    assert_close(a[0][:, hs], ro, "bf16", "out")
    assert_close(a[1][:, hs], rf, "bf16", "final_state")
    assert_close(a[2][:, hs], rck, "bf16", "checkpoints")
