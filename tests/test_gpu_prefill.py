"""Prefill (kda_chunk_fwd) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = inputs.WORKLOADS


@pytest.fixture(params=["split", "fused"])
def tc_path(request, monkeypatch):
    """Both tensor-core forms: the split preparation + state kernels (the
    default for few sequence-head pairs) and the fused kernel."""
    monkeypatch.setenv("KDA_CHUNK_PATH", request.param)
    return request.param


def _run(d, chunk=64):
    out, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                             d["cu_seqlens"], chunk=chunk)
    torch.cuda.synchronize()
    return out, fin


def _oracle(d, heads=None):
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    s0 = d["init_state"]
    if heads is not None:
        hs = torch.tensor(heads, device=x[0].device)
        x = [t[:, hs] for t in x]
        s0 = None if s0 is None else s0[:, hs]
    return oracle.prefill(*x, s0, d["cu_seqlens"])


def test_oracle_scale_fp32_config():
    """B=1, H=1, T=256, dk=dv=64, fp32, zero state, chunk 64."""
    w = W["prefill_T256_H1_d64_f32"]
    d = inputs.make_prefill(w, seed=0, device=DEV)
    out, fin = _run(d)
    ro, rf = _oracle(d)
    assert_close(out, ro, "f32", "out")
    assert_close(fin, rf, "f32", "final_state")


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("lengths", [[300], [0, 1, 63, 64, 65, 129, 200]])
def test_bf16_ragged_and_varlen(lengths, chunk, tc_path):
    w = W["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=1, device=DEV, lengths=lengths, heads=3)
    out, fin = _run(d, chunk)
    ro, rf = _oracle(d)
    assert_close(out, ro, "bf16", "out")
    assert_close(fin, rf, "bf16", "final_state")


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128), (128, 128)])
def test_fp32_head_dims(dk, dv):
    w = inputs.Workload("f32_dims", heads=2, dk=dk, dv=dv, dtype="f32", init_state=True)
    d = inputs.make_prefill(w, seed=2, device=DEV, lengths=[70, 0, 33])
    out, fin = _run(d)
    ro, rf = _oracle(d)
    assert_close(out, ro, "f32", "out")
    assert_close(fin, rf, "f32", "final_state")


def test_empty_sequence_passes_state_through(tc_path):
    w = W["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=3, device=DEV, lengths=[0, 5, 0], heads=2)
    out, fin = _run(d)
    assert torch.equal(fin[0], d["init_state"][0]) and torch.equal(fin[2], d["init_state"][2])


def test_final_state_may_alias_init_state(tc_path):
    w = W["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=4, device=DEV, lengths=[90], heads=2)
    ref_out, ref_fin = _run(d)
    s = d["init_state"].clone()
    out, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], s, d["cu_seqlens"],
                             final_state=s)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(s, ref_fin)


def test_deterministic(tc_path):
    w = W["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=5, device=DEV, lengths=[200, 77], heads=4)
    o1, f1 = _run(d)
    o2, f2 = _run(d)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_prefill_8k_full_size(tc_path):
    """H=96, T=8192, bf16, random initial state: every head checked."""
    w = W["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=0, device=DEV)
    out, fin = _run(d)
    ro, rf = _oracle(d)
    assert_close(out, ro, "bf16", "out")
    assert_close(fin, rf, "bf16", "final_state")


def test_varlen_32seq_full_size_sampled():
    """32 packed sequences (~270K tokens), H=96: all outputs computed on the
    GPU, a sample of heads followed by the oracle over every sequence."""
    w = W["varlen_32seq_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=0, device=DEV)
    out, fin = _run(d)
    heads = [0, 61]
    ro, rf = _oracle(d, heads)
    hs = torch.tensor(heads, device=DEV)
    assert_close(out[:, hs], ro, "bf16", "out")
    assert_close(fin[:, hs], rf, "bf16", "final_state")


def test_prefill_1m_full_size_sampled():
    """T = 1,048,576, H=32, saturated a in [-8, 8]: one head followed by the
    oracle end to end (outputs and final state).  The split path runs it in
    windows of chunks (its record buffer is capped), carrying the state."""
    assert kda.algorithm(1, 1 << 20, 32, 128, 128) == "tcgen05_split"
    w = W["prefill_T1M_H32_d128_bf16"]
    d = inputs.make_prefill(w, seed=0, device=DEV)
    out, fin = _run(d)
    heads = [13]
    ro, rf = _oracle(d, heads)
    hs = torch.tensor(heads, device=DEV)
    assert_close(fin[:, hs], rf, "bf16", "final_state")
    assert_close(out[:, hs], ro, "bf16", "out")


@pytest.mark.parametrize("with_final", [True, False])
def test_split_windows_with_minimum_workspace(with_final):
    """The split path with a workspace that holds one record per pair: one
    chunk per window, the state carried between windows (in final_state, or
    in the workspace when no final state is asked for)."""
    w = W["prefill_T8192_H96_d128_bf16"]
    lengths = [300, 70, 0, 129, 64]
    d = inputs.make_prefill(w, seed=6, device=DEV, lengths=lengths, heads=3)
    N, H = len(lengths), 3
    order = (N * 4 + 255) // 256 * 256
    ws = torch.empty(order + N * H * 128 * 128 * 4 + N * H * 66048, dtype=torch.uint8,
                     device=DEV)
    out, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                             d["cu_seqlens"], chunk=64, workspace=ws,
                             output_final_state=with_final)
    torch.cuda.synchronize()
    ro, rf = _oracle(d)
    assert_close(out, ro, "bf16", "out")
    if with_final:
        assert_close(fin, rf, "bf16", "final_state")


def test_split_overlapped_windows_match_serial(monkeypatch):
    """The split form's overlapped windows (state passes on the library's
    helper stream beside the preparation of the next window) give exactly the
    results of the same kernels run one window after another."""
    monkeypatch.setenv("KDA_CHUNK_PATH", "split")
    w = W["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=7, device=DEV, lengths=[4000, 16384, 1500], heads=4)
    o1, f1 = _run(d)
    monkeypatch.setenv("KDA_SPLIT_SERIAL", "1")
    o2, f2 = _run(d)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    ro, rf = _oracle(d)
    assert_close(o1, ro, "bf16", "out")
    assert_close(f1, rf, "bf16", "final_state")


@pytest.mark.parametrize("tail", [None, "5"])
def test_split_front_loaded_windows_match_serial(monkeypatch, tail):
    """Pairs that fill more than half the SMs but fit in one wave run as two
    windows: the first (most chunks) prepared on every SM, its state pass
    beside the preparation of the short second one.  Results equal the
    serial single window bit for bit.  One sequence spans both windows; the
    other ends in the first and is carried through the second."""
    monkeypatch.setenv("KDA_CHUNK_PATH", "split")
    if tail is not None:
        monkeypatch.setenv("KDA_SPLIT_TAIL", tail)
    w = W["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=9, device=DEV, lengths=[5000, 100], heads=48)
    o1, f1 = _run(d)
    monkeypatch.setenv("KDA_SPLIT_SERIAL", "1")
    o2, f2 = _run(d)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    heads = [0, 17, 47]
    ro, rf = _oracle(d, heads)
    hs = torch.tensor(heads, device=DEV)
    assert_close(o1[:, hs], ro, "bf16", "out")
    assert_close(f1[:, hs], rf, "bf16", "final_state")


def test_launch_count_follows_the_window_schedule(monkeypatch):
    """kda_chunk_fwd_launch_count on the split form: front-loaded windows (two
    preparations, two state passes), one serial window, overlapped windows
    (a preparation and a state pass each)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    monkeypatch.delenv("KDA_SPLIT_SERIAL", raising=False)
    monkeypatch.delenv("KDA_SPLIT_TAIL", raising=False)
    H = sms * 5 // 8                                   # between half the SMs and all of them
    assert kda.launch_count(1, 8192, H, 128, 128) == 4
    monkeypatch.setenv("KDA_SPLIT_SERIAL", "1")
    assert kda.launch_count(1, 8192, H, 128, 128) == 2
    monkeypatch.delenv("KDA_SPLIT_SERIAL")
    # Few pairs, 2^20 tokens: overlapped windows, a preparation and a state
    # pass each; the same pairs and windows from two sequences add the
    # length-order kernel.
    c1 = kda.launch_count(1, 1 << 20, 32, 128, 128)
    assert c1 >= 4 and c1 % 2 == 0
    assert kda.launch_count(2, 1 << 20, 16, 128, 128, varlen=True) == c1 + 1


@pytest.mark.parametrize("lengths,heads", [([8192], 96), ([4096], 8), ([3000, 700], 8)])
def test_launch_count_matches_the_kernels_launched(lengths, heads, monkeypatch):
    """kda.launch_count (the figure bench.py reports as gpu_launches) equals
    the library kernels one kda_chunk_fwd call launches, counted by the
    PyTorch profiler's device activity: front-loaded windows (96 heads), one
    serial window (8 heads), and packed sequences (the length-order kernel
    too)."""
    from torch.profiler import ProfilerActivity, profile
    monkeypatch.delenv("KDA_SPLIT_SERIAL", raising=False)
    monkeypatch.delenv("KDA_CHUNK_PATH", raising=False)
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=11, device=DEV,
                            lengths=lengths, heads=heads)
    N, T = len(lengths), sum(lengths)
    cu = d["cu_seqlens"] if N > 1 else None
    run = lambda: kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], cu,
                                chunk=64, n_seqs=N)
    run()
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]):   # the profiler's first session may
        torch.ones(1, device=DEV).add_(1)              # miss kernels: warm it up
        torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        run()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if "kda::" in e.name or "chunk_" in e.name
             or "order_kernel" in e.name]
    if not names:
        pytest.skip("the profiler recorded no device kernels here")
    assert len(names) == kda.launch_count(N, T, heads, 128, 128, varlen=N > 1), names


def test_split_many_pairs_few_sequences_windows():
    """More than 304 sequence-head pairs from few sequences take the split form
    by default; with a workspace a few records per pair larger than the
    minimum the input runs in several windows, the state carried between
    them."""
    w = W["prefill_T8192_H96_d128_bf16"]
    lengths = [700, 64, 1, 450, 0, 513, 129, 300]
    N, H = len(lengths), 40
    assert kda.algorithm(N, sum(lengths), H, 128, 128) == "tcgen05_split"
    d = inputs.make_prefill(w, seed=8, device=DEV, lengths=lengths, heads=H)
    order = (N * 4 + 255) // 256 * 256
    ws = torch.empty(order + N * H * 128 * 128 * 4 + 3 * N * H * 66048, dtype=torch.uint8,
                     device=DEV)
    out, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                             d["cu_seqlens"], chunk=64, workspace=ws)
    torch.cuda.synchronize()
    heads = [0, 17, 39]
    ro, rf = _oracle(d, heads)
    hs = torch.tensor(heads, device=DEV)
    assert_close(fin[:, hs], rf, "bf16", "final_state")
    assert_close(out[:, hs], ro, "bf16", "out")
