"""Output epilogue (head-wise RMSNorm, then the full-rank sigmoid gate):
kda_chunk_fwd_gated on every prefill path and kda_decode_step_gated, against
the fp64 oracle's recurrence followed by its epilogue.  Each case also checks
the gated result against the oracle's epilogue applied to the same call's
ungated GPU output, which pins the epilogue kernels alone."""
import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close, assert_close_gated, to64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = inputs.WORKLOADS


def _epilogue_only(got, o_gpu, gate, tag):
    """The gated output equals the oracle epilogue of the GPU's own o up to
    the epilogue's arithmetic (fp32 math on the rounded o, then one rounding)."""
    ref = oracle.output_gate(to64(o_gpu), *gate)
    tol = 1e-5 if tag == "f32" else 2.0 ** -7
    err = abs(to64(got) - ref).max() / max(abs(ref).max(), 1e-30)
    assert err <= tol, f"epilogue vs own output: {err:.3e} > {tol}"


def _check(d, tag, chunk=64):
    T, H, _ = d["q"].shape
    dv = d["v"].shape[-1]
    gate = inputs.make_output_gate(T, H, dv, d["v"].dtype, seed=3, device=DEV)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    o0, _ = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=chunk)
    out, fin = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=chunk, gate=gate)
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
    assert_close_gated(out, ro, gate, tag, "gated out")
    assert_close(fin, rf, tag, "final_state")
    _epilogue_only(out, o0, gate, tag)


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("lengths", [[300, 0, 64, 129, 1], [0, 1, 63, 64, 65, 129, 200]])
def test_gated_prefill_tensor_core(path, lengths, monkeypatch):
    monkeypatch.setenv("KDA_CHUNK_PATH", path)
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=31, device=DEV,
                            lengths=lengths, heads=3)
    _check(d, "bf16")


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128)])
def test_gated_prefill_cuda_core_f32(dk, dv):
    w = inputs.Workload("gate_f32", heads=2, dk=dk, dv=dv, dtype="f32", init_state=True)
    d = inputs.make_prefill(w, seed=32, device=DEV, lengths=[70, 0, 33])
    _check(d, "f32")


def test_gated_prefill_full_size():
    """The headline workload (T=8192, H=96) through the default path."""
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=0, device=DEV)
    _check(d, "bf16")


def test_gated_front_loaded_windows_match_serial(monkeypatch):
    """96 sequence-head pairs run as front-loaded windows on the split form;
    the gated state pass gives the serial single window's results bit for bit
    (the gate tiles of the second window's chunks included)."""
    monkeypatch.setenv("KDA_CHUNK_PATH", "split")
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=34, device=DEV,
                            lengths=[5000, 100], heads=48)
    T, H, dv = d["v"].shape
    gate = inputs.make_output_gate(T, H, dv, d["v"].dtype, seed=4, device=DEV)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    run = lambda: kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64, gate=gate)
    o1, f1 = run()
    monkeypatch.setenv("KDA_SPLIT_SERIAL", "1")
    o2, f2 = run()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_gated_decode_chain():
    wd = W["decode_256seq_H96_d128_64steps"]
    N, H = 8, 4
    state = inputs.make_decode_state(wd, seed=33, device=DEV, n_seqs=N, heads=H)
    plain_state = state.clone()
    ref_state = state.clone()
    for step in range(3):
        toks = inputs.make_decode_tokens(wd, step, seed=33, device=DEV, n_seqs=N, heads=H)
        gate = inputs.make_output_gate(N, H, wd.dv, wd.torch_dtype, seed=step, device=DEV)
        out = kda.decode_step(*toks, state, gate=gate)
        o0 = kda.decode_step(*toks, plain_state)
        torch.cuda.synchronize()
        ro, ref_state = oracle.decode(*toks, ref_state)
        assert_close_gated(out, ro, gate, "bf16", f"gated decode out step {step}")
        assert_close(state, ref_state, "bf16", f"decode state step {step}")
        assert torch.equal(state, plain_state)
        _epilogue_only(out, o0, gate, "bf16")


def test_gated_split_windows():
    """The split form's gated state pass across several windows (a workspace
    three records per pair above the minimum), overlapped with the next
    window's preparation: inside a window a full chunk's epilogue runs during
    the next chunk's MMA2, and every window's last chunk finishes in place."""
    lengths = [700, 64, 1, 450, 0, 513, 129, 300]
    N, H = len(lengths), 3
    d = inputs.make_prefill(W["prefill_T8192_H96_d128_bf16"], seed=34, device=DEV,
                            lengths=lengths, heads=H)
    assert kda.algorithm(N, sum(lengths), H, 128, 128) == "tcgen05_split"
    order = (N * 4 + 255) // 256 * 256
    ws = torch.empty(order + N * H * 128 * 128 * 4 + 3 * N * H * 66048, dtype=torch.uint8,
                     device=DEV)
    gate = inputs.make_output_gate(sum(lengths), H, 128, d["v"].dtype, seed=4, device=DEV)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    o0, _ = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64, workspace=ws)
    out, fin = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64, workspace=ws,
                             gate=gate)
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
    assert_close_gated(out, ro, gate, "bf16", "gated out")
    assert_close(fin, rf, "bf16", "final_state")
    _epilogue_only(out, o0, gate, "bf16")
