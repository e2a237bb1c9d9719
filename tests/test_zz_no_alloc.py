"""kda_chunk_fwd_noalloc, the prefill entry point for callers that cannot
allocate device memory (an engine plugin that only receives pre-planned
buffers, a serving loop that must not call cudaMalloc).  Its outputs are
checked against the fp64 oracle, on two calls in a row, because every call
shares one scratch array inside the library: with several packed sequences
(the longest-first order in the array), with one sequence (no order needed),
and with 8,193 sequences (above the 8,192 that the longest-first sort serves,
the order written there is the identity).

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _noalloc_fn():
    lib = kda.load()
    fn = lib.kda_chunk_fwd_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.POINTER(kda._Dims),
                   vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(fn, d, chunk=64):
    T, H, dk = d["q"].shape
    dv = d["v"].shape[-1]
    N = d["cu_seqlens"].numel() - 1
    out = torch.empty((T, H, dv), dtype=d["q"].dtype, device=DEV)
    fin = torch.empty((N, H, dk, dv), dtype=torch.float32, device=DEV)
    dims = kda._Dims(N, T, H, dk, dv, kda._DTYPES[d["q"].dtype])
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = fn(p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]), p(d["beta"]), p(d["init_state"]),
            p(d["cu_seqlens"]), p(out), p(fin), chunk, ctypes.byref(dims), None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, kda.load().kda_status_string(rc)
    return out, fin


def _oracle(d):
    return oracle.prefill(*(d[n] for n in ("q", "k", "v", "g", "beta")), d["init_state"],
                          d["cu_seqlens"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_oracle_twice(dtype):
    fn = _noalloc_fn()
    tag = "bf16" if dtype == torch.bfloat16 else "f32"
    w = inputs.Workload("noalloc", heads=3, dk=128, dv=128, dtype=tag, init_state=True)
    # Two calls in a row with different sequence counts and lengths: the
    # second must not see anything the first left in the shared array.
    for seed, lengths in ((11, [130, 7, 0, 64, 300]), (12, [5, 65, 1, 190, 0, 64, 33, 129, 2])):
        d = inputs.make_prefill(w, seed=seed, device=DEV, lengths=lengths)
        out, fin = _call_noalloc(fn, d)
        torch.cuda.synchronize()
        ro, rf = _oracle(d)
        assert_close(out, ro, tag, "noalloc out vs oracle")
        assert_close(fin, rf, tag, "noalloc final_state vs oracle")


def test_noalloc_one_sequence():
    fn = _noalloc_fn()
    w = inputs.Workload("noalloc1", heads=2, dk=128, dv=128, dtype="bf16", init_state=True)
    d = inputs.make_prefill(w, seed=13, device=DEV, lengths=[517])
    out, fin = _call_noalloc(fn, d)
    torch.cuda.synchronize()
    ro, rf = _oracle(d)
    assert_close(out, ro, "bf16", "noalloc one-sequence out")
    assert_close(fin, rf, "bf16", "noalloc one-sequence final_state")


def test_noalloc_many_sequences_then_a_small_call():
    """8,193 sequences of 1 to 3 tokens (one head), one more than the
    longest-first sort serves; the next call, with few sequences, must not
    read what the big one left in the array."""
    fn = _noalloc_fn()
    w = inputs.Workload("noalloc_many", heads=1, dk=128, dv=128, dtype="bf16", init_state=True)
    rng = torch.Generator().manual_seed(14)
    lengths = (torch.randint(1, 4, (8193,), generator=rng)).tolist()
    d = inputs.make_prefill(w, seed=14, device=DEV, lengths=lengths)
    out, fin = _call_noalloc(fn, d)
    torch.cuda.synchronize()
    ro, rf = _oracle(d)
    assert_close(out, ro, "bf16", "noalloc 8193-sequence out")
    assert_close(fin, rf, "bf16", "noalloc 8193-sequence final_state")
    d = inputs.make_prefill(w, seed=15, device=DEV, lengths=[40, 3, 90])
    out, fin = _call_noalloc(fn, d)
    torch.cuda.synchronize()
    ro, rf = _oracle(d)
    assert_close(out, ro, "bf16", "noalloc small call after the big one: out")
    assert_close(fin, rf, "bf16", "noalloc small call after the big one: final_state")


def test_noalloc_rejects_too_many_sequences():
    fn = _noalloc_fn()
    n = 65536 + 1
    dims = kda._Dims(n, n, 1, 128, 128, kda.KDA_BF16)
    fake = ctypes.c_void_p(1 << 20)
    rc = fn(fake, fake, fake, fake, fake, None, fake, fake, None, 64, ctypes.byref(dims), None,
            None)
    assert rc == -7
