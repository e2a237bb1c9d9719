"""Failure detection on the GPU without a fault: the library's bounded
mbarrier wait, on a barrier nothing arrives at, gives up after its limit,
reports KDA_ERR_TIMEOUT through dev_status and leaves the context usable."""
import time

import pytest
import torch

import hybrid_linear_attention_02_gb300 as kda
import oracle
from hybrid_linear_attention_02_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
KDA_ERR_TIMEOUT = -4


def test_expired_wait_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kda.debug_wait_timeout(status, 50_000)   # 50 ms limit
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == KDA_ERR_TIMEOUT
    assert 0.04 < elapsed < 5.0, elapsed
    # The context still works: a small prefill matches the oracle.
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=9, device=DEV, lengths=[130, 64], heads=2)
    out, fin = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                             d["cu_seqlens"], chunk=64)
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                            d["cu_seqlens"])
    assert_close(out, ro, "bf16", "out")
    assert_close(fin, rf, "bf16", "final_state")


def test_wait_timeout_argument_checks():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(kda.KDAError):
        kda.debug_wait_timeout(status, 0)
    with pytest.raises(kda.KDAError):
        kda.debug_wait_timeout(status, 20_000_000)


@pytest.mark.parametrize("which", [1, 2, 3])
def test_production_kernel_gives_up_and_reports(which, monkeypatch):
    """The production prefill kernels' own abort path: one copy is never issued
    (1: the split state kernel's first record; 2: the split preparation
    kernel's first raw tiles; 3: the fused kernel's first raw tiles).  Every
    role of the block must give up within the bounded wait (about 2 s), report
    KDA_ERR_TIMEOUT through dev_status and free its resources; afterwards a
    normal prefill on both tensor-core forms still matches the oracle."""
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=19, device=DEV, lengths=[128], heads=2)   # 1 pair x 2 chunks
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kda.debug_chunk_fwd_withhold(which, *x, d["init_state"], status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == KDA_ERR_TIMEOUT, (which, int(status.item()))
    assert 1.0 < elapsed < 20.0, elapsed
    for path in ("split", "fused"):
        monkeypatch.setenv("KDA_CHUNK_PATH", path)
        out, fin = kda.chunk_fwd(*x, d["init_state"], d["cu_seqlens"], chunk=64)
        torch.cuda.synchronize()
        ro, rf = oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
        assert_close(out, ro, "bf16", f"{path} out after the self-test")
        assert_close(fin, rf, "bf16", f"{path} final_state after the self-test")
