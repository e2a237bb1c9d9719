"""The inputs' range precondition on the device (kda_check_inputs, and the
KDA_DEBUG_BOUNDS build that runs it inside every prefill and decode call).

The bound is the lower-bounded decay of "[Paper Review] Kimi K3: Open
Frontier Intelligence", section "Kimi Delta Attention (KDA)": g = g_min
sigmoid(.) with g_min = -5 keeps g in [-5, 0]; beta lies in [0, 1].  A value
outside is reported as KDA_ERR_RANGE through dev_status; nothing traps, and
the context stays usable.
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
KDA_ERR_RANGE = -8


def _case(dtype=torch.bfloat16, T=200, H=3):
    w = inputs.Workload("range", heads=H, dk=128, dv=128,
                        dtype="bf16" if dtype == torch.bfloat16 else "f32")
    return inputs.make_prefill(w, seed=31, device=DEV, lengths=[T])


def _status_after(g, beta):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.check_inputs(g, beta, st)
    torch.cuda.synchronize()
    return int(st.item())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_check_inputs_flags_each_violation(dtype):
    d = _case(dtype)
    g, beta = d["g"], d["beta"]
    assert _status_after(g, beta) == 0
    # The bound itself is inside: g = -5 and g = 0 exactly, beta = 0 and 1.
    assert _status_after(torch.full_like(g, -5.0), torch.ones_like(beta)) == 0
    assert _status_after(torch.zeros_like(g), torch.zeros_like(beta)) == 0
    for where, val in (((7, 1, 5), -5.25), ((199, 2, 127), 0.5), ((0, 0, 0), float("nan"))):
        bad = g.clone()
        bad[where] = val
        assert _status_after(bad, beta) == KDA_ERR_RANGE, (where, val)
    bad_b = beta.clone()
    bad_b[100, 1] = 1.5
    assert _status_after(g, bad_b) == KDA_ERR_RANGE
    bad_b[100, 1] = -0.25
    assert _status_after(g, bad_b) == KDA_ERR_RANGE
    # An earlier error code is kept.
    st = torch.full((1,), -4, dtype=torch.int32, device=DEV)
    bad = g.clone()
    bad[3, 0, 3] = 1.0
    kda.check_inputs(bad, beta, st)
    torch.cuda.synchronize()
    assert int(st.item()) == -4


def _raw_prefill(lib, d, out, fin, st):
    T, H, dk = d["q"].shape
    dims = kda._Dims(1, T, H, dk, dk, kda._DTYPES[d["q"].dtype])
    need = int(lib.kda_chunk_fwd_workspace_size(ctypes.byref(dims), 64))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = lib.kda_chunk_fwd(p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]), p(d["beta"]),
                           p(d["init_state"]), None, p(out), p(fin), 64, ctypes.byref(dims),
                           p(ws), need, p(st),
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    return ws


def test_debug_bounds_build_reports_range_inside_the_call():
    lib = kda.load_debug_bounds()
    assert lib.kda_debug_bounds_build() == 1
    d = _case()
    T, H = d["q"].shape[:2]
    out = torch.empty_like(d["v"])
    fin = torch.empty_like(d["init_state"])
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _raw_prefill(lib, d, out, fin, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rf = oracle.prefill(*(d[n] for n in ("q", "k", "v", "g", "beta")), d["init_state"],
                            d["cu_seqlens"])
    assert_close(out, ro, "bf16", "debug build out")
    assert_close(fin, rf, "bf16", "debug build final_state")
    # One out-of-range decay: reported, the call still completes.
    d["g"][50, 2, 17] = -6.0
    _raw_prefill(lib, d, out, fin, st)
    torch.cuda.synchronize()
    assert int(st.item()) == KDA_ERR_RANGE
    assert torch.isfinite(out.float()).all()
    # Decode in the debug build: beta above 1 is reported.
    st.zero_()
    N = 4
    gen = torch.Generator(device=DEV).manual_seed(32)
    state = inputs.draw_states(N, H, 128, 128, gen, DEV)
    q, k, v, g, beta = inputs.draw_token_tensors(N, H, 128, 128, torch.bfloat16, gen, DEV)
    beta[2, 1] = 1.25
    dims = kda._Dims(N, N, H, 128, 128, kda.KDA_BF16)
    o = torch.empty_like(v)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.kda_decode_step(p(q), p(k), p(v), p(g), p(beta), p(state), p(o), ctypes.byref(dims),
                             p(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == KDA_ERR_RANGE
