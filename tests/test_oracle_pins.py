"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics.

None of these tests call the CUDA library.  Each pin is chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign or index, the decay
applied after the write, a transposed state) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, T, H, dk, dv, g_scale=1.0, unit_k=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((T, H, dk)))) * g_scale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


def _bruteforce(q, k, v, g, beta, S0):
    """Explicit per-token transition matrices: S_t = M_t S_{t-1} + beta k v^T,
    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t); o_t = S_t^T q_t (one head)."""
    T, dk = q.shape
    S = S0.copy()
    outs = []
    for t in range(T):
        M = (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        S = M @ S + beta[t] * np.outer(k[t], v[t])
        outs.append(S.T @ q[t])
    return np.array(outs), S


def test_hand_worked_example():
    """Two tokens worked by hand (derivation stored in the fixture)."""
    ex = json.load(open(os.path.join(GOLDEN, "kda_hand_example.json")))
    arr = {n: np.array(ex[n], dtype=np.float64) for n in ("q", "k", "v", "g", "beta")}
    out, fin = oracle.prefill(arr["q"], arr["k"], arr["v"], arr["g"], arr["beta"])
    np.testing.assert_allclose(out, np.array(ex["out"]), rtol=0, atol=ex["tolerance"])
    np.testing.assert_allclose(fin, np.array(ex["final_state"]), rtol=0, atol=ex["tolerance"])


@pytest.mark.parametrize("dk,dv", [(3, 5), (8, 8), (6, 2)])
def test_bruteforce_transition_matrices(dk, dv):
    rng = np.random.default_rng(dk * 100 + dv)
    T, H = 11, 2
    q, k, v, g, beta = _rand_case(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0)
    for h in range(H):
        o_ref, s_ref = _bruteforce(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], S0[0, h])
        np.testing.assert_allclose(out[:, h], o_ref, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(fin[0, h], s_ref, rtol=1e-13, atol=1e-13)


def test_beta0_g0_leaves_state_unchanged():
    rng = np.random.default_rng(1)
    T, H, dk, dv = 9, 3, 5, 4
    q, k, v, _, _ = _rand_case(rng, T, H, dk, dv)
    g = np.zeros((T, H, dk))
    beta = np.zeros((T, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0)
    assert np.array_equal(fin, S0)
    for h in range(H):
        np.testing.assert_allclose(out[:, h], q[:, h] @ S0[0, h], rtol=1e-14, atol=1e-14)


def test_beta0_closed_form_decay():
    """beta = 0: S_t = Diag(exp(sum_{s<=t} g_s)) S_0 exactly, o_t = S_t^T q_t."""
    rng = np.random.default_rng(2)
    T, H, dk, dv = 13, 2, 6, 3
    q, k, v, g, _ = _rand_case(rng, T, H, dk, dv)
    beta = np.zeros((T, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0)
    G = np.cumsum(g, axis=0)
    for h in range(H):
        St = np.exp(G[:, h])[:, :, None] * S0[0, h][None]
        np.testing.assert_allclose(out[:, h], np.einsum("tcj,tc->tj", St, q[:, h]), rtol=1e-12)
        np.testing.assert_allclose(fin[0, h], St[-1], rtol=1e-12)


def test_scalar_state_closed_form():
    """dk = dv = 1 with k = +-1: s_t = (1 - beta_t) alpha_t s_{t-1} + beta_t k_t v_t."""
    rng = np.random.default_rng(3)
    T = 20
    k = rng.choice([-1.0, 1.0], size=(T, 1, 1))
    q = rng.standard_normal((T, 1, 1))
    v = rng.standard_normal((T, 1, 1))
    g = -rng.uniform(0, 5, size=(T, 1, 1))
    beta = rng.uniform(0, 1, size=(T, 1))
    s0 = np.array([[[[0.7]]]])
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=s0)
    s = 0.7
    for t in range(T):
        s = (1 - beta[t, 0]) * math.exp(g[t, 0, 0]) * s + beta[t, 0] * k[t, 0, 0] * v[t, 0, 0]
        assert out[t, 0, 0] == pytest.approx(s * q[t, 0, 0], rel=1e-13, abs=1e-15)
    assert fin[0, 0, 0, 0] == pytest.approx(s, rel=1e-13)


def test_orthonormal_key_recall():
    """beta = 1, g = 0, S0 = 0: writing (k_j, v_j) for orthonormal k_j gives
    S^T k_j = v_j exactly; read back with q = k_j on tokens that write nothing."""
    rng = np.random.default_rng(4)
    dk, dv, m = 16, 7, 10
    Q, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Q[:, :m].T                      # m orthonormal keys
    vals = rng.standard_normal((m, dv))
    T = 2 * m
    k = np.zeros((T, 1, dk)); q = np.zeros((T, 1, dk)); v = np.zeros((T, 1, dv))
    beta = np.zeros((T, 1)); g = np.zeros((T, 1, dk))
    k[:m, 0] = keys; v[:m, 0] = vals; beta[:m, 0] = 1.0
    k[m:, 0] = keys; q[m:, 0] = keys                   # beta = 0: pure reads
    out, fin = oracle.prefill(q, k, v, g, beta)
    np.testing.assert_allclose(out[m:, 0], vals, atol=1e-12)
    np.testing.assert_allclose(fin[0, 0].T @ keys.T, vals.T, atol=1e-12)


def test_delta_rule_shrinks_the_error_on_the_written_key():
    """The erase-then-write update is the delta rule's error-correcting step:
    with S' = Diag(alpha_t) S_{t-1}, the prediction error on the written key
    after the update is (1 - beta_t |k_t|^2) times the error before it,
    S_t^T k_t - v_t = (1 - beta_t |k_t|^2) (S'^T k_t - v_t).  States before and
    after each token come from separate oracle runs over the two prefixes;
    keys are not normalised, so |k|^2 enters too."""
    rng = np.random.default_rng(41)
    T, dk, dv = 9, 6, 5
    q, k, v, g, beta = _rand_case(rng, T, 1, dk, dv, unit_k=False)
    S0 = rng.standard_normal((1, 1, dk, dv)) * 0.3
    prev = S0[0, 0]
    for t in range(T):
        _, fin = oracle.prefill(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1], beta[:t + 1],
                                init_state=S0)
        cur = fin[0, 0]
        decayed = np.exp(g[t, 0])[:, None] * prev
        kt, vt, bt = k[t, 0], v[t, 0], beta[t, 0]
        before = decayed.T @ kt - vt
        after = cur.T @ kt - vt
        np.testing.assert_allclose(after, (1.0 - bt * (kt @ kt)) * before, rtol=1e-10, atol=1e-12)
        prev = cur


@pytest.mark.parametrize("split", [1, 7, 16, 31])
def test_split_carry(split):
    """Running [0, T) equals [0, t) then [t, T) with the state carried over."""
    rng = np.random.default_rng(5 + split)
    T, H, dk, dv = 32, 2, 8, 6
    q, k, v, g, beta = _rand_case(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0)
    s = slice(0, split), slice(split, T)
    o1, f1 = oracle.prefill(*(x[s[0]] for x in (q, k, v, g, beta)), init_state=S0)
    o2, f2 = oracle.prefill(*(x[s[1]] for x in (q, k, v, g, beta)), init_state=f1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), out, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(f2, fin, rtol=1e-13, atol=1e-13)


def test_varlen_packing_restarts_state():
    """Packed sequences equal separate calls; each starts from its own state."""
    rng = np.random.default_rng(6)
    lens = [5, 0, 17, 1, 9]
    T, H, dk, dv = sum(lens), 2, 6, 5
    q, k, v, g, beta = _rand_case(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.cumsum([0] + lens)
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0, cu_seqlens=cu)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        o, f = oracle.prefill(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b],
                              init_state=S0[n:n + 1])
        np.testing.assert_allclose(out[a:b], o, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(fin[n], f[0], rtol=1e-14, atol=1e-14)
    assert np.array_equal(fin[1], S0[1])  # empty sequence: state passes through


def test_linear_in_values_and_initial_state():
    rng = np.random.default_rng(7)
    T, H, dk, dv = 15, 1, 5, 4
    q, k, v1, g, beta = _rand_case(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    s1, s2 = rng.standard_normal((2, 1, H, dk, dv))
    a, b = 0.37, -1.9
    o1, f1 = oracle.prefill(q, k, v1, g, beta, init_state=s1)
    o2, f2 = oracle.prefill(q, k, v2, g, beta, init_state=s2)
    o, f = oracle.prefill(q, k, a * v1 + b * v2, g, beta, init_state=a * s1 + b * s2)
    np.testing.assert_allclose(o, a * o1 + b * o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f, a * f1 + b * f2, rtol=1e-12, atol=1e-12)


def test_contraction_bound():
    """||k|| = 1, beta in [0,1], g <= 0: ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||."""
    rng = np.random.default_rng(8)
    T, dk, dv = 40, 8, 8
    q, k, v, g, beta = _rand_case(rng, T, 1, dk, dv, g_scale=0.05)
    S = rng.standard_normal((1, 1, dk, dv)) * 3
    for t in range(T):
        _, S_new = oracle.decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                 beta[t:t + 1], S)
        lhs = np.linalg.norm(S_new[0, 0], 2)
        rhs = np.linalg.norm(S[0, 0], 2) + beta[t, 0] * np.linalg.norm(v[t, 0])
        assert lhs <= rhs * (1 + 1e-12)
        S = S_new


def test_decode_chain_equals_prefill():
    rng = np.random.default_rng(9)
    T, N, H, dk, dv = 6, 3, 2, 5, 4
    q, k, v, g, beta = _rand_case(rng, T * N, H, dk, dv)
    S0 = rng.standard_normal((N, H, dk, dv))
    # sequence n owns tokens n*T .. n*T+T-1 in the packed prefill layout
    cu = np.arange(N + 1) * T
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0, cu_seqlens=cu)
    S = S0
    for t in range(T):
        idx = cu[:-1] + t
        o, S = oracle.decode(q[idx], k[idx], v[idx], g[idx], beta[idx], S)
        np.testing.assert_allclose(o, out[idx], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S, fin, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_chunk_form_matches_recurrence(chunk):
    """The chunkwise parallel form equals the token recurrence (ragged tails, varlen)."""
    rng = np.random.default_rng(10 + chunk)
    lens = [chunk * 2 + 5, 3, chunk]
    T, H, dk, dv = sum(lens), 2, 16, 12
    q, k, v, g, beta = _rand_case(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv)) * 0.1
    cu = np.cumsum([0] + lens)
    out, fin = oracle.prefill(q, k, v, g, beta, init_state=S0, cu_seqlens=cu)
    o2, f2 = oracle.chunk_form(q, k, v, g, beta, init_state=S0, cu_seqlens=cu, chunk=chunk)
    np.testing.assert_allclose(o2, out, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(f2, fin, rtol=1e-10, atol=1e-11)


def test_bf16_inputs_are_read_exactly():
    """bf16 inputs widen exactly: an fp32 call on the same rounded values agrees bit for bit."""
    w = inputs.WORKLOADS["prefill_T8192_H96_d128_bf16"]
    d = inputs.make_prefill(w, seed=0, heads=2, seq_len=40)
    o_b, f_b = oracle.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                              d["cu_seqlens"])
    o_f, f_f = oracle.prefill(*(d[n].float() for n in ("q", "k", "v", "g", "beta")),
                              d["init_state"], d["cu_seqlens"])
    assert np.array_equal(o_b, o_f) and np.array_equal(f_b, f_f)


def test_page_decay_bound_facts():
    """Facts the page prints about the lower-bounded decay, checked on generated inputs."""
    facts = json.load(open(os.path.join(GOLDEN, "decay_bound_facts.json")))
    g_min = facts["g_min"]
    assert round(math.exp(g_min), 4) == pytest.approx(facts["alpha_min_stated"], abs=5e-5)
    # e^80 fits the BF16 range (same exponent range as fp32)
    assert math.exp(facts["reciprocal_bound_exponent"]) < torch.finfo(torch.bfloat16).max
    for name in ("prefill_T8192_H96_d128_bf16", "prefill_T1M_H32_d128_bf16"):
        w = inputs.WORKLOADS[name]
        d = inputs.make_prefill(w, seed=0, heads=4, seq_len=4096)
        g = d["g"].double()
        assert float(g.min()) >= g_min and float(g.max()) <= 0.0
        tiles = g.reshape(-1, facts["tile_tokens"], 4, w.dk).sum(dim=1)
        assert float(tiles.min()) > facts["tile_log_decay_lower"]
    # the saturating workload really reaches the bound in bf16
    w = inputs.WORKLOADS["prefill_T1M_H32_d128_bf16"]
    d = inputs.make_prefill(w, seed=0, heads=2, seq_len=4096)
    assert float(d["g"].float().min()) == g_min


def test_generator_recipe_shapes_and_norms():
    w = inputs.WORKLOADS["varlen_32seq_H96_d128_bf16"]
    lens = inputs.seq_lengths(w, 0)
    assert len(lens) == 32 and min(lens) >= 512 and max(lens) <= 16384
    assert sum(lens) == 284_058                      # the recipe's seed-0 total
    assert list(inputs.seq_lengths(w, 0)) == list(lens)
    assert list(inputs.seq_lengths(w, 1)) != list(lens)
    d = inputs.make_prefill(w, seed=0, lengths=[70, 3], heads=3)
    assert d["q"].shape == (73, 3, 128) and d["beta"].shape == (73, 3)
    assert d["init_state"] is None
    nrm = d["k"].float().norm(dim=-1)
    assert float((nrm - 1).abs().max()) < 2e-2
    b = d["beta"].float()
    assert float(b.min()) > 0 and float(b.max()) < 1


def test_checkpoints_equal_prefix_final_states():
    """A checkpoint after j * interval tokens is the final state of the prefix
    [start, start + j * interval) of its sequence, with the same initial state."""
    rng = np.random.default_rng(20)
    lens, interval = [20, 7, 16, 0, 33], 8
    T, H, dk, dv = sum(lens), 2, 5, 4
    q, k, v, g, beta = _rand_case(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.cumsum([0] + lens)
    out, fin, ck = oracle.prefill(q, k, v, g, beta, init_state=S0, cu_seqlens=cu,
                                  ckpt_interval=interval)
    offs = oracle.checkpoint_offsets(cu, interval)
    assert list(np.diff(offs)) == [n // interval for n in lens]
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        for j in range(1, (b - a) // interval + 1):
            e = a + j * interval
            _, f = oracle.prefill(q[a:e], k[a:e], v[a:e], g[a:e], beta[a:e],
                                  init_state=S0[n:n + 1])
            np.testing.assert_array_equal(ck[offs[n] + j - 1], f[0])
    # outputs are unchanged by asking for checkpoints
    o2, f2 = oracle.prefill(q, k, v, g, beta, init_state=S0, cu_seqlens=cu)
    assert np.array_equal(o2, out) and np.array_equal(f2, fin)


# ---------------------------------------------------------------- output gate
# Head-wise RMSNorm then the full-rank gate, y = o / sqrt(mean(o^2) + eps) * w
# * sigmoid(z) (paper review, section "Kimi Delta Attention (KDA)", paragraph
# "Full-rank gate"; the formula is read from the prose, the page lost it).

def test_output_gate_hand_example():
    gold = json.load(open(os.path.join(GOLDEN, "output_gate_hand.json")))
    y = oracle.output_gate(np.array(gold["o"]), np.array(gold["z"]), np.array(gold["w"]),
                           gold["eps"])
    np.testing.assert_allclose(y, gold["y"], rtol=1e-14)
    # exact values 0.3 sqrt(2) and 1.2 sqrt(2)
    np.testing.assert_allclose(y, [0.3 * np.sqrt(2.0), 1.2 * np.sqrt(2.0)], rtol=1e-14)


def test_output_gate_constant_rows_and_symmetries():
    rng = np.random.default_rng(5)
    dv = 16
    a = rng.standard_normal((7, 1))
    o = np.repeat(a, dv, axis=1)                       # constant rows: rms = |a|
    z = rng.standard_normal((7, dv))
    w = rng.standard_normal(dv)
    y = oracle.output_gate(o, z, w, 0.0)
    np.testing.assert_allclose(y, np.sign(a) * w / (1.0 + np.exp(-z)), rtol=1e-13)
    o = rng.standard_normal((5, 3, dv))
    z = rng.standard_normal((5, 3, dv))
    y = oracle.output_gate(o, z, w, 0.0)
    np.testing.assert_allclose(oracle.output_gate(3.7 * o, z, w, 0.0), y, rtol=1e-13)
    np.testing.assert_allclose(oracle.output_gate(-o, z, w, 0.0), -y, rtol=1e-13)
    # w = 1 and a saturated gate: every row has unit mean square.
    y1 = oracle.output_gate(o, np.full_like(z, 60.0), np.ones(dv), 0.0)
    np.testing.assert_allclose(np.mean(y1 * y1, axis=-1), 1.0, rtol=1e-13)
    # eps far above the mean square: y -> o w sigmoid(z) / sqrt(eps).
    big = 1e12
    np.testing.assert_allclose(oracle.output_gate(o, z, w, big),
                               o * w / (1.0 + np.exp(-z)) / np.sqrt(big), rtol=1e-9)


# ---------------------------------------------------------------- KCP composition
# The paper review's infrastructure section: KDA context parallelism computes
# each segment's state transition locally and composes the segments
# associatively.  A segment maps its entry state to S_end = M S_0 + H with
# M = product of the per-token (I - beta k k^T) Diag(alpha) (dk x dk) and H the
# end state from S_0 = 0; M is the end state of the same tokens run from S_0 = I
# with v = 0.  Two segments compose as (M2, H2) o (M1, H1) = (M2 M1, M2 H1 + H2).

def _transition(x, cu):
    """(M [N, H, dk, dk], H [N, H, dk, dv]) of each sequence, from the oracle."""
    q, k, v, g, b = x
    N = len(cu) - 1
    Hh, dk = q.shape[1], q.shape[2]
    eye = np.broadcast_to(np.eye(dk), (N, Hh, dk, dk)).copy()
    _, M = oracle.prefill(q, k, torch.zeros(v.shape[0], Hh, dk, dtype=v.dtype), g, b, eye, cu)
    _, Hs = oracle.prefill(q, k, v, g, b, None, cu)
    return M, Hs


def test_kcp_transition_is_the_segment_map():
    # Slow decay (g in [-0.05, 0]) and weak erasure keep M of order one over
    # the 37 tokens, so a wrong M cannot hide below the tolerances (at the
    # generator's decay M shrinks below 1e-15).
    w = inputs.Workload("kcp", heads=2, dk=8, dv=8, dtype="f32", init_state=True)
    d = inputs.make_prefill(w, seed=41, device="cpu", lengths=[37])
    gen = torch.Generator().manual_seed(410)
    d["g"] = -0.05 * torch.rand(d["g"].shape, generator=gen, dtype=torch.float32)
    d["beta"] = 0.2 * d["beta"]          # weak erasure: the product of 37 steps stays O(1)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    M, Hs = _transition(x, d["cu_seqlens"])
    assert np.abs(M).max() > 0.3, "M must be of order one for this pin to mean anything"
    _, fin = oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
    s0 = d["init_state"].double().numpy()
    np.testing.assert_allclose(M @ s0 + Hs, fin, rtol=1e-12, atol=1e-12)
    # M is the product of the explicit per-token transition matrices.
    q, k, v, g, b = (t.double().numpy() for t in x)
    for h in range(2):
        P = np.eye(8)
        for t in range(37):
            A = (np.eye(8) - b[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(np.exp(g[t, h]))
            P = A @ P
        np.testing.assert_allclose(M[0, h], P, rtol=1e-12, atol=1e-13)


def test_kcp_composition_is_associative_and_matches_the_whole_sequence():
    w = inputs.Workload("kcp", heads=2, dk=8, dv=6, dtype="f32", init_state=True)
    T = 90
    d = inputs.make_prefill(w, seed=42, device="cpu", lengths=[T])
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    cuts = [0, 20, 51, 77, T]
    seg = torch.tensor(cuts, dtype=torch.int32)
    M, Hs = _transition(x, seg)                       # one transition per segment
    Mall, Hall = _transition(x, d["cu_seqlens"])      # the whole sequence at once

    def compose(a, b):                                # b after a
        return b[0] @ a[0], b[0] @ a[1] + b[1]

    parts = [(M[i], Hs[i]) for i in range(len(cuts) - 1)]
    left = parts[0]
    for p in parts[1:]:
        left = compose(left, p)                       # ((1 2) 3) 4
    right = parts[-1]
    for p in reversed(parts[:-1]):
        right = compose(p, right)                     # 1 (2 (3 4))
    for a, b_ in ((left, right), (left, (Mall[0], Hall[0]))):
        np.testing.assert_allclose(a[0], b_[0], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(a[1], b_[1], rtol=1e-11, atol=1e-12)
    # Segment entry states from the composed prefixes reproduce the outputs of
    # the whole sequence when each segment is run from its own entry state.
    s = d["init_state"].double().numpy()[0]
    starts = []
    for Mi, Hi in parts:
        starts.append(s)
        s = Mi @ s + Hi
    out_seg, fin_seg = oracle.prefill(*x, np.stack(starts), seg)
    out, fin = oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
    np.testing.assert_allclose(out_seg, out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fin_seg[-1], fin[0], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- prologue
# ShortConv (4 causal depthwise taps, tap 3 on the current token) -> Swish ->
# L2 norm for q and k; g = -5 sigmoid(exp(A_h) z) (paper review, section
# "Kimi Delta Attention (KDA)"; the formulas are read from the prose).

def test_prologue_hand_example():
    gold = json.load(open(os.path.join(GOLDEN, "prologue_hand.json")))
    x = np.array(gold["q_pre"])
    w = np.array(gold["conv"])
    q, k, g = oracle.prologue(x, x, np.array(gold["z"]), w, w, np.array(gold["a_log"]),
                              None, eps=0.0)
    np.testing.assert_allclose(q, gold["q"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(k, q, rtol=0, atol=0)
    np.testing.assert_allclose(g, gold["g"], rtol=1e-14)


def test_prologue_kernels_shifts_norms_and_decay():
    rng = np.random.default_rng(61)
    T, H, dk = 23, 2, 8
    x = rng.standard_normal((T, H, dk))
    z = rng.standard_normal((T, H, dk))
    cu = np.array([0, 9, 9, 23])
    imp = np.zeros((H, dk, 4))
    imp[:, :, 3] = 1.0                         # the current token only
    q, _, _ = oracle.prologue(x, x, z, imp, imp, np.zeros(H), cu, eps=0.0)
    sw = x / (1.0 + np.exp(-x))
    np.testing.assert_allclose(q, sw / np.linalg.norm(sw, axis=-1, keepdims=True), rtol=1e-13)
    shift = np.zeros((H, dk, 4))
    shift[:, :, 2] = 1.0                       # the previous token only
    q, _, _ = oracle.prologue(x, x, z, shift, shift, np.zeros(H), cu, eps=1e-6)
    for t0 in (0, 9):                          # nothing before a sequence start
        assert np.all(q[t0] == 0.0)
    swp = np.roll(sw, 1, axis=0)
    for t in list(range(1, 9)) + list(range(10, 23)):
        np.testing.assert_allclose(q[t], swp[t] / np.sqrt(np.sum(swp[t] ** 2, -1, keepdims=True)
                                                           + 1e-6), rtol=1e-13)
    w = rng.standard_normal((H, dk, 4))
    a = rng.standard_normal(H)
    q, k, g = oracle.prologue(x, x, z, w, w, a, cu, eps=0.0)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_array_equal(k, q)               # same input, same kernel, same branch
    assert np.all(g < 0) and np.all(g > -5)
    _, _, g0 = oracle.prologue(x, x, np.exp(a)[None, :, None] * z, w, w, np.zeros(H), cu)
    np.testing.assert_allclose(g, g0, rtol=1e-14)
    _, _, gz = oracle.prologue(x, x, np.zeros_like(z), w, w, a, cu)
    np.testing.assert_allclose(gz, -2.5, rtol=1e-15)
    # Packing is separate calls: no tap reaches across a sequence boundary.
    qa, _, _ = oracle.prologue(x[:9], x[:9], z[:9], w, w, a, None)
    qb, _, _ = oracle.prologue(x[9:], x[9:], z[9:], w, w, a, None)
    q, _, _ = oracle.prologue(x, x, z, w, w, a, cu)
    np.testing.assert_allclose(q, np.concatenate([qa, qb]), rtol=1e-14)
