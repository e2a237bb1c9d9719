"""The C ABI loads on a machine without a GPU, exports what include/kda.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import hybrid_linear_attention_02_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return kda.load()


def test_every_declared_symbol_is_exported(lib):
    syms = _declared_symbols()
    assert {"kda_chunk_fwd", "kda_decode_step", "kda_chunk_fwd_workspace_size",
            "kda_status_string", "kda_version"} <= syms
    for s in sorted(syms):
        assert hasattr(lib, s), f"{s} declared in include/ but not exported"


def test_wait_timeout_self_test_rejects_bad_arguments(lib):
    # (no launch happens: the arguments are refused on the host)
    assert lib.kda_debug_wait_timeout(None, 1000, None) == -1
    assert lib.kda_debug_wait_timeout(ctypes.c_void_p(16), 0, None) == -1


def test_withhold_self_test_rejects_bad_arguments(lib):
    d = _dims(n=1, t=128)
    call = lambda which, st: lib.kda_debug_chunk_fwd_withhold(
        which, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, ctypes.byref(d), None, 0, st, None)
    assert call(0, FAKE) == -1 and call(4, FAKE) == -1     # unknown form
    assert call(1, None) == -1                              # dev_status required
    assert call(1, FAKE) == -6                              # the split form needs a workspace
    dd = _dims(n=1, t=128, dtype=0)                         # fp32: no tensor-core kernel
    assert lib.kda_debug_chunk_fwd_withhold(3, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                                            ctypes.byref(dd), None, 0, FAKE, None) == -2


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.kda_status_string(code)
    assert b"[-5, 0]" in lib.kda_status_string(-8)      # KDA_ERR_RANGE
    assert lib.kda_status_string(12345) == b"unknown status"
    assert lib.kda_version() >= 10000


def test_range_check_host_validation(lib):
    """kda_check_inputs refuses bad arguments on the host (no launch); the
    default build does not run it inside the prefill and decode calls."""
    d = _dims(n=1, t=64)
    assert lib.kda_check_inputs(FAKE, FAKE, ctypes.byref(d), None, None) == -1   # no status
    assert lib.kda_check_inputs(None, FAKE, ctypes.byref(d), FAKE, None) == -1   # no g
    assert lib.kda_check_inputs(MISALIGNED, FAKE, ctypes.byref(d), FAKE, None) == -5
    assert lib.kda_check_inputs(FAKE, FAKE, ctypes.byref(_dims(dk=96)), FAKE, None) == -2
    assert lib.kda_check_inputs(FAKE, FAKE, ctypes.byref(_dims(n=0, t=0)), FAKE, None) == 0
    assert lib.kda_debug_bounds_build() == 0


def test_noalloc_validates_like_kda_chunk_fwd(lib):
    """Both prefill entry points share their argument checks: the same status
    for the same arguments (only the scratch limit is the no-alloc call's)."""
    vp = ctypes.c_void_p
    fn = lib.kda_chunk_fwd_noalloc
    fn.argtypes = [vp] * 9 + [ctypes.c_int, ctypes.POINTER(kda._Dims), vp, vp]
    fn.restype = ctypes.c_int
    cases = [
        (_dims(n=0, t=0), FAKE, MISALIGNED, 64),   # empty call, misaligned state: fine
        (_dims(), FAKE, MISALIGNED, 64),           # misaligned state
        (_dims(), MISALIGNED, None, 64),           # misaligned input
        (_dims(), FAKE, None, 48),                 # unsupported chunk
        (_dims(n=3, t=64), FAKE, None, 64),        # not divisible
        (_dims(dk=96), FAKE, None, 64),
    ]
    for d, q, s0, chunk in cases:
        a = lib.kda_chunk_fwd(q, FAKE, FAKE, FAKE, FAKE, s0, None, FAKE, None, chunk,
                              ctypes.byref(d), None, 0, None, None)
        b = fn(q, FAKE, FAKE, FAKE, FAKE, s0, None, FAKE, None, chunk, ctypes.byref(d), None,
               None)
        assert a == b, (d.n_seqs, d.total_tokens, chunk, a, b)


def _dims(n=1, t=64, h=2, dk=128, dv=128, dtype=1):
    return kda._Dims(n, t, h, dk, dv, dtype)


FAKE = ctypes.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced
MISALIGNED = ctypes.c_void_p((1 << 20) + 8)


def _prefill(lib, d, chunk=64, q=FAKE, cu=None, ws=None, ws_bytes=0):
    return lib.kda_chunk_fwd(q, FAKE, FAKE, FAKE, FAKE, None, cu, FAKE, None, chunk,
                             ctypes.byref(d), ws, ws_bytes, None, None)


def test_host_validation_prefill(lib):
    assert _prefill(lib, _dims(), chunk=48) == -2          # unsupported chunk
    assert _prefill(lib, _dims(dk=96)) == -2               # unsupported head dim
    assert _prefill(lib, _dims(dtype=7)) == -2             # unknown dtype
    assert _prefill(lib, _dims(t=-1)) == -1                # negative size
    assert _prefill(lib, _dims(), q=None) == -1            # null input
    assert _prefill(lib, _dims(), q=MISALIGNED) == -5      # misaligned input
    assert _prefill(lib, _dims(n=3, t=64)) == -1           # 64 tokens not divisible by 3
    assert _prefill(lib, _dims(n=3, t=63), cu=FAKE) == -6  # varlen needs workspace
    assert lib.kda_chunk_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None, 64, None,
                             None, 0, None, None) == -1    # null dims
    # nothing to do: no tokens, no sequences
    assert _prefill(lib, _dims(n=0, t=0)) == 0


def test_host_validation_checkpoints(lib):
    d = _dims(n=1, t=128)

    def call(ck=FAKE, offs=FAKE, interval=64):
        return lib.kda_chunk_fwd_checkpoints(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                             64, ctypes.byref(d), None, 0, None, None, ck, offs,
                                             interval)

    assert call(ck=None) == -1              # checkpoint buffer is required
    assert call(offs=None) == -1            # so are the offsets
    assert call(interval=0) == -1           # interval must be positive
    assert call(interval=-64) == -1
    assert call(interval=100) == -2         # and a multiple of 64
    assert call(ck=MISALIGNED) == -5


def test_host_validation_gated(lib):
    d = _dims(n=1, t=64)

    def call(gate=FAKE, w=FAKE, eps=1e-6):
        return lib.kda_chunk_fwd_gated(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, gate, w,
                                       ctypes.c_float(eps), FAKE, None, 64, ctypes.byref(d),
                                       None, 0, None, None)

    assert call(gate=None) == -1
    assert call(w=None) == -1
    assert call(eps=-1.0) == -1
    assert call(eps=float("nan")) == -1
    assert call(gate=MISALIGNED) == -5
    dd = _dims(n=4, t=4)
    assert lib.kda_decode_step_gated(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, MISALIGNED,
                                     ctypes.c_float(1e-6), FAKE, FAKE, ctypes.byref(dd), None,
                                     None) == -5


def test_host_validation_decode(lib):
    d = _dims(n=4, t=5)
    assert lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(d),
                               None, None) == -1           # total_tokens != n_seqs
    d = _dims(n=4, t=4)
    assert lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, ctypes.byref(d),
                               None, None) == -1           # null state
    assert lib.kda_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, MISALIGNED, FAKE,
                               ctypes.byref(d), None, None) == -5


REC = 66048          # one chunk record of the split tensor-core path


def test_workspace_size(lib):
    size = lambda d, c=64: lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), c)
    algo = lambda d, c=64: lib.kda_chunk_fwd_algorithm(ctypes.byref(d), c)
    # CUDA-core path (fp32): only the longest-first order of packed sequences.
    assert algo(_dims(n=1, dtype=0)) == 0 and size(_dims(n=1, dtype=0)) == 0
    ws = size(_dims(n=32, t=1000, dtype=0))
    assert ws >= 32 * 4 and ws % 256 == 0
    # bf16, d = 128, few pairs: split path, carried states + a record per chunk.
    d = _dims(n=1, t=8192, h=96)
    assert algo(d) == 2
    assert size(d) == 96 * 128 * 128 * 4 + 96 * (8192 // 64 + 1) * REC
    # Long inputs: the record buffer is capped (2 GiB for pairs that run
    # overlapped windows), the rest runs in windows.
    d = _dims(n=1, t=1 << 20, h=32)
    assert size(d) == 32 * 128 * 128 * 4 + ((2 << 30) // REC) * REC
    # Many pairs from few sequences: still split; all 408,000 records (26.9 GB)
    # fit under the 32 GiB cap, so the call runs in one window.
    d = _dims(n=32, t=270000, h=96)
    assert algo(d) == 2
    assert size(d) == 256 + 32 * 96 * 128 * 128 * 4 + 96 * (270000 // 64 + 32) * REC
    # Many pairs from many sequences: one fused kernel per pair, order array only.
    d = _dims(n=64, t=270000, h=96)
    assert algo(d) == 1 and size(d) == 256
    # bf16 chunk 16 or 32 is served by the tensor-core kernels' 64-token
    # chunks (no silent fall back to the CUDA-core path).
    for c in (16, 32):
        assert algo(_dims(n=1, t=8192, h=96), c) == 2
        assert size(_dims(n=1, t=8192, h=96), c) == size(_dims(n=1, t=8192, h=96), 64)
        assert algo(_dims(n=64, t=270000, h=96), c) == 1
    assert algo(_dims(n=1, t=8192, h=96, dtype=0), 32) == 0   # fp32: the recurrence
    assert size(_dims(dk=7)) == 0


def test_dispatch_boundaries(lib, monkeypatch):
    """The split form serves up to 304 sequence-head pairs, or any pair count
    from at most 32 sequences, and never more than 1024 sequences; its record
    buffer is capped at 2 GiB up to 76 pairs (overlapped windows) and at
    32 GiB above."""
    monkeypatch.delenv("KDA_CHUNK_PATH", raising=False)
    algo = lambda d: lib.kda_chunk_fwd_algorithm(ctypes.byref(d), 64)
    size = lambda d: lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), 64)
    assert algo(_dims(n=38, t=38 * 512, h=8)) == 2      # 304 pairs
    assert algo(_dims(n=39, t=39 * 512, h=8)) == 1      # 312 pairs, 39 sequences
    assert algo(_dims(n=32, t=32 * 512, h=64)) == 2     # 2048 pairs, 32 sequences
    assert algo(_dims(n=33, t=33 * 512, h=64)) == 1     # 33 sequences
    assert algo(_dims(n=1024, t=1024 * 64, h=1)) == 1   # more than 304 pairs
    assert algo(_dims(n=1025, t=1025 * 64, h=1)) == 1   # over the sequence cap
    order = lambda n: (n * 4 + 255) // 256 * 256
    states = lambda n, h: n * h * 128 * 128 * 4
    cap = lambda gib: ((gib << 30) // REC) * REC
    t = 1 << 20
    assert size(_dims(n=1, t=t, h=76)) == states(1, 76) + cap(2)
    assert size(_dims(n=1, t=t, h=77)) == states(1, 77) + cap(32)
    assert size(_dims(n=2, t=t, h=38)) == order(2) + states(2, 38) + cap(2)


def test_launch_count_host_cases(lib):
    """Kernels per kda_chunk_fwd call where no device query is needed: the
    fused and token-recurrence paths launch one kernel, plus the length-order
    kernel with cu_seqlens and more than one sequence."""
    lc = lambda d, ws=0, varlen=0, c=64: lib.kda_chunk_fwd_launch_count(ctypes.byref(d), c, ws,
                                                                        varlen)
    fused = _dims(n=64, t=64 * 8192, h=96)                 # 6,144 pairs of 64 sequences
    assert lib.kda_chunk_fwd_algorithm(ctypes.byref(fused), 64) == 1
    assert lc(fused, ws=1 << 20) == 1 and lc(fused, ws=1 << 20, varlen=1) == 2
    assert lc(fused, ws=0, varlen=1) == -6                 # KDA_ERR_WORKSPACE, as the call
    # Split by default, but a workspace below one record per pair: fused.
    assert lc(_dims(n=1, t=8192, h=96), ws=1024) == 1
    assert lc(_dims(n=1, t=256, h=1, dk=64, dv=64, dtype=0)) == 1   # token recurrence
    assert lc(_dims(n=0, t=0, h=96)) == 0
    assert lc(fused, c=48) == -2                           # KDA_ERR_UNSUPPORTED


def test_path_override(lib, monkeypatch):
    d = _dims(n=1, t=8192, h=96)
    monkeypatch.setenv("KDA_CHUNK_PATH", "fused")
    assert lib.kda_chunk_fwd_algorithm(ctypes.byref(d), 64) == 1
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), 64) == 0
    monkeypatch.setenv("KDA_CHUNK_PATH", "split")
    d = _dims(n=64, t=270000, h=96)
    assert lib.kda_chunk_fwd_algorithm(ctypes.byref(d), 64) == 2


def test_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 2, 128)
    with pytest.raises(ValueError):
        kda.chunk_fwd(x, x, x, x, torch.zeros(4, 2))
