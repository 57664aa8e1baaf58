"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching the device."""

import ctypes
import os
import re

import pytest
import torch

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def L():
    path = __graft_entry__._build_module().build()
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.kda_chunk_fwd_workspace_size.argtypes = [i64, i32, i32, i32]
    lib.kda_chunk_fwd_workspace_size.restype = sz
    lib.kda_chunk_fwd_ex.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32,
                                     vp, vp, vp, sz, vp, ctypes.c_uint]
    lib.kda_chunk_fwd.argtypes = lib.kda_chunk_fwd_ex.argtypes[:-1]
    lib.kda_chunk_fwd_gated.argtypes = [vp, vp, vp, i32, vp, vp, ctypes.c_float, vp, vp, vp, i32,
                                        i32, i64, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.kda_gate.argtypes = [vp, i32, vp, ctypes.c_float, vp, i64, i32, i32, vp, vp, i32, vp]
    lib.kda_recurrent_step.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.kda_last_error_string.restype = ctypes.c_char_p
    lib.kda_version.restype = ctypes.c_char_p
    return lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("kda_gate", "kda_chunk_fwd", "kda_recurrent_step"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in kda.h but not exported"


def test_version(L):
    assert re.match(rb"^\d+\.\d+\.\d+$", L.kda_version())


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case below fails on the host


def _chunk(L, dtype=1, dk=128, dv=128, H=2, B=1, T=64, ws=FAKE, ws_bytes=1 << 40, q=FAKE,
           cu=None, n_seqs=0, flags=0):
    return L.kda_chunk_fwd_ex(q, FAKE, FAKE, dtype, FAKE, FAKE, None, cu, n_seqs, B, T, H, dk, dv,
                              FAKE, FAKE, ws, ws_bytes, None, flags)


def test_chunk_rejects_bad_arguments(L):
    assert _chunk(L, dk=64) == 2
    assert _chunk(L, dv=256) == 2
    assert _chunk(L, H=0) == 2
    assert _chunk(L, dtype=7) == 3
    assert _chunk(L, q=FAKE + 8) == 4
    assert _chunk(L, ws=FAKE + 16) == 4
    assert _chunk(L, ws_bytes=16) == 5
    assert _chunk(L, flags=64) == 1  # an unknown flag bit
    assert _chunk(L, B=2, cu=FAKE, n_seqs=2) == 1  # B must be 1 with cu_seqlens
    assert _chunk(L, cu=FAKE, n_seqs=0) == 1
    assert _chunk(L, q=None) == 1
    assert b"workspace" in L.kda_last_error_string() or L.kda_last_error_string()


def _gated(L, dtype=1, g_min=-5.0, z=FAKE, A=FAKE, dk=128, ws_bytes=1 << 40):
    return L.kda_chunk_fwd_gated(FAKE, FAKE, FAKE, dtype, z, A, g_min, FAKE, None, None, 0, 1, 64,
                                 2, dk, 128, FAKE, FAKE, FAKE, ws_bytes, None)


def test_chunk_gated_rejects_bad_arguments(L):
    assert _gated(L, dtype=0) == 3       # fp32: call kda_gate, then kda_chunk_fwd
    assert _gated(L, g_min=-6.0) == 1    # below the tile range bound
    assert _gated(L, g_min=0.0) == 1
    assert _gated(L, z=None) == 1
    assert _gated(L, A=None) == 1
    assert _gated(L, z=FAKE + 8) == 4
    assert _gated(L, dk=64) == 2
    assert _gated(L, ws_bytes=16) == 5
    assert b"kda_chunk_fwd_gated" in L.kda_last_error_string()


def _ckpt(L, dtype=1, ckpt=FAKE, every=512, cap=4, flags=0):
    vp, i32, i64, sz, u32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                             ctypes.c_uint)
    L.kda_chunk_fwd_checkpointed.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i64, i32,
                                             i32, i32, vp, vp, vp, i32, i64, vp, sz, vp, u32]
    return L.kda_chunk_fwd_checkpointed(FAKE, FAKE, FAKE, dtype, FAKE, FAKE, None, None, 0, 1, 64,
                                        2, 128, 128, FAKE, FAKE, ckpt, every, cap, FAKE, 1 << 40,
                                        None, flags)


def test_chunk_checkpointed_rejects_bad_arguments(L):
    assert _ckpt(L, dtype=0) == 3        # checkpoints come from the tensor-core chain only
    assert _ckpt(L, flags=1) == 3        # fp32-core evaluation requested
    assert _ckpt(L, every=100) == 1      # not a multiple of the 64-token chunk
    assert _ckpt(L, every=0) == 1
    assert _ckpt(L, cap=-1) == 1
    assert _ckpt(L, ckpt=None) == 1      # no buffer for a positive capacity
    assert _ckpt(L, ckpt=FAKE + 16) == 4  # 32-byte stores
    assert _ckpt(L, flags=64) == 1       # unknown flag bit
    assert b"kda_chunk_fwd_checkpointed" in L.kda_last_error_string()


def _fused(L, dtype=1, g=None, z=0x10000, g_min=-5.0, qk=-1.0, gate=None, w=None, eps=1e-6,
           flags=0):
    vp, i32, i64, f32, sz, u32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                  ctypes.c_size_t, ctypes.c_uint)
    L.kda_chunk_fwd_fused.argtypes = [vp, vp, vp, i32, vp, vp, vp, f32, vp, vp, vp, i32, i32, i64,
                                      i32, i32, i32, f32, vp, vp, f32, vp, vp, vp, sz, vp, u32]
    return L.kda_chunk_fwd_fused(FAKE, FAKE, FAKE, dtype, g, z, FAKE, g_min, FAKE, None, None, 0,
                                 1, 64, 2, 128, 128, qk, gate, w, eps, FAKE, FAKE, FAKE, 1 << 40,
                                 None, flags)


def test_chunk_fused_rejects_bad_arguments(L):
    assert _fused(L, dtype=0) == 3                 # tensor-core (bf16) path only
    assert _fused(L, flags=1) == 3
    assert _fused(L, g=FAKE) == 1                  # both g and z
    assert _fused(L, z=None) == 1                  # neither
    assert _fused(L, g_min=-6.0) == 1
    assert _fused(L, qk=float("inf")) == 1
    assert _fused(L, gate=FAKE, eps=-1.0) == 1
    assert _fused(L, gate=FAKE, eps=float("nan")) == 1
    assert _fused(L, w=FAKE) == 1                  # a weight without the gate
    assert _fused(L, gate=FAKE + 8) == 4
    assert _fused(L, flags=4) == 3                 # the unbounded-gate mode is not fused
    assert _fused(L, flags=8) == 1                 # scalar gates with z
    assert _fused(L, flags=64) == 1                # an unknown flag bit
    assert b"kda_chunk_fwd_fused" in L.kda_last_error_string()


def test_output_gate_rejects_bad_arguments(L):
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    L.kda_output_gate.argtypes = [vp, i32, vp, vp, f32, vp, i64, i32, i32, vp]
    og = lambda dtype=1, o=FAKE, x=FAKE, w=None, eps=1e-6, y=FAKE, n=10, H=2, dv=128: \
        L.kda_output_gate(o, dtype, x, w, eps, y, n, H, dv, None)
    assert og(dtype=5) == 3
    assert og(dv=64) == 2
    assert og(H=0) == 2
    assert og(eps=-1.0) == 1
    assert og(eps=float("inf")) == 1
    assert og(n=-1) == 1
    assert og(x=None) == 1
    assert og(y=FAKE + 2) == 4
    assert og(w=FAKE + 4) == 4
    assert og(n=0) == 0                          # nothing to do, no device needed
    assert b"kda_output_gate" in L.kda_last_error_string()


def test_workspace_size(L):
    L.kda_chunk_fwd_workspace_size_ex.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_uint]
    L.kda_chunk_fwd_workspace_size_ex.restype = ctypes.c_size_t
    # chain segments add state scratch; sequential and fp32-core evaluation do not
    seg = L.kda_chunk_fwd_workspace_size_ex(16384, 1, 2, 1, 16 << 16)
    seq = L.kda_chunk_fwd_workspace_size_ex(16384, 1, 2, 1, 2)
    assert seg > seq > 0
    assert L.kda_chunk_fwd_workspace_size_ex(8192, 1, 96, 1, 0) == L.kda_chunk_fwd_workspace_size(8192, 1, 96, 1)
    a = L.kda_chunk_fwd_workspace_size(8192, 1, 96, 1)
    b = L.kda_chunk_fwd_workspace_size(8192, 1, 96, 0)
    assert a > 0 and b > 0
    assert L.kda_chunk_fwd_workspace_size(-1, 1, 96, 1) == 0
    assert L.kda_chunk_fwd_workspace_size(10, 0, 96, 1) == 0
    assert L.kda_chunk_fwd_workspace_size(10, 1, 96, 5) == 0
    # scalar gates: read as they are on the tensor-core path, spread over the
    # channels in the workspace on the fp32-core paths
    assert L.kda_chunk_fwd_workspace_size_ex(8192, 1, 96, 1, 8) == a
    spread = 8192 * 96 * 128 * 4
    assert L.kda_chunk_fwd_workspace_size_ex(8192, 1, 96, 0, 8) >= b + spread
    assert L.kda_chunk_fwd_workspace_size_ex(8192, 1, 96, 1, 9) >= \
        L.kda_chunk_fwd_workspace_size_ex(8192, 1, 96, 1, 1) + spread
    # grows with tokens and heads
    assert L.kda_chunk_fwd_workspace_size(16384, 1, 96, 1) > a
    assert L.kda_chunk_fwd_workspace_size(8192, 1, 97, 1) > a


def test_segment_choice_for_long_sequences(L):
    """The automatic chain segmentation of one 2^20-token sequence with 16 heads uses
    10 segments of 1,639 chunks (the wave cost model: 16 x 18 CTAs, then 16 x 9, on
    148-152 SMs), visible through the workspace the choice needs."""
    L.kda_chunk_fwd_workspace_size_ex.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_uint]
    L.kda_chunk_fwd_workspace_size_ex.restype = ctypes.c_size_t
    f = L.kda_chunk_fwd_workspace_size_ex
    auto = f(1 << 20, 1, 16, 1, 0)
    assert auto == f(1 << 20, 1, 16, 1, 1639 << 16)
    assert auto != f(1 << 20, 1, 16, 1, 1821 << 16)       # the former 9-segment choice
    assert f(1 << 20, 1, 16, 1, 2) < auto                  # sequential: no segment state
    # enough chains to fill the GPU: no segments
    assert f(8192, 1, 96, 1, 0) == f(8192, 1, 96, 1, 2)


def test_gate_rejects_bad_arguments(L):
    assert L.kda_gate(FAKE, 0, FAKE, -5.0, FAKE, 10, 2, 64, None, None, 1, None) == 2
    assert L.kda_gate(FAKE, 3, FAKE, -5.0, FAKE, 10, 2, 128, None, None, 1, None) == 3
    assert L.kda_gate(FAKE, 0, FAKE, 1.0, FAKE, 10, 2, 128, None, None, 1, None) == 1
    assert L.kda_gate(FAKE + 4, 0, FAKE, -5.0, FAKE, 10, 2, 128, None, None, 1, None) == 4
    assert L.kda_gate(None, 0, FAKE, -5.0, FAKE, 10, 2, 128, None, None, 1, None) == 1
    assert L.kda_gate(FAKE, 0, FAKE, -5.0, FAKE, 0, 2, 128, None, None, 1, None) == 0  # no-op


def test_recurrent_multi_step_rejects_bad_arguments(L):
    L.kda_recurrent_multi_step.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] + \
        [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    args = [FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, None, 4, 8, 2, 128, 128, None]
    bad = list(args); bad[10] = 17           # T above the supported 16
    assert L.kda_recurrent_multi_step(*bad) == 2
    bad = list(args); bad[10] = 0
    assert L.kda_recurrent_multi_step(*bad) == 2
    bad = list(args); bad[12] = 64
    assert L.kda_recurrent_multi_step(*bad) == 2
    bad = list(args); bad[3] = 5
    assert L.kda_recurrent_multi_step(*bad) == 3
    bad = list(args); bad[6] = FAKE + 4
    assert L.kda_recurrent_multi_step(*bad) == 4
    bad = list(args); bad[0] = None
    assert L.kda_recurrent_multi_step(*bad) == 1
    bad = list(args); bad[9] = 0
    assert L.kda_recurrent_multi_step(*bad) == 0   # N = 0 is a no-op


def test_recurrent_step_rejects_bad_arguments(L):
    args = [FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 128, None]
    bad = list(args); bad[10] = 64
    assert L.kda_recurrent_step(*bad) == 2
    bad = list(args); bad[3] = 9
    assert L.kda_recurrent_step(*bad) == 3
    bad = list(args); bad[6] = FAKE + 4
    assert L.kda_recurrent_step(*bad) == 4
    bad = list(args); bad[0] = None
    assert L.kda_recurrent_step(*bad) == 1
    bad = list(args); bad[8] = 0
    assert L.kda_recurrent_step(*bad) == 0  # N = 0 is a no-op


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_fails_cleanly(L):
    st = _chunk(L)
    assert st in (6, 8), st


def test_python_binding_imports_and_refuses_cpu_tensors():
    import chunked_gated_delta_fwd_gb300 as kda

    z = torch.zeros(4, 2, 128)
    with pytest.raises(ValueError):
        kda.gate(z, torch.zeros(2))


def test_wait_selftest_rejects_bad_limits_on_the_host(L):
    """The bounded-wait self-test checks its limit before touching the device."""
    f = L.kda_selftest_wait_timeout
    f.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_int), ctypes.c_void_p]
    f.restype = ctypes.c_int
    n = ctypes.c_int(-1)
    assert f(0, ctypes.byref(n), None) == 1
    assert f(2_000_000, ctypes.byref(n), None) == 1
    assert f(1000, None, None) == 1
    assert n.value == -1
