"""kda_chunk_fwd_noalloc: the prefill for callers that may not allocate.

Some callers run the prefill where they are not allowed to allocate device
memory (an engine that reserved all of it at start-up, a plugin host without an
allocator, a latency-critical loop).  For them the library keeps a fixed scratch
array in device memory and kda_chunk_fwd_noalloc takes only inputs and outputs.
These tests call it through the C ABI twice in a row, on different inputs, and
check each result against kda_chunk_fwd with a caller workspace, within the
tolerances of the other parity tests.  The file is named to be collected last.
"""

import ctypes

import pytest
import torch

import workloads
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import chunked_gated_delta_fwd_gb300 as m

    fn = m.lib.kda_chunk_fwd_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32, vp, vp, vp]
    fn.restype = ctypes.c_int
    m.lib.kda_chunk_fwd_noalloc_capacity.restype = ctypes.c_size_t
    return m


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _inputs(lens, H, dtype, seed):
    w = workloads.custom(lens, H=H, dtype=dtype, seed=seed, h0_std=0.3)
    inp = workloads.make_inputs(w, "cuda")
    g = workloads.uniform_decay((w.n_tokens, H, 128), "cuda", seed=seed + 1)
    return inp, g, w


def _noalloc(kda, inp, g, w, batched=False):
    """One call through the C ABI: packed with cu_seqlens, or (batched) as B equal
    sequences of T tokens without cu_seqlens."""
    o = torch.empty_like(inp["v"])
    hT = torch.empty(w.n_seqs, w.H, 128, 128, dtype=torch.float32, device="cuda")
    code = kda.BF16 if inp["q"].dtype == torch.bfloat16 else kda.F32
    if batched:
        B, T, cu, n = w.n_seqs, w.seq_lens[0], None, 0
    else:
        B, T, cu, n = 1, w.n_tokens, inp["cu_seqlens"], w.n_seqs
    st = kda.lib.kda_chunk_fwd_noalloc(
        _p(inp["q"]), _p(inp["k"]), _p(inp["v"]), code, _p(g), _p(inp["beta"]), _p(inp["h0"]),
        _p(cu), n, B, T, w.H, 128, 128, _p(o), _p(hT),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, kda.lib.kda_last_error_string()
    return o, hT


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_entry_point_twice(kda, dtype):
    cases = [([300, 0, 129, 64], 4, 71), ([1, 200, 65], 3, 72)]
    for lens, H, seed in cases:  # two calls in a row, different inputs
        inp, g, w = _inputs(lens, H, dtype, seed)
        o, hT = _noalloc(kda, inp, g, w)
        o_ref, h_ref = kda.chunk_fwd(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
        torch.cuda.synchronize()
        assert_close(o, o_ref, dtype, f"o, lens={lens}")
        assert_close(hT, h_ref, dtype, f"hT, lens={lens}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_fixed_batch_without_cu_seqlens(kda, dtype):
    """B = 2 sequences of 150 tokens, no cu_seqlens (the plan derives the offsets),
    two calls in a row against kda_chunk_fwd with a caller workspace."""
    B, T, H = 2, 150, 3
    for seed in (81, 82):
        inp, g, w = _inputs([T] * B, H, dtype, seed)
        o, hT = _noalloc(kda, inp, g, w, batched=True)
        shp = lambda t: t.view(B, T, *t.shape[1:])
        o_ref, h_ref = kda.chunk_fwd(shp(inp["q"]), shp(inp["k"]), shp(inp["v"]), shp(g),
                                     shp(inp["beta"]), inp["h0"], None)
        torch.cuda.synchronize()
        assert_close(o, o_ref.view_as(o), dtype, f"o batched, seed={seed}")
        assert_close(hT, h_ref, dtype, f"hT batched, seed={seed}")


def test_noalloc_reports_malformed_calls_before_the_capacity(kda):
    """A call that is both too large for the scratch array and malformed (dk = 64)
    gets the error of its malformed argument, not the capacity error."""
    H, NT = 96, 2048
    inp, g, w = _inputs([NT], H, torch.bfloat16, 74)
    o = torch.empty_like(inp["v"])
    st = kda.lib.kda_chunk_fwd_noalloc(
        _p(inp["q"]), _p(inp["k"]), _p(inp["v"]), kda.BF16, _p(g), _p(inp["beta"]), None,
        _p(inp["cu_seqlens"]), 1, 1, NT, H, 64, 128, _p(o), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 2, kda.lib.kda_last_error_string()  # KDA_ERR_UNSUPPORTED_SHAPE


def test_noalloc_rejects_problems_larger_than_its_scratch(kda):
    cap = kda.lib.kda_chunk_fwd_noalloc_capacity()
    H, NT = 96, 2048
    need = kda.chunk_fwd_workspace_size(NT, 1, H, torch.bfloat16)
    assert need > cap
    inp, g, w = _inputs([NT], H, torch.bfloat16, 73)
    o = torch.empty_like(inp["v"])
    st = kda.lib.kda_chunk_fwd_noalloc(
        _p(inp["q"]), _p(inp["k"]), _p(inp["v"]), kda.BF16, _p(g), _p(inp["beta"]), None,
        _p(inp["cu_seqlens"]), 1, 1, NT, H, 128, 128, _p(o), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 5
    assert b"scratch" in kda.lib.kda_last_error_string()
