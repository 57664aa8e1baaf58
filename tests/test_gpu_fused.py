"""GPU parity of kda_chunk_fwd_fused (prologue and epilogue fused) against the oracle.

The oracle side runs the steps one after another in fp64: q and k L2-normalised
(``oracle.l2_normalize``), the gate from z (``oracle.gate``), the recurrence, and
the head-wise RMSNorm x Sigmoid output gate (``oracle.output_gate``).  q and k
are drawn off unit norm (rows scaled by 0.25 .. 4) so that the normalisation
matters.  Tolerances are the bf16 ones of ``gpu_helpers``; for the gated output
the max-abs bound applies to the error carried back to the units of o
(``assert_close_gated``).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_close, assert_close_gated

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import chunked_gated_delta_fwd_gb300 as m

    return m


def _case(lens, H, seed, h0=True, scale_qk=True):
    w = workloads.custom(lens, H=H, dtype=torch.bfloat16, seed=seed, h0_std=0.3 if h0 else None)
    inp = workloads.make_inputs(w, "cpu")
    gen = torch.Generator().manual_seed(seed + 7)
    NT = w.n_tokens
    sq = 0.25 + 3.75 * torch.rand(NT, H, 1, generator=gen)
    sk = 0.25 + 3.75 * torch.rand(NT, H, 1, generator=gen)
    if scale_qk:  # rows off unit norm; otherwise the workload's unit rows
        inp["q"] = (inp["q"].float() * sq).to(torch.bfloat16)
        inp["k"] = (inp["k"].float() * sk).to(torch.bfloat16)
    inp["gz"] = (2.0 * torch.randn(NT, H, 128, generator=gen)).to(torch.bfloat16)
    inp["w"] = 0.5 + torch.rand(128, generator=gen)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    return inp, dev


def _reference(inp, qk_eps, use_gate, use_w, eps, g=None):
    q, k = inp["q"], inp["k"]
    if qk_eps is not None:
        q, k = oracle.l2_normalize(q, qk_eps), oracle.l2_normalize(k, qk_eps)
    if g is None:
        g = oracle.gate(inp["z"], inp["A"])
    o, hT = oracle.recurrence(q, k, inp["v"], g, inp["beta"], inp["h0"], inp["cu_seqlens"])
    y = oracle.output_gate(o, inp["gz"], inp["w"] if use_w else None, eps) if use_gate else None
    return o, y, hT


def _check(o, hT, inp, ref, use_gate, use_w, eps, what):
    o_ref, y_ref, h_ref = ref
    if use_gate:
        assert_close_gated(o, y_ref, o_ref, inp["gz"], inp["w"] if use_w else None, eps,
                           f"y {what}")
    else:
        assert_close(o, o_ref, torch.bfloat16, f"o {what}")
    assert_close(hT, h_ref, torch.bfloat16, f"hT {what}")


@pytest.mark.parametrize("qk,gate,wt,flags", [(True, True, True, 0), (True, False, False, 0),
                                              (False, True, False, 0), (False, True, True, 0),
                                              (True, True, True, 32)],
                         ids=["all", "qk-only", "gate-only", "gate+w", "all-precise"])
def test_fused_varlen(kda, qk, gate, wt, flags):
    lens = [5, 0, 70, 64, 129, 1, 300]
    inp, dev = _case(lens, H=3, seed=81, scale_qk=qk)  # without the norm: unit rows
    qk_eps = 1e-6 if qk else None
    o, hT = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"], dev["cu_seqlens"],
                                z=dev["z"], A=dev["A"], qk_l2_eps=qk_eps,
                                out_gate=dev["gz"] if gate else None,
                                out_norm_weight=dev["w"] if wt else None, out_norm_eps=1e-5,
                                flags=flags)
    kda.get_device_error()
    _check(o, hT, inp, _reference(inp, qk_eps, gate, wt, 1e-5), gate, wt, 1e-5, "fused")


def test_fused_with_g_and_segments(kda):
    """g given directly, a 1489-token sequence cut into segments of 3 chunks plus a
    short one: the gate is applied wherever outputs are written (serial phase of
    the first segment and the rerun of the others)."""
    lens = [64 * 23 + 17, 200]
    inp, dev = _case(lens, H=2, seed=83)
    g = workloads.uniform_decay((sum(lens), 2, 128), "cpu", seed=84)
    o, hT = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                                dev["cu_seqlens"], g=g.cuda(), qk_l2_eps=1e-6,
                                out_gate=dev["gz"], out_norm_weight=dev["w"], out_norm_eps=1e-6,
                                flags=kda.segment_chunks(3))
    kda.get_device_error()
    _check(o, hT, inp, _reference(inp, 1e-6, True, True, 1e-6, g=g), True, True, 1e-6,
           "fused segmented")


def test_gate_in_the_chain_agrees_with_the_standalone_kernel(kda):
    """The output gate applied by the chain's store warps (from o in fp32) against
    kda_output_gate on the ungated bf16 o of the same prefill: the two differ only
    by where o is rounded to bf16 and by the approximate sigmoid, so every element
    agrees within a few bf16 roundings of |y|, plus a 1e-6 floor near zero."""
    lens = [5, 0, 70, 64, 129, 1, 300]
    inp, dev = _case(lens, H=3, seed=88)
    kw = dict(z=dev["z"], A=dev["A"], qk_l2_eps=1e-6)
    y, _ = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                               dev["cu_seqlens"], out_gate=dev["gz"], out_norm_weight=dev["w"],
                               out_norm_eps=1e-6, **kw)
    o, _ = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                               dev["cu_seqlens"], **kw)
    y2 = kda.output_gate(o, dev["gz"], dev["w"], 1e-6)
    a, b = y.double(), y2.double()
    assert bool((a - b).abs().le(4 * 2.0 ** -8 * b.abs() + 1e-6).all()), \
        float(((a - b).abs() / (b.abs() + 1e-6)).max())


def test_fused_scalar_gate_equals_broadcast(kda):
    """Scalar gates ([NT, H], SCALAR_GATE) with q/k normalisation and the output
    gate give the same bits as the broadcast [NT, H, 128] gate; with q/k
    normalisation alone they agree with the oracle.  (One decay for all channels
    forgets the state in every channel at once, so a few rows of o come out ~100x
    below the median; the output RMSNorm scales each row to unit size and would
    weigh those rows' rounding 100x, which says nothing about the kernels.)"""
    lens = [300, 0, 77]
    inp, dev = _case(lens, H=2, seed=86)
    g1 = workloads.uniform_decay((sum(lens), 2), "cpu", seed=87)
    gb = g1[..., None].expand(-1, -1, 128).contiguous()
    kw = dict(qk_l2_eps=1e-6, out_gate=dev["gz"], out_norm_weight=dev["w"], out_norm_eps=1e-6)
    o1, h1 = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                                 dev["cu_seqlens"], g=g1.cuda(), flags=kda.SCALAR_GATE, **kw)
    o2, h2 = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                                 dev["cu_seqlens"], g=gb.cuda(), **kw)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    o3, h3 = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                                 dev["cu_seqlens"], g=g1.cuda(), flags=kda.SCALAR_GATE,
                                 qk_l2_eps=1e-6)
    _check(o3, h3, inp, _reference(inp, 1e-6, False, False, 1e-6, g=gb), False, False, 1e-6,
           "fused scalar gate")


def test_fused_without_options_equals_gated(kda):
    """No normalisation and no output gate: the same kernels as kda_chunk_fwd_gated,
    bit for bit."""
    lens = [300, 77]
    _, dev = _case(lens, H=2, seed=85)
    o1, h1 = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                                 dev["cu_seqlens"], z=dev["z"], A=dev["A"])
    o2, h2 = kda.chunk_fwd_gated(dev["q"], dev["k"], dev["v"], dev["z"], dev["A"], dev["beta"],
                                 dev["h0"], dev["cu_seqlens"])
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_fused_full_size_sampled(kda):
    """B=1, T=8192, H=96 with every fusion on, checked on two heads against the
    oracle (the other heads run in the same launch)."""
    w = workloads.prefill()
    dev = workloads.make_inputs(w, "cuda")
    gen = torch.Generator(device="cuda").manual_seed(86)
    NT, H = w.n_tokens, w.H
    q = (dev["q"].float() * (0.25 + 3.75 * torch.rand(NT, H, 1, generator=gen, device="cuda"))).to(torch.bfloat16)
    gz = (2.0 * torch.randn(NT, H, 128, generator=gen, device="cuda")).to(torch.bfloat16)
    wt = 0.5 + torch.rand(128, generator=gen, device="cuda")
    o, hT = kda.chunk_fwd_fused(q, dev["k"], dev["v"], dev["beta"], dev["h0"], dev["cu_seqlens"],
                                z=dev["z"], A=dev["A"], qk_l2_eps=1e-6, out_gate=gz,
                                out_norm_weight=wt, out_norm_eps=1e-6)
    torch.cuda.synchronize()
    for h in (5, 77):
        sl = lambda t: t[:, h:h + 1]
        qn, kn = oracle.l2_normalize(sl(q), 1e-6), oracle.l2_normalize(sl(dev["k"]), 1e-6)
        g = oracle.gate(sl(dev["z"]), dev["A"][h:h + 1])
        o_ref, h_ref = oracle.recurrence(qn, kn, sl(dev["v"]), g, sl(dev["beta"]),
                                         dev["h0"][:, h:h + 1])
        y_ref = oracle.output_gate(o_ref, sl(gz), wt, 1e-6)
        assert_close_gated(sl(o), y_ref, o_ref, sl(gz), wt, 1e-6, f"y head {h}")
        assert_close(hT[:, h:h + 1], h_ref, torch.bfloat16, f"hT head {h}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_output_gate_kernel(kda, dtype):
    """kda_output_gate on given outputs (row scales 1e-3 .. 10) against the oracle:
    fp32 rel_L2 <= 1e-5; bf16 elementwise |y - y_ref| <= 2^-8 |y_ref| (one bf16
    rounding of y after fp32 arithmetic on the given bf16 inputs); in place too."""
    gen = torch.Generator().manual_seed(87)
    NT, H = 300, 3
    o = torch.randn(NT, H, 128, generator=gen) * torch.logspace(-3, 1, NT).view(NT, 1, 1)
    x = 3.0 * torch.randn(NT, H, 128, generator=gen)
    w = 0.5 + torch.rand(128, generator=gen)
    o, x = o.to(dtype), x.to(dtype)
    y = kda.output_gate(o.cuda(), x.cuda(), w.cuda(), 1e-6)
    ref = oracle.output_gate(o, x, w, 1e-6)
    if dtype == torch.float32:
        assert_close(y, ref, torch.float32, "output gate f32")
    else:
        err = np.abs(y.cpu().double().numpy() - ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-30), float(np.max(err / np.abs(ref)))
    oc = o.cuda()
    kda.output_gate(oc, x.cuda(), w.cuda(), 1e-6, out=oc)
    assert torch.equal(oc, y)
