"""GPU parity of the gate (K1) and the decode step (K5) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_close, errors, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import chunked_gated_delta_fwd_gb300 as m

    return m


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gate_matches_oracle(kda, dtype):
    w = workloads.custom([300], H=3, dtype=dtype, z_std=3.0, A_range=1.0, seed=41)
    inp = workloads.make_inputs(w, "cpu")
    g = kda.gate(inp["z"].cuda(), inp["A"].cuda())
    ref = oracle.gate(inp["z"], inp["A"])
    _, mabs = errors(g, ref)
    assert mabs <= 2e-6, mabs
    assert float(g.max()) <= 0.0 and float(g.min()) >= -5.0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gate_softplus_matches_oracle(kda, dtype):
    """The unbounded gate, z ~ N(0, 9) and A in [-1, 1]: relative error <= 1e-6
    elementwise (fp32 arithmetic), g far below -5 where z is large."""
    w = workloads.custom([300], H=3, dtype=dtype, z_std=3.0, A_range=1.0, seed=43)
    inp = workloads.make_inputs(w, "cpu")
    g = kda.gate_softplus(inp["z"].cuda(), inp["A"].cuda())
    ref = oracle.gate_softplus(inp["z"], inp["A"])
    rel = np.max(np.abs(to64(g) - ref) / np.abs(ref))
    assert rel <= 1e-6, rel
    assert float(g.max()) < 0.0 and float(g.min()) < -5.0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gate_chunk_cumsum_matches_oracle(kda, dtype):
    lens = [100, 0, 200, 1, 64, 65]
    w = workloads.custom(lens, H=2, dtype=dtype, seed=42)
    inp = workloads.make_inputs(w, "cpu")
    cu = inp["cu_seqlens"]
    g, gc = kda.gate(inp["z"].cuda(), inp["A"].cuda(), with_cumsum=True, cu_seqlens=cu.cuda())
    g_ref = oracle.gate(inp["z"], inp["A"])
    assert errors(g, g_ref)[1] <= 2e-6
    assert errors(gc, oracle.chunk_cumsum(g_ref, cu))[1] <= 1e-4
    # without cu_seqlens: one sequence
    g1, gc1 = kda.gate(inp["z"].cuda(), inp["A"].cuda(), with_cumsum=True)
    assert errors(gc1, oracle.chunk_cumsum(g_ref, None))[1] <= 1e-4


def _decode_case(kda, N, H, dtype, steps, seed, sample=None):
    """Runs `steps` decode steps on the GPU from a seeded state; the oracle follows
    the sampled (n, h) states.  Gate on both sides (GPU gate vs oracle gate)."""
    w = workloads.DecodeWorkload("t", N=N, H=H, dtype=dtype, steps=steps, seed=seed)
    S = workloads.make_decode_state(w, "cuda")
    if sample is None:
        sel = [(n, h) for n in range(N) for h in range(H)]
    else:
        r = np.random.default_rng(seed)
        sel = sorted({(int(r.integers(N)), int(r.integers(H))) for _ in range(sample)})
    ns = torch.tensor([s[0] for s in sel])
    hs = torch.tensor([s[1] for s in sel])
    S_ref = to64(S[ns, hs])[:, None]  # [m, 1, dv, dk]
    worst = (0.0, 0.0)
    for step in range(steps):
        inp = workloads.make_decode_step(w, step, "cuda")
        g = kda.gate(inp["z"], inp["A"])
        o = kda.recurrent_step(inp["q"], inp["k"], inp["v"], g, inp["beta"], S)
        pick = lambda t: t[ns, hs].unsqueeze(1)
        z_sel = to64(pick(inp["z"]))  # [m, 1, dk]
        A_sel = to64(inp["A"][hs])  # per sample
        g_ref = np.stack([oracle.gate(z_sel[i:i + 1], A_sel[i:i + 1]) for i in range(len(sel))])[:, 0]
        o_ref, S_ref = oracle.decode_step(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]), g_ref,
                                          pick(inp["beta"]), S_ref)
        rel, mabs = assert_close(o[ns, hs].unsqueeze(1), o_ref, dtype, f"o step {step}")
        worst = (max(worst[0], rel), max(worst[1], mabs))
    assert_close(S[ns, hs].unsqueeze(1), S_ref, dtype, "final state")
    return worst


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_small(kda, dtype):
    _decode_case(kda, N=5, H=3, dtype=dtype, steps=4, seed=51)


def test_decode_full_size_sampled(kda):
    """512 sequences x 96 heads, fp32 state (3.2 GB), 100 in-place steps; the
    oracle follows 48 sampled (sequence, head) states through all steps."""
    _decode_case(kda, N=512, H=96, dtype=torch.bfloat16, steps=100, seed=1005, sample=48)


def test_decode_zero_sequences_is_noop(kda):
    S = torch.zeros(0, 2, 128, 128, device="cuda")
    q = torch.zeros(0, 2, 128, device="cuda", dtype=torch.bfloat16)
    o = kda.recurrent_step(q, q, q, torch.zeros(0, 2, 128, device="cuda"),
                           torch.zeros(0, 2, device="cuda", dtype=torch.bfloat16), S)
    assert o.shape == (0, 2, 128)


# ------------------------------------------------------ several tokens per step
def _multi_inputs(N, T, H, dtype, seed):
    w = workloads.custom([T] * N, H=H, dtype=dtype, seed=seed, h0_std=0.5)
    inp = workloads.make_inputs(w, "cpu")
    g = workloads.uniform_decay((N * T, H, 128), "cpu", seed=seed + 1, lo=-5.0, hi=0.0)
    return inp, g


def _multi_reference(inp, g, N, T, adv):
    """Outputs of all tokens, and the state after the first adv[n] tokens, from the
    oracle (the truncated sequences run as a packed batch)."""
    o_ref, _ = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                 inp["cu_seqlens"])
    rows = torch.cat([torch.arange(n * T, n * T + a) for n, a in enumerate(adv)]).long()
    cu = torch.tensor([0] + list(np.cumsum(adv)), dtype=torch.int32)
    sel = lambda t: t[rows]
    _, h_ref = oracle.recurrence(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(g),
                                 sel(inp["beta"]), inp["h0"], cu)
    return o_ref, h_ref


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_multi_step_outputs_and_partial_commit(kda, dtype):
    """N=5 sequences of T=6 draft tokens, H=3: outputs of all tokens, and each
    state advanced by its own accepted count (0, 1, 3, 6, 6)."""
    N, T, H = 5, 6, 3
    inp, g = _multi_inputs(N, T, H, dtype, seed=61)
    adv = [0, 1, 3, 6, 6]
    S = inp["h0"].clone().cuda()
    shp = lambda t: t.cuda().view(N, T, *t.shape[1:])
    o = kda.recurrent_multi_step(shp(inp["q"]), shp(inp["k"]), shp(inp["v"]), shp(g),
                                 shp(inp["beta"]), S,
                                 torch.tensor(adv, dtype=torch.int32, device="cuda"))
    o_ref, h_ref = _multi_reference(inp, g, N, T, adv)
    assert_close(o.view(N * T, H, 128), o_ref, dtype, "o multi")
    assert_close(S, h_ref, dtype, "S multi")


def test_multi_step_full_advance_and_state_only(kda):
    """n_advance omitted advances all T tokens; with outputs off only S changes."""
    N, T, H = 4, 16, 2
    inp, g = _multi_inputs(N, T, H, torch.bfloat16, seed=63)
    shp = lambda t: t.cuda().view(N, T, *t.shape[1:])
    S1 = inp["h0"].clone().cuda()
    o = kda.recurrent_multi_step(shp(inp["q"]), shp(inp["k"]), shp(inp["v"]), shp(g),
                                 shp(inp["beta"]), S1)
    S2 = inp["h0"].clone().cuda()
    none = kda.recurrent_multi_step(shp(inp["q"]), shp(inp["k"]), shp(inp["v"]), shp(g),
                                    shp(inp["beta"]), S2, return_outputs=False)
    assert none is None
    o_ref, h_ref = _multi_reference(inp, g, N, T, [T] * N)
    assert_close(o.view(N * T, H, 128), o_ref, torch.bfloat16, "o multi full")
    assert_close(S1, h_ref, torch.bfloat16, "S multi full")
    assert torch.equal(S1, S2)


def test_multi_step_one_token_matches_recurrent_step(kda):
    """T = 1 against the single-token decode step, both against the oracle."""
    N, H = 7, 4
    inp, g = _multi_inputs(N, 1, H, torch.bfloat16, seed=65)
    S_multi = inp["h0"].clone().cuda()
    S_one = inp["h0"].clone().cuda()
    o_multi = kda.recurrent_multi_step(*(t.cuda().view(N, 1, *t.shape[1:]) for t in
                                         (inp["q"], inp["k"], inp["v"], g, inp["beta"])),
                                       S_multi)
    o_one = kda.recurrent_step(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), g.cuda(),
                               inp["beta"].cuda(), S_one)
    o_ref, h_ref = _multi_reference(inp, g, N, 1, [1] * N)
    assert_close(o_multi.view(N, H, 128), o_ref, torch.bfloat16, "o multi T=1")
    assert_close(o_one, o_ref, torch.bfloat16, "o step")
    assert_close(S_multi, h_ref, torch.bfloat16, "S multi T=1")
    assert_close(S_one, h_ref, torch.bfloat16, "S step")


def test_multi_step_full_size_sampled(kda):
    """512 sequences x 96 heads, fp32 state (3.2 GB), 4 tokens per sequence with a
    partial commit (accepted prefix 0..4 tokens), as the bench runs it; 24 sampled
    (sequence, head) pairs against the oracle (outputs of all 4 tokens, the state
    after the accepted prefix)."""
    dw = workloads.decode()
    N, H, T = dw.N, dw.H, 4
    S = workloads.make_decode_state(dw, "cuda")
    steps = [workloads.make_decode_step(dw, i, "cuda") for i in range(T)]
    stack = lambda key: torch.stack([st[key] for st in steps], dim=1).contiguous()  # [N, T, ...]
    q, k, v, beta, z = stack("q"), stack("k"), stack("v"), stack("beta"), stack("z")
    A = steps[0]["A"]
    g = kda.gate(z, A)  # the GPU run's gate; the oracle forms its own from z
    adv = (torch.arange(N, dtype=torch.int32) % (T + 1)).cuda()
    r = np.random.default_rng(7)
    pairs = sorted({(int(r.integers(N)), int(r.integers(H))) for _ in range(24)})
    S0 = {p: S[p[0], p[1]].cpu().clone() for p in pairs}
    o = kda.recurrent_multi_step(q, k, v, g, beta, S, adv)
    torch.cuda.synchronize()
    for n, h in pairs:
        a = int(adv[n])
        seq = lambda t: t[n, :, h:h + 1]  # [T, 1, ...]
        g_ref = oracle.gate(seq(z), A[h:h + 1])
        o_ref, _ = oracle.recurrence(seq(q), seq(k), seq(v), g_ref, seq(beta),
                                     S0[(n, h)].view(1, 1, 128, 128))
        assert_close(o[n, :, h:h + 1], o_ref, torch.bfloat16, f"o seq {n} head {h}")
        if a > 0:
            _, s_ref = oracle.recurrence(seq(q)[:a], seq(k)[:a], seq(v)[:a], g_ref[:a],
                                         seq(beta)[:a], S0[(n, h)].view(1, 1, 128, 128))
        else:
            s_ref = S0[(n, h)].view(1, 1, 128, 128)
        assert_close(S[n, h:h + 1].unsqueeze(0), s_ref, torch.bfloat16, f"state seq {n} head {h}")
