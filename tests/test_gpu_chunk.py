"""GPU parity of the chunked prefill (kda_chunk_fwd) against the fp64 oracle.

Small cases cover ragged tails (T = 1 .. 200 around the 16-token tile and the
64-token chunk), variable-length packing with empty sequences, initial states,
near-bound decays and both evaluation paths for bf16 inputs (tensor cores and
fp32 CUDA cores).  Full-size workloads are checked on sampled heads or
sequences, or on the prefix the oracle can afford.
"""

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


def _inputs(lens, H, dtype, seed, h0=True, g_lo=-5.0, g_hi=0.0, device="cuda"):
    w = workloads.custom(lens, H=H, dtype=dtype, seed=seed, h0_std=0.5 if h0 else None)
    inp = workloads.make_inputs(w, "cpu")
    NT = w.n_tokens
    g = workloads.uniform_decay((NT, H, 128), "cpu", seed=seed + 1, lo=g_lo, hi=g_hi)
    dev = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dev["g"] = g.to(device)
    return inp, g, dev


def _run(kda, dev, flags=0, varlen=True):
    return kda.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"],
                         dev["cu_seqlens"] if varlen else None, flags=flags)


PRECISE = 32  # KDA_CHUNK_PRECISE: the tensor-core path with the state update at tf32
PATHS = [(torch.float32, 0), (torch.bfloat16, 0), (torch.bfloat16, 1), (torch.bfloat16, PRECISE)]
PATH_IDS = ["f32", "bf16-tc", "bf16-f32cores", "bf16-tc-precise"]


@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 127, 200])
@pytest.mark.parametrize("dtype,flags", PATHS, ids=PATH_IDS)
def test_single_sequence_ragged(kda, T, dtype, flags):
    inp, g, dev = _inputs([T], H=2, dtype=dtype, seed=100 + T)
    o, hT = _run(kda, dev, flags)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, f"o T={T}")
    assert_close(hT, h_ref, dtype, f"hT T={T}")


@pytest.mark.parametrize("dtype,flags", PATHS, ids=PATH_IDS)
def test_varlen_with_empty_sequences(kda, dtype, flags):
    lens = [5, 0, 70, 64, 129, 1, 0, 300]
    inp, g, dev = _inputs(lens, H=3, dtype=dtype, seed=7)
    o, hT = _run(kda, dev, flags)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, "o varlen")
    assert_close(hT, h_ref, dtype, "hT varlen")


@pytest.mark.parametrize("dtype,flags", PATHS, ids=PATH_IDS)
def test_batched_without_cu_seqlens(kda, dtype, flags):
    B, T, H = 3, 130, 2
    inp, g, dev = _inputs([T] * B, H=H, dtype=dtype, seed=9)
    shp = lambda t: t.view(B, T, *t.shape[1:])
    o, hT = kda.chunk_fwd(shp(dev["q"]), shp(dev["k"]), shp(dev["v"]), shp(dev["g"]),
                          shp(dev["beta"]), dev["h0"], None, flags=flags)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o.view(B * T, H, 128), o_ref, dtype, "o batched")
    assert_close(hT, h_ref, dtype, "hT batched")


@pytest.mark.parametrize("dtype,flags", PATHS, ids=PATH_IDS)
def test_near_bound_decay_and_zero_state(kda, dtype, flags):
    """All decays in [-5, -4.5]: every 16-token tile sits near the e^80 edge."""
    inp, g, dev = _inputs([256, 77], H=2, dtype=dtype, seed=11, h0=False, g_lo=-5.0, g_hi=-4.5)
    o, hT = _run(kda, dev, flags)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], None,
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, "o near-bound")
    assert_close(hT, h_ref, dtype, "hT near-bound")


@pytest.mark.parametrize("dtype,flags", PATHS, ids=PATH_IDS)
def test_no_decay_slow_forgetting(kda, dtype, flags):
    """g in [-0.01, 0]: almost no forgetting, the state accumulates over 4 chunks."""
    inp, g, dev = _inputs([256], H=2, dtype=dtype, seed=12, g_lo=-0.01, g_hi=0.0)
    o, hT = _run(kda, dev, flags)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, "o slow decay")
    assert_close(hT, h_ref, dtype, "hT slow decay")


# (dtype, flags, key noise): keys = normalise(base + noise * N(0, 1)) per head, so
# k_i . k_j is about 0.99 at noise 0.1 and 0.92 at 0.3.  The fp32 paths and the
# tensor-core path with the precise state update are held to the bound at 0.1; the
# default tensor-core path, whose Kt and Vt enter the state update in bf16, is a
# little over it there (final state rel-L2 1.2e-2 at 0.1, 1.0e-2 at 0.15, measured)
# and is held to it at 0.3 (7.8e-3).
CORRELATED = [(torch.float32, 0, 0.1), (torch.bfloat16, 1, 0.1), (torch.bfloat16, PRECISE, 0.1),
              (torch.bfloat16, 0, 0.3)]


@pytest.mark.parametrize("dtype,flags,noise", CORRELATED,
                         ids=["f32", "bf16-f32cores", "bf16-tc-precise", "bf16-tc"])
def test_correlated_keys_full_erase(kda, dtype, flags, noise):
    """beta = 1 and the keys of each head nearly parallel under slow decay: the
    strictly lower A_kk has entries near 1 in every block, so the fp32 inverse and
    the W/U products work with large, nearly cancelling terms."""
    inp, g, dev = _inputs([200, 64], H=2, dtype=dtype, seed=21, g_lo=-0.05, g_hi=0.0)
    gen = torch.Generator().manual_seed(22)
    NT = inp["k"].shape[0]
    base = torch.randn(1, 2, 128, generator=gen, dtype=torch.float64)
    k = base + noise * torch.randn(NT, 2, 128, generator=gen, dtype=torch.float64)
    k = (k / k.norm(dim=-1, keepdim=True)).to(dtype)
    inp["k"] = k
    inp["beta"] = torch.ones_like(inp["beta"])
    dev["k"] = k.cuda()
    dev["beta"] = inp["beta"].cuda()
    o, hT = _run(kda, dev, flags)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, "o correlated keys")
    assert_close(hT, h_ref, dtype, "hT correlated keys")


def test_correlated_keys_default_tc_limit(kda):
    """The stated limit of the default tensor-core path on the hardest correlated
    case (noise 0.1, k_i . k_j ~ 0.99, beta = 1, slow decay): its final state is
    about 1.2e-2 from the oracle in relative L2, over the bf16 bound of 1e-2, while
    the precise state update on the same inputs is inside it.  Pinned here so that
    the limit the header states cannot grow unnoticed (the run is deterministic)."""
    inp, g, dev = _inputs([200, 64], H=2, dtype=torch.bfloat16, seed=21, g_lo=-0.05, g_hi=0.0)
    gen = torch.Generator().manual_seed(22)
    NT = inp["k"].shape[0]
    base = torch.randn(1, 2, 128, generator=gen, dtype=torch.float64)
    k = base + 0.1 * torch.randn(NT, 2, 128, generator=gen, dtype=torch.float64)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    inp["k"] = k
    inp["beta"] = torch.ones_like(inp["beta"])
    dev["k"] = k.cuda()
    dev["beta"] = inp["beta"].cuda()
    _, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                 inp["cu_seqlens"])
    _, hT = _run(kda, dev, 0)
    rel_default, _ = errors(hT, h_ref)
    _, hT_p = _run(kda, dev, PRECISE)
    rel_precise, _ = errors(hT_p, h_ref)
    assert rel_default <= 1.5e-2, f"default tensor-core path: hT rel_L2 {rel_default:.3e}"
    assert rel_precise <= 1e-2, f"precise state update: hT rel_L2 {rel_precise:.3e}"
    assert rel_precise < rel_default


def test_final_state_may_alias_initial_state(kda):
    inp, g, dev = _inputs([100, 40], H=2, dtype=torch.bfloat16, seed=13)
    h = dev["h0"].clone()
    kda.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], h, dev["cu_seqlens"],
                  final_state_out=h)
    _, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                 inp["cu_seqlens"])
    assert_close(h, h_ref, torch.bfloat16, "aliased hT")


def test_all_sequences_empty_returns_initial_state(kda):
    H = 2
    h0 = torch.randn(3, H, 128, 128, device="cuda")
    z = torch.zeros(0, H, 128, device="cuda", dtype=torch.bfloat16)
    cu = torch.zeros(4, dtype=torch.int32, device="cuda")
    _, hT = kda.chunk_fwd(z, z, z, torch.zeros(0, H, 128, device="cuda"),
                          torch.zeros(0, H, device="cuda", dtype=torch.bfloat16), h0, cu)
    assert torch.equal(hT, h0)


def test_bad_cu_seqlens_is_reported_not_faulted(kda):
    inp, g, dev = _inputs([64, 64], H=1, dtype=torch.bfloat16, seed=14)
    bad = torch.tensor([0, 100, 50], dtype=torch.int32, device="cuda")  # decreasing
    kda.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], None, bad)
    with pytest.raises(kda.KdaError) as ei:
        kda.get_device_error()
    assert ei.value.status == 1
    kda.get_device_error()  # cleared


def test_tiny_fp32_workload_end_to_end(kda):
    """B=1, H=2, T=256, fp32 inputs, A=0, zero state: gate + chunked prefill on the
    GPU against the oracle's gate + recurrence, relative L2 <= 1e-5."""
    w = workloads.tiny()
    inp = workloads.make_inputs(w, "cpu")
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g = kda.gate(dev["z"], dev["A"])
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g, dev["beta"], None, dev["cu_seqlens"])
    g_ref = oracle.gate(inp["z"], inp["A"])
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g_ref, inp["beta"], None,
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.float32, "o tiny")
    assert_close(hT, h_ref, torch.float32, "hT tiny")


def _full_size(kda, w, sample_pairs, seed, gated=False):
    """Runs gate + chunk (or the fused-gate chunk) on a full-size workload (inputs
    generated on the GPU) and checks sampled (sequence, head) pairs against the oracle."""
    dev = workloads.make_inputs(w, "cuda")
    if gated:
        o, hT = kda.chunk_fwd_gated(dev["q"], dev["k"], dev["v"], dev["z"], dev["A"],
                                    dev["beta"], dev["h0"], dev["cu_seqlens"])
    else:
        g = kda.gate(dev["z"], dev["A"])
        o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g, dev["beta"], dev["h0"],
                              dev["cu_seqlens"])
    torch.cuda.synchronize()
    cu = dev["cu_seqlens"].cpu().numpy().astype(np.int64)
    r = np.random.default_rng(seed)
    pairs = sorted({(int(r.integers(w.n_seqs)), int(r.integers(w.H))) for _ in range(sample_pairs)})
    for n, h in pairs:
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda t: t[a:b, h:h + 1]
        g_ref = oracle.gate(sl(dev["z"]), dev["A"][h:h + 1])
        h0 = None if dev["h0"] is None else dev["h0"][n:n + 1, h:h + 1]
        o_ref, h_ref = oracle.recurrence(sl(dev["q"]), sl(dev["k"]), sl(dev["v"]), g_ref,
                                         sl(dev["beta"]), h0)
        assert_close(sl(o), o_ref, w.dtype, f"o seq {n} head {h}")
        assert_close(hT[n:n + 1, h:h + 1], h_ref, w.dtype, f"hT seq {n} head {h}")


def test_prefill_full_size_sampled(kda):
    """B=1, T=8192, H=96, bf16, random h0: 12 sampled heads against the oracle."""
    _full_size(kda, workloads.prefill(), 12, seed=2)


def test_varlen_full_size_sampled(kda):
    """32 packed sequences (~270K tokens), H=96: 6 sampled (sequence, head) pairs."""
    _full_size(kda, workloads.varlen(), 6, seed=3)


def test_prefill_full_size_sampled_gated(kda):
    """The same workload through kda_chunk_fwd_gated (gate formed inside the kernels)."""
    _full_size(kda, workloads.prefill(), 12, seed=4, gated=True)


def test_varlen_full_size_sampled_gated(kda):
    _full_size(kda, workloads.varlen(), 6, seed=5, gated=True)


@pytest.mark.parametrize("z_scale,A_val", [(1.0, None), (6.0, 1.0), (6.0, -3.0)],
                         ids=["random-A", "near-bound", "slow"])
def test_gated_ragged_varlen(kda, z_scale, A_val):
    """Fused gate on ragged packed sequences (empty ones included): decays spread
    over (-5, 0), pushed to the -5 bound (z, A large) and to almost no decay."""
    lens = [5, 0, 70, 64, 129, 1, 0, 300, 17]
    w = workloads.custom(lens, H=3, dtype=torch.bfloat16, seed=21, h0_std=0.5)
    inp = workloads.make_inputs(w, "cpu")
    z = (inp["z"].float() * z_scale).to(torch.bfloat16)
    A = inp["A"] if A_val is None else torch.full_like(inp["A"], A_val)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o, hT = kda.chunk_fwd_gated(dev["q"], dev["k"], dev["v"], z.cuda(), A.cuda(), dev["beta"],
                                dev["h0"], dev["cu_seqlens"])
    g_ref = oracle.gate(z, A)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g_ref, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o gated")
    assert_close(hT, h_ref, torch.bfloat16, "hT gated")


def test_precise_mode_with_fused_gate_and_checkpoints(kda):
    """The precise state update behind the fused gate (z read by the prepare kernel,
    Kt written in fp32 straight to the workspace) and with state checkpoints."""
    lens = [5, 0, 70, 64, 129, 300, 17]
    w = workloads.custom(lens, H=3, dtype=torch.bfloat16, seed=23, h0_std=0.5)
    inp = workloads.make_inputs(w, "cpu")
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o, hT = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"],
                                dev["cu_seqlens"], z=dev["z"], A=dev["A"], flags=PRECISE)
    g_ref = oracle.gate(inp["z"], inp["A"])
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g_ref, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o precise gated")
    assert_close(hT, h_ref, torch.bfloat16, "hT precise gated")
    g = kda.gate(dev["z"], dev["A"])
    o2, h2, ck = kda.chunk_fwd_checkpointed(dev["q"], dev["k"], dev["v"], g, dev["beta"],
                                            dev["h0"], dev["cu_seqlens"], ckpt_tokens=64,
                                            flags=PRECISE)
    assert_close(o2, o_ref, torch.bfloat16, "o precise checkpointed")
    assert_close(h2, h_ref, torch.bfloat16, "hT precise checkpointed")
    ck_ref = _oracle_checkpoints(dict(inp), g_ref, lens, 64)
    assert ck.shape[0] == ck_ref.shape[0]
    for i in range(ck.shape[0]):
        assert_close(ck[i], ck_ref[i], torch.bfloat16, f"checkpoint {i}")


def test_gated_rejects_fp32(kda):
    w = workloads.custom([64], H=2, dtype=torch.float32, seed=1)
    dev = workloads.make_inputs(w, "cuda")
    with pytest.raises(kda.KdaError):
        kda.chunk_fwd_gated(dev["q"], dev["k"], dev["v"], dev["z"], dev["A"], dev["beta"], None,
                            dev["cu_seqlens"])


def test_long_context_full_instance(kda):
    """The long-context workload itself (B=1, T=1,048,576, H=16, z ~ N(0, 2)) run as
    the benchmark runs it -- kda_chunk_fwd_gated, the chain cut into automatic
    segments joined by the end-state scan ("Kimi K3 technical report review",
    section 8.1, Eq. 17):
      * its first 4096 outputs equal a run on the 4096-token prefix (causality),
        and that prefix run matches the oracle on every head;
      * one head's o over all 1,048,576 tokens and its final state match the oracle
        (token-by-token fp64 recurrence, about half a minute on one host thread);
      * every head's final state matches the serial chain (KDA_CHUNK_SEQUENTIAL)."""
    w = workloads.long_context()
    dev = workloads.make_inputs(w, "cuda")
    P = 4096
    o_full, h_full = kda.chunk_fwd_gated(dev["q"], dev["k"], dev["v"], dev["z"], dev["A"],
                                         dev["beta"], None, dev["cu_seqlens"])
    pre = workloads.make_inputs(w, "cuda", tokens=P)  # the same values, drawn on their own
    for key in ("q", "k", "v", "z", "beta"):
        assert torch.equal(pre[key], dev[key][:P]), key
    oP, hP = kda.chunk_fwd_gated(pre["q"], pre["k"], pre["v"], pre["z"], pre["A"], pre["beta"],
                                 None, pre["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(o_full[:P], oP)
    g_ref = oracle.gate(pre["z"], pre["A"])
    o_ref, h_ref = oracle.recurrence(pre["q"], pre["k"], pre["v"], g_ref, pre["beta"], None)
    assert_close(oP, o_ref, torch.bfloat16, "o prefix")
    assert_close(hP, h_ref, torch.bfloat16, "hT prefix")
    del pre, oP, hP, o_ref, h_ref, g_ref
    # the serial chain on the same instance: hT of every head
    _, h_seq = kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], None,
                                   dev["cu_seqlens"], z=dev["z"], A=dev["A"],
                                   flags=kda.SEQUENTIAL)
    torch.cuda.synchronize()
    assert_close(h_full, h_seq.double(), torch.bfloat16, "hT segmented vs serial")
    # one head over the whole sequence against the oracle
    h = 11
    sl = lambda t: t[:, h:h + 1]
    g_ref = oracle.gate(sl(dev["z"]), dev["A"][h:h + 1])
    o_ref, h_ref = oracle.recurrence(sl(dev["q"]), sl(dev["k"]), sl(dev["v"]), g_ref,
                                     sl(dev["beta"]), None, n_threads=1)
    assert_close(sl(o_full), o_ref, torch.bfloat16, f"o head {h}, all tokens")
    assert_close(h_full[:, h:h + 1], h_ref, torch.bfloat16, f"hT head {h}")


# ---------------------------------------------------------------- chain segments
@pytest.mark.parametrize("seg", [1, 3, 5])
@pytest.mark.parametrize("precise", [0, PRECISE], ids=["default", "precise"])
def test_segmented_chain_single_sequence(kda, seg, precise):
    """A 1489-token sequence (24 chunks, ragged tail) whose chain is cut into
    segments of `seg` chunks, joined by the end-state scan, against the oracle."""
    inp, g, dev = _inputs([64 * 23 + 17], H=2, dtype=torch.bfloat16, seed=300 + seg)
    o, hT = _run(kda, dev, flags=kda.segment_chunks(seg) | precise)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, f"o seg={seg}")
    assert_close(hT, h_ref, torch.bfloat16, f"hT seg={seg}")


def test_segmented_chain_varlen(kda):
    """Segments of 3 chunks over packed sequences: empty, one chunk, ragged, long."""
    lens = [300, 0, 1000, 64, 2000, 1]
    inp, g, dev = _inputs(lens, H=3, dtype=torch.bfloat16, seed=41)
    o, hT = _run(kda, dev, flags=kda.segment_chunks(3))
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o segmented varlen")
    assert_close(hT, h_ref, torch.bfloat16, "hT segmented varlen")


def test_segmented_chain_slow_decay(kda):
    """Slow decays carry state across many segments: the scan's transitions matter."""
    inp, g, dev = _inputs([64 * 40], H=2, dtype=torch.bfloat16, seed=43, g_lo=-0.02, g_hi=0.0)
    o, hT = _run(kda, dev, flags=kda.segment_chunks(4))
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o segmented slow decay")
    assert_close(hT, h_ref, torch.bfloat16, "hT segmented slow decay")


def test_sequential_flag_and_auto_segments_agree_with_oracle(kda):
    """B=1, T=32768, H=4 bf16: the automatic choice splits the chain (few chains,
    long sequence); the sequential flag does not.  Both against the oracle on two
    heads."""
    w = workloads.custom([32768], H=4, dtype=torch.bfloat16, seed=51, h0_std=0.02)
    dev = workloads.make_inputs(w, "cuda")
    o_auto, h_auto = kda.chunk_fwd_gated(dev["q"], dev["k"], dev["v"], dev["z"], dev["A"],
                                         dev["beta"], dev["h0"], dev["cu_seqlens"])
    g = kda.gate(dev["z"], dev["A"])
    o_seq, h_seq = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g, dev["beta"], dev["h0"],
                                 dev["cu_seqlens"], flags=kda.SEQUENTIAL)
    torch.cuda.synchronize()
    for h in (0, 3):
        sl = lambda t: t[:, h:h + 1]
        g_ref = oracle.gate(sl(dev["z"]), dev["A"][h:h + 1])
        o_ref, h_ref = oracle.recurrence(sl(dev["q"]), sl(dev["k"]), sl(dev["v"]), g_ref,
                                         sl(dev["beta"]), dev["h0"][:, h:h + 1])
        for name, o_, h_ in (("auto", o_auto, h_auto), ("sequential", o_seq, h_seq)):
            assert_close(sl(o_), o_ref, torch.bfloat16, f"o {name} head {h}")
            assert_close(h_[:, h:h + 1], h_ref, torch.bfloat16, f"hT {name} head {h}")


# ---------------------------------------------------------------- state checkpoints
def _oracle_checkpoints(inp, g, lens, every):
    """The oracle state after every `every` tokens of each sequence: the recurrence
    run block by block, each block starting from the oracle's state at the end of
    the previous one (the state is all the recurrence carries between tokens)."""
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    out = []
    for n, L in enumerate(lens):
        S = to64(inp["h0"][n:n + 1]) if inp["h0"] is not None else None
        for i in range(L // every):
            a, b = cu[n] + i * every, cu[n] + (i + 1) * every
            sl = lambda t: t[a:b]
            _, S = oracle.recurrence(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(g),
                                     sl(inp["beta"]), S)
            out.append(S[0])
    H = inp["q"].shape[1]
    return np.stack(out) if out else np.zeros((0, H, 128, 128))


@pytest.mark.parametrize("every", [512, 128, 64])
@pytest.mark.parametrize("flags", [0, 3 << 16], ids=["serial", "seg3"])
def test_checkpoints_varlen(kda, every, flags):
    """Packed sequences (empty, shorter than one interval, exact multiples, ragged)
    with checkpoints every 512, 128 and 64 tokens, on the serial chain and on
    segments of 3 chunks (checkpoints at segment ends and inside segments)."""
    lens = [1024, 700, 512, 0, 1500, 64, 33]
    inp, g, dev = _inputs(lens, H=2, dtype=torch.bfloat16, seed=61 + every)
    o, hT, ck = kda.chunk_fwd_checkpointed(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                           dev["h0"], dev["cu_seqlens"], ckpt_tokens=every,
                                           flags=flags)
    kda.get_device_error()
    assert ck.shape[0] == sum(L // every for L in lens)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o with checkpoints")
    assert_close(hT, h_ref, torch.bfloat16, "hT with checkpoints")
    ck_ref = _oracle_checkpoints(inp, g, lens, every)
    for i in range(ck.shape[0]):
        assert_close(ck[i], ck_ref[i], torch.bfloat16, f"checkpoint {i} every={every}")


def test_checkpoint_at_sequence_end_equals_final_state(kda):
    """A sequence that ends on a checkpoint boundary: its last checkpoint is hT, bit
    for bit (both are written from the same accumulator)."""
    lens = [256, 640]
    inp, g, dev = _inputs(lens, H=3, dtype=torch.bfloat16, seed=71)
    _, hT, ck = kda.chunk_fwd_checkpointed(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                           dev["h0"], dev["cu_seqlens"], ckpt_tokens=128)
    assert ck.shape[0] == 2 + 5
    assert torch.equal(ck[1], hT[0]) and torch.equal(ck[6], hT[1])


def test_checkpoints_batched_and_slow_decay_segments(kda):
    """B=2 batched sequences of 3000 tokens with slow decays, segments of 4 chunks,
    checkpoints every 512 tokens (5 per sequence)."""
    B, T, H = 2, 3000, 2
    inp, g, dev = _inputs([T] * B, H=H, dtype=torch.bfloat16, seed=73, g_lo=-0.05, g_hi=0.0)
    shp = lambda t: t.view(B, T, *t.shape[1:])
    o, hT, ck = kda.chunk_fwd_checkpointed(shp(dev["q"]), shp(dev["k"]), shp(dev["v"]),
                                           shp(dev["g"]), shp(dev["beta"]), dev["h0"], None,
                                           ckpt_tokens=512, flags=kda.segment_chunks(4))
    assert ck.shape[0] == 10
    ck_ref = _oracle_checkpoints(inp, g, [T] * B, 512)
    for i in range(10):
        assert_close(ck[i], ck_ref[i], torch.bfloat16, f"checkpoint {i}")


def test_checkpoint_capacity_overflow_is_reported(kda):
    """Fewer slots than checkpoints: the first `capacity` are written, nothing past
    them, and the device error reads back as an invalid argument."""
    lens = [700, 1100]
    inp, g, dev = _inputs(lens, H=2, dtype=torch.bfloat16, seed=75)
    buf = torch.full((6, 2, 128, 128), 7.0, device="cuda")
    _, _, ck = kda.chunk_fwd_checkpointed(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                          dev["h0"], dev["cu_seqlens"], ckpt_tokens=256,
                                          ckpt_capacity=3, ckpt_out=buf)
    with pytest.raises(kda.KdaError):
        kda.get_device_error()
    kda.get_device_error()  # the flag was cleared by the read
    ck_ref = _oracle_checkpoints(inp, g, lens, 256)  # 2 + 4 checkpoints
    for i in range(3):
        assert_close(buf[i], ck_ref[i], torch.bfloat16, f"checkpoint {i}")
    assert bool((buf[3:] == 7.0).all())


# ------------------------------------------------ unbounded gate (range-robust mode)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_unbounded_softplus_gate(kda, dtype):
    """g = -exp(A) Softplus(z) with A in [0, 2] and z ~ N(0, 4): per-token log-decays
    down to about -50, 16-token sums far below the bounded path's -80.  The
    range-robust mode against the oracle (fp32 or bf16 tolerance by input type)."""
    lens = [5, 0, 70, 64, 129, 300]
    w = workloads.custom(lens, H=3, dtype=dtype, seed=91, z_std=2.0, A_range=0.0, h0_std=0.5)
    inp = workloads.make_inputs(w, "cpu")
    A = torch.linspace(0.0, 2.0, 3)
    g = torch.from_numpy(oracle.gate_softplus(inp["z"], A)).float()
    assert float(g.min()) < -30.0
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g_dev = kda.gate_softplus(dev["z"], A.cuda())
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g_dev, dev["beta"], dev["h0"],
                          dev["cu_seqlens"], flags=kda.UNBOUNDED_GATE)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, "o unbounded")
    assert_close(hT, h_ref, dtype, "hT unbounded")


def test_unbounded_mode_extremes(kda):
    """fp32: g = -10^4 on some tokens (the state is wiped there), g = 0 on others, and
    bounded g elsewhere, through the range-robust mode."""
    lens = [200, 77]
    inp, g, dev = _inputs(lens, H=2, dtype=torch.float32, seed=93)
    gen = torch.Generator().manual_seed(94)
    sel = torch.rand(sum(lens), 2, 1, generator=gen)
    g = torch.where(sel < 0.1, torch.full_like(g, -1e4), torch.where(sel > 0.9, torch.zeros_like(g), g))
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g.cuda(), dev["beta"], dev["h0"],
                          dev["cu_seqlens"], flags=kda.UNBOUNDED_GATE)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.float32, "o extremes")
    assert_close(hT, h_ref, torch.float32, "hT extremes")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_unbounded_mode_on_bounded_gate(kda, dtype):
    """The range-robust mode on ordinary bounded decays gives the same answer."""
    inp, g, dev = _inputs([5, 0, 70, 129, 300], H=2, dtype=dtype, seed=95)
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"],
                          dev["cu_seqlens"], flags=kda.UNBOUNDED_GATE)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, "o robust on bounded")
    assert_close(hT, h_ref, dtype, "hT robust on bounded")


def test_scalar_gate_gated_deltanet(kda):
    """Gated DeltaNet (one decay per token and head, "Kimi K3 notes", section
    "Kimi Delta Attention": alpha_t (I - b k k^T) S + b k v^T) is KDA with g constant
    over the channels; bf16 tensor-core path against the oracle."""
    lens = [300, 64, 5]
    inp, g, dev = _inputs(lens, H=2, dtype=torch.bfloat16, seed=97)
    gs = g[..., :1].expand_as(g).contiguous()
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], gs.cuda(), dev["beta"], dev["h0"],
                          dev["cu_seqlens"])
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], gs, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o GDN")
    assert_close(hT, h_ref, torch.bfloat16, "hT GDN")


@pytest.mark.parametrize("dtype,flags", PATHS, ids=PATH_IDS)
def test_scalar_gate_layout(kda, dtype, flags):
    """SCALAR_GATE: g given as [NT, H] (one log-decay per token and head, 4 bytes
    instead of 512 per token-head) on every path, against the oracle run with that
    decay on every channel; on the tensor-core path the result equals the run with
    the broadcast [NT, H, 128] g bit for bit."""
    lens = [300, 0, 64, 5, 129]
    inp, g, dev = _inputs(lens, H=3, dtype=dtype, seed=98)
    g1 = g[..., 0].contiguous()                       # [NT, H]
    gb = g1[..., None].expand_as(g).contiguous()      # the same decay on every channel
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g1.cuda(), dev["beta"], dev["h0"],
                          dev["cu_seqlens"], flags=flags | kda.SCALAR_GATE)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], gb, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, dtype, "o scalar gate")
    assert_close(hT, h_ref, dtype, "hT scalar gate")
    ob, hb = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], gb.cuda(), dev["beta"], dev["h0"],
                           dev["cu_seqlens"], flags=flags)
    assert torch.equal(o, ob) and torch.equal(hT, hb)


def test_scalar_gate_unbounded_and_checkpoints(kda):
    """Scalar gates with the unbounded mode (decays down to -40 per token) and with
    state checkpoints on the tensor-core path."""
    inp, g, dev = _inputs([256, 70], H=2, dtype=torch.bfloat16, seed=99, g_lo=-40.0)
    g1 = g[..., 0].contiguous()
    gb = g1[..., None].expand_as(g).contiguous()
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g1.cuda(), dev["beta"], dev["h0"],
                          dev["cu_seqlens"], flags=kda.SCALAR_GATE | kda.UNBOUNDED_GATE)
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], gb, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o scalar unbounded")
    assert_close(hT, h_ref, torch.bfloat16, "hT scalar unbounded")
    gc = (g1 / 8).cuda()  # inside [-5, 0] for the tensor-core path
    o1, h1, c1 = kda.chunk_fwd_checkpointed(dev["q"], dev["k"], dev["v"], gc, dev["beta"],
                                            dev["h0"], dev["cu_seqlens"], ckpt_tokens=128,
                                            flags=kda.SCALAR_GATE)
    gcb = gc[..., None].expand(-1, -1, 128).contiguous()
    o2, h2, c2 = kda.chunk_fwd_checkpointed(dev["q"], dev["k"], dev["v"], gcb, dev["beta"],
                                            dev["h0"], dev["cu_seqlens"], ckpt_tokens=128)
    assert torch.equal(o1, o2) and torch.equal(h1, h2) and torch.equal(c1, c2)


def test_each_path_launches_only_its_own_kernels(kda):
    """The bf16 entry runs the plan and the tensor-core kernels only; the fp32-core
    flag runs the CUDA-core kernels only (a second path on the same workspace would
    write past it); the fused entry with an output gate runs the same kernels (the
    chain applies the gate before it writes o)."""
    inp, g, dev = _inputs([300, 77], H=2, dtype=torch.bfloat16, seed=99)
    args = (dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"], dev["cu_seqlens"])

    def launched(fn):
        torch.cuda.synchronize()
        kda.profile_enable(True)
        fn()
        torch.cuda.synchronize()
        names = set(kda.profile_collect())
        kda.profile_enable(False)
        return names

    tc = launched(lambda: kda.chunk_fwd(*args, flags=kda.SEQUENTIAL))
    assert tc == {"kda_plan", "kda_tc_prep", "kda_tc_chain"}, tc
    simt = launched(lambda: kda.chunk_fwd(*args, flags=kda.FP32_CORES))
    assert simt == {"kda_plan", "kda_simt_prep", "kda_simt_chain"}, simt
    gz = torch.randn_like(dev["v"].float()).to(torch.bfloat16)
    fused = launched(lambda: kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"],
                                                 dev["h0"], dev["cu_seqlens"], g=dev["g"],
                                                 out_gate=gz, flags=kda.SEQUENTIAL))
    # the output gate is applied by the chain's store warps: no kernel of its own
    assert fused == {"kda_plan", "kda_tc_prep", "kda_tc_chain"}, fused


def test_checkpoints_full_size_sampled(kda):
    """B=1, T=8192, H=96, bf16, a checkpoint every 512 tokens (16), as the bench runs
    it: all 16 checkpoints of 2 sampled heads against the oracle run block by block."""
    w = workloads.prefill()
    dev = workloads.make_inputs(w, "cuda")
    g = kda.gate(dev["z"], dev["A"])
    _, hT, ck = kda.chunk_fwd_checkpointed(dev["q"], dev["k"], dev["v"], g, dev["beta"],
                                           dev["h0"], dev["cu_seqlens"], ckpt_tokens=512)
    torch.cuda.synchronize()
    assert ck.shape[0] == 16
    for h in (3, 90):
        sl = lambda t: t[:, h:h + 1]
        inp = dict(q=sl(dev["q"]), k=sl(dev["k"]), v=sl(dev["v"]), beta=sl(dev["beta"]),
                   h0=dev["h0"][:, h:h + 1])
        g_ref = oracle.gate(sl(dev["z"]), dev["A"][h:h + 1])
        ck_ref = _oracle_checkpoints(inp, g_ref, [w.n_tokens], 512)
        for i in range(16):
            assert_close(ck[i, h:h + 1], ck_ref[i], torch.bfloat16, f"checkpoint {i} head {h}")
        assert torch.equal(ck[15], hT[0])
