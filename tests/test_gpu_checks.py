"""Failure detection and input checks on the GPU, with no GPU fault.

* The bounded waits: kda_selftest_wait_timeout runs the same wait and drain code
  as the tensor-core kernels on a barrier that nothing signals, with a 1 ms
  limit.  Every waiting warp must return, the device flag must read back as
  KDA_ERR_DEVICE_TIMEOUT, and a prefill right after must still match the oracle
  (the context is usable).
* The input-precondition pass (KDA_CHUNK_CHECK_INPUTS, or KDA_CHECKS=1): the
  tensor-core path relies on g in [-5, 0] (the 16-token tile bound, "Kimi K3
  technical report review", section 3.2) and beta in [0, 1].  Out-of-range
  values made on the host (values, not faults) must raise the device flag;
  in-range inputs must not.
"""

import os
import subprocess
import sys

import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    import chunked_gated_delta_fwd_gb300 as m

    m.get_device_error()  # start from a clear flag
    return m


def _small(seed=5):
    w = workloads.custom([100, 0, 150], H=2, dtype=torch.bfloat16, seed=seed, h0_std=0.1)
    inp = workloads.make_inputs(w, "cpu")
    g = workloads.uniform_decay((w.n_tokens, 2, 128), "cpu", seed=seed + 1)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dev["g"] = g.cuda()
    return inp, g, dev


def test_bounded_wait_gives_up_and_the_context_stays_usable(kda):
    for _ in range(2):
        n = kda.selftest_wait_timeout(1000)
        assert n == 4, f"{n} of 4 waiting warps returned unsatisfied"
        with pytest.raises(kda.KdaError) as ei:
            kda.get_device_error()
        assert ei.value.status == 7  # KDA_ERR_DEVICE_TIMEOUT
        kda.get_device_error()  # the read cleared it
    inp, g, dev = _small()
    o, hT = kda.chunk_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["h0"],
                          dev["cu_seqlens"])
    kda.get_device_error()  # nothing raised by a normal prefill
    o_ref, h_ref = oracle.recurrence(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                     inp["cu_seqlens"])
    assert_close(o, o_ref, torch.bfloat16, "o after the timeout self-test")
    assert_close(hT, h_ref, torch.bfloat16, "hT after the timeout self-test")


def test_selftest_rejects_bad_limits(kda):
    for bad in (0, 2_000_000):
        with pytest.raises(kda.KdaError) as ei:
            kda.selftest_wait_timeout(bad)
        assert ei.value.status == 1


def _check_run(kda, dev, g, beta, flags):
    kda.chunk_fwd(dev["q"], dev["k"], dev["v"], g, beta, dev["h0"], dev["cu_seqlens"],
                  flags=flags | kda.CHECK_INPUTS)
    try:
        kda.get_device_error()
        return None
    except kda.KdaError as e:
        return e


@pytest.mark.parametrize("flags", [0, 1], ids=["bf16-tc", "bf16-f32cores"])
def test_input_check_accepts_in_range_and_flags_out_of_range(kda, flags):
    inp, g, dev = _small(7)
    assert _check_run(kda, dev, dev["g"], dev["beta"], flags) is None
    edge = dev["g"].clone()
    edge[3, 1, 7], edge[4, 0, 0] = -5.0, 0.0  # the closed interval's ends pass
    assert _check_run(kda, dev, edge, dev["beta"], flags) is None
    cases = {}
    g_low = dev["g"].clone()
    g_low[17, 1, 100] = -5.001
    cases["g below -5"] = (g_low, dev["beta"])
    g_pos = dev["g"].clone()
    g_pos[-1, 0, 127] = 1e-3  # the last element (the vector pass's tail)
    cases["g above 0"] = (g_pos, dev["beta"])
    g_nan = dev["g"].clone()
    g_nan[0, 0, 0] = float("nan")
    cases["g NaN"] = (g_nan, dev["beta"])
    b_hi = dev["beta"].clone()
    b_hi[42, 1] = 1.5
    cases["beta above 1"] = (dev["g"], b_hi)
    b_lo = dev["beta"].clone()
    b_lo[0, 0] = -0.25
    cases["beta below 0"] = (dev["g"], b_lo)
    for name, (gg, bb) in cases.items():
        e = _check_run(kda, dev, gg, bb, flags)
        assert e is not None and e.status == 1 and "input check" in str(e), name


def test_input_check_modes(kda):
    """The unbounded mode accepts any finite g <= 0; the scalar-gate layout is
    checked as [NT, H]; a gate formed from z leaves only beta to check."""
    inp, g, dev = _small(9)
    deep = dev["g"] * 20.0  # down to -100: fine for the unbounded mode only
    assert _check_run(kda, dev, deep, dev["beta"], kda.UNBOUNDED_GATE) is None
    e = _check_run(kda, dev, deep, dev["beta"], 0)
    assert e is not None and e.status == 1
    inf = dev["g"].clone()
    inf[5, 1, 5] = float("-inf")
    assert _check_run(kda, dev, inf, dev["beta"], kda.UNBOUNDED_GATE) is not None
    gs = dev["g"][..., 0].contiguous()
    assert _check_run(kda, dev, gs, dev["beta"], kda.SCALAR_GATE) is None
    gs[-1, -1] = -6.0
    assert _check_run(kda, dev, gs, dev["beta"], kda.SCALAR_GATE) is not None
    b_bad = dev["beta"].clone()
    b_bad[7, 0] = 2.0
    kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], b_bad, dev["h0"], dev["cu_seqlens"],
                        z=dev["z"], A=dev["A"], flags=kda.CHECK_INPUTS)
    with pytest.raises(kda.KdaError):
        kda.get_device_error()
    kda.chunk_fwd_fused(dev["q"], dev["k"], dev["v"], dev["beta"], dev["h0"], dev["cu_seqlens"],
                        z=dev["z"], A=dev["A"], flags=kda.CHECK_INPUTS)
    kda.get_device_error()


def test_input_check_from_the_environment(kda):
    """KDA_CHECKS=1 turns the pass on for every chunk call (a fresh process: the
    variable is read once)."""
    code = (
        "import torch, workloads, chunked_gated_delta_fwd_gb300 as kda\n"
        "w = workloads.custom([80], H=2, dtype=torch.bfloat16, seed=3)\n"
        "d = workloads.make_inputs(w, 'cuda')\n"
        "g = workloads.uniform_decay((80, 2, 128), 'cuda', seed=4)\n"
        "g[10, 1, 3] = -7.0\n"
        "kda.chunk_fwd(d['q'], d['k'], d['v'], g, d['beta'], None, d['cu_seqlens'])\n"
        "try:\n"
        "    kda.get_device_error()\n"
        "    print('NOT FLAGGED')\n"
        "except kda.KdaError as e:\n"
        "    print('FLAGGED', e.status)\n")
    env = dict(os.environ, KDA_CHECKS="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "FLAGGED 1" in r.stdout, r.stdout + r.stderr[-2000:]
