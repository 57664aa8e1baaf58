"""The oracle against the facts that pin it (CPU only).

See ``oracle_pins.py`` for each pin and the passage or theorem behind it.
"""

import math
import os

import numpy as np
import pytest

import oracle
from tests import oracle_pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split("=", 1)
                vals[key.strip()] = float(val)
    return vals


def test_golden_range_margin():
    """Numbers printed for the bounded-decay range argument."""
    gv = _read_golden("range_margin.txt")
    assert gv["g_min"] * gv["tile_tokens"] == gv["tile_log_decay_floor"]
    assert math.exp(-gv["tile_log_decay_floor"]) == pytest.approx(gv["inv_gamma_bound"], rel=0.01)
    import torch

    assert float(torch.finfo(torch.bfloat16).max) == pytest.approx(gv["bf16_max"], rel=0.01)
    assert float(torch.finfo(torch.float32).max) == pytest.approx(gv["bf16_max"], rel=0.01)
    assert gv["inv_gamma_bound"] < gv["bf16_max"]


def test_golden_state_sizes():
    """State sizes printed for one K3 request; the benchmark's decode byte count
    (fp32 state read + write) is built from the same element count."""
    gv = _read_golden("state_sizes.txt")
    elems = gv["heads"] * gv["dk"] * gv["dv"]
    assert elems == gv["state_elems_per_layer"]
    assert elems * 2 / 2**20 == gv["bf16_mib_per_layer"]
    per_req = elems * 2 * gv["kda_layers"] / 2**20
    assert per_req == pytest.approx(gv["bf16_mib_per_request"], abs=0.5)
    assert 2 * per_req == pytest.approx(gv["decode_rw_mib_per_request_step"], abs=1.0)
    from bench import decode_bytes_per_head_step

    # fp32 state read and written, q, k, v and o in bf16, g in fp32, beta in bf16
    assert decode_bytes_per_head_step(128, 128) == 2 * 128 * 128 * 4 + 128 * 2 * 4 + 128 * 4 + 2


def test_oracle_rejects_bad_cu_seqlens(oracle_lib):
    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.recurrence(q, q, q, q, np.zeros((4, 1)), None, cu_seqlens=[0, 3, 2, 4],
                          lib=oracle_lib)


def test_oracle_threads_agree(oracle_lib):
    q, k, v, g, beta, S0 = oracle_pins.random_case(30, T=33, H=5, N=1)
    a = oracle.recurrence(q, k, v, g, beta, S0, n_threads=1, lib=oracle_lib)
    b = oracle.recurrence(q, k, v, g, beta, S0, n_threads=4, lib=oracle_lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
