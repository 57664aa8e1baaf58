"""Shared helpers of the GPU parity tests: tolerances and error metrics.

Tolerances (stated for the KDA forward with these input types):
* bf16 q/k/v/beta with fp32 state: relative L2 error <= 1e-2 and max abs
  error <= 3e-2, on o and on the final states;
* fp32 inputs: relative L2 error <= 1e-5.
rel_L2 = |x - ref|_2 / |ref|_2 over the whole tensor, max_abs = max |x - ref|.
"""

import numpy as np
import torch

BF16_REL_L2 = 1e-2
BF16_MAX_ABS = 3e-2
F32_REL_L2 = 1e-5


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def errors(got, ref):
    got, ref = to64(got), to64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    diff = got - ref
    nref = np.linalg.norm(ref.ravel())
    rel = np.linalg.norm(diff.ravel()) / (nref if nref > 0 else 1.0)
    mabs = float(np.max(np.abs(diff))) if diff.size else 0.0
    return float(rel), mabs


def assert_close(got, ref, dtype, what=""):
    rel, mabs = errors(got, ref)
    if dtype == torch.float32:
        assert rel <= F32_REL_L2, f"{what}: rel_L2 {rel:.3e} > {F32_REL_L2}"
    else:
        assert rel <= BF16_REL_L2, f"{what}: rel_L2 {rel:.3e} > {BF16_REL_L2}"
        assert mabs <= BF16_MAX_ABS, f"{what}: max_abs {mabs:.3e} > {BF16_MAX_ABS}"
    return rel, mabs


def cuda_ok():
    if not torch.cuda.is_available():
        return False
    return torch.cuda.get_device_capability(0) == (10, 3)


def assert_close_gated(got, ref, o_ref, x, w, eps, what=""):
    """Parity of the gated output y = Sigmoid(x) w o / rms(o) against the oracle's y.

    The gate is a per-token, per-channel factor f = Sigmoid(x) w / rms(o) applied
    to the KDA output, so an error e in o becomes f e in y.  The bf16 bounds above
    are stated for o; here rel_L2 <= 1e-2 is checked on y itself and the max-abs
    bound on the error carried back to the units of o, (y - y_ref) / f.
    """
    got64, ref64 = to64(got), to64(ref)
    o64, x64 = to64(o_ref), to64(x)
    f = 1.0 / (1.0 + np.exp(-x64)) / np.sqrt(np.mean(o64 * o64, axis=-1, keepdims=True) + eps)
    if w is not None:
        f = f * to64(w)
    rel, _ = errors(got64, ref64)
    assert rel <= BF16_REL_L2, f"{what}: rel_L2 {rel:.3e} > {BF16_REL_L2}"
    mabs = float(np.max(np.abs((got64 - ref64) / f))) if f.size else 0.0
    assert mabs <= BF16_MAX_ABS, f"{what}: max_abs in o units {mabs:.3e} > {BF16_MAX_ABS}"
