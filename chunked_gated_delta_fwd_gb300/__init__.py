"""GB300 Kimi Delta Attention (KDA) forward -- Python binding of libkda.

A thin ctypes layer over the C ABI in ``include/kda.h``: it checks tensor
dtypes, devices and contiguity, passes ``data_ptr()`` values and the current
CUDA stream, and raises :class:`KdaError` on a non-OK status.  Every step of
the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and importing this package fails if ``libkda.so`` has not
been built (``python chunked_gated_delta_fwd_gb300/_build.py``).

Entry points (same names as the C calls, without the ``kda_`` prefix):

* :func:`gate` -- ``g = g_min * Sigmoid(exp(A_h) z)`` (optionally the in-chunk
  running sum),
* :func:`chunk_fwd` -- prefill over whole (packed, variable-length) sequences,
* :func:`recurrent_step` -- one decode token per sequence, state in place.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = ["KdaError", "gate", "chunk_fwd", "chunk_fwd_gated", "chunk_fwd_workspace_size", "recurrent_step",
           "library_path", "lib", "get_device_error", "profile_enable", "profile_collect", "G_MIN", "F32", "BF16", "FP32_CORES", "SEQUENTIAL",
           "segment_chunks", "recurrent_multi_step", "chunk_fwd_checkpointed",
           "chunk_fwd_fused", "gate_softplus", "UNBOUNDED_GATE",
           "output_gate", "SCALAR_GATE", "CHECK_INPUTS", "PRECISE", "selftest_wait_timeout"]

G_MIN = -5.0
F32, BF16 = 0, 1
FP32_CORES = 1  # flag of chunk_fwd: evaluate bf16 inputs on fp32 CUDA cores
SEQUENTIAL = 2  # flag of chunk_fwd: never split a sequence's chain into segments
UNBOUNDED_GATE = 4  # flag of chunk_fwd: any g <= 0 (range-robust fp32-core evaluation)
SCALAR_GATE = 8  # flag of chunk_fwd: g is [..., H], one log-decay per token and head
CHECK_INPUTS = 16  # flag of chunk_fwd: check g and beta against their ranges on the device
PRECISE = 32  # flag of chunk_fwd (bf16 tensor cores): the state update at tf32 precision

_STATUS = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED_SHAPE",
    3: "KDA_ERR_UNSUPPORTED_DTYPE", 4: "KDA_ERR_MISALIGNED", 5: "KDA_ERR_WORKSPACE_TOO_SMALL",
    6: "KDA_ERR_CUDA", 7: "KDA_ERR_DEVICE_TIMEOUT", 8: "KDA_ERR_NO_DEVICE",
}


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return os.environ.get("KDA_LIBRARY", _build.LIB)


def _load() -> ctypes.CDLL:
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"libkda.so not found at {path}; build it with "
                          f"`python chunked_gated_delta_fwd_gb300/_build.py`")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, sz, u32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                  ctypes.c_size_t, ctypes.c_uint)
    L.kda_gate.argtypes = [vp, i32, vp, f32, vp, i64, i32, i32, vp, vp, i32, vp]
    L.kda_gate_softplus.argtypes = [vp, i32, vp, vp, i64, i32, i32, vp]
    L.kda_output_gate.argtypes = [vp, i32, vp, vp, f32, vp, i64, i32, i32, vp]
    L.kda_chunk_fwd_workspace_size.argtypes = [i64, i32, i32, i32]
    L.kda_chunk_fwd_workspace_size.restype = sz
    L.kda_chunk_fwd_workspace_size_ex.argtypes = [i64, i32, i32, i32, u32]
    L.kda_chunk_fwd_workspace_size_ex.restype = sz
    L.kda_chunk_fwd.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32, vp,
                                vp, vp, sz, vp]
    L.kda_chunk_fwd_ex.argtypes = L.kda_chunk_fwd.argtypes + [u32]
    L.kda_chunk_fwd_checkpointed.argtypes = (L.kda_chunk_fwd.argtypes[:16] + [vp, i32, i64]
                                             + L.kda_chunk_fwd.argtypes[16:] + [u32])
    L.kda_chunk_fwd_fused.argtypes = [vp, vp, vp, i32, vp, vp, vp, f32, vp, vp, vp, i32, i32, i64,
                                      i32, i32, i32, f32, vp, vp, f32, vp, vp, vp, sz, vp, u32]
    L.kda_chunk_fwd_gated.argtypes = [vp, vp, vp, i32, vp, vp, f32, vp, vp, vp, i32, i32, i64,
                                      i32, i32, i32, vp, vp, vp, sz, vp]
    L.kda_recurrent_step.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, vp]
    L.kda_recurrent_multi_step.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32,
                                           i32, i32, vp]
    L.kda_selftest_wait_timeout.argtypes = [u32, ctypes.POINTER(i32), vp]
    L.kda_selftest_wait_timeout.restype = ctypes.c_int
    L.kda_last_error_string.restype = ctypes.c_char_p
    L.kda_get_device_error.argtypes = [vp]
    L.kda_version.restype = ctypes.c_char_p
    L.kda_profile_enable.argtypes = [i32]
    L.kda_profile_get.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i32),
                                  ctypes.POINTER(ctypes.c_double)]
    for fn in (L.kda_gate, L.kda_chunk_fwd, L.kda_chunk_fwd_ex, L.kda_chunk_fwd_gated,
               L.kda_recurrent_step, L.kda_recurrent_multi_step, L.kda_get_device_error):
        fn.restype = ctypes.c_int
    return L


lib = _load()


def _check(status: int):
    if status != 0:
        raise KdaError(status, lib.kda_last_error_string().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _need(t: torch.Tensor, name: str, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def gate(z: torch.Tensor, A: torch.Tensor, g_min: float = G_MIN, *, out=None,
         with_cumsum: bool = False, cu_seqlens: Optional[torch.Tensor] = None):
    """g = g_min * Sigmoid(exp(A[h]) * z) for z of shape [..., H, 128] (bf16/fp32).

    Returns g (fp32, z's shape), or (g, gcum) with ``with_cumsum`` where gcum is the
    running sum of g inside each 64-token chunk of each sequence.
    """
    _need(z, "z")
    _need(A, "A", torch.float32, z.device)
    H, dk = z.shape[-2], z.shape[-1]
    NT = z.numel() // (H * dk) if z.numel() else 0
    g = out if out is not None else torch.empty(z.shape, dtype=torch.float32, device=z.device)
    _need(g, "out", torch.float32, z.device)
    gcum = torch.empty_like(g) if with_cumsum else None
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, z.device)
    n_seqs = cu_seqlens.numel() - 1 if cu_seqlens is not None else 1
    with torch.cuda.device(z.device):
        _check(lib.kda_gate(_ptr(z), _dtype_code(z), _ptr(A), float(g_min), _ptr(g), NT, H, dk,
                            _ptr(gcum), _ptr(cu_seqlens), n_seqs, _stream(z.device)))
    return (g, gcum) if with_cumsum else g


def output_gate(o: torch.Tensor, gate: torch.Tensor, weight=None, eps: float = 1e-6, *,
                out=None):
    """y = Sigmoid(gate) * weight * o / sqrt(mean(o^2) + eps) over the 128 channels of
    each (token, head); o, gate [..., H, 128] (bf16/fp32, same dtype), weight fp32
    [128] or None.  ``out=o`` works in place."""
    _need(o, "o")
    _need(gate, "gate", o.dtype, o.device)
    if tuple(gate.shape) != tuple(o.shape):
        raise ValueError("gate must have the shape of o")
    if weight is not None:
        _need(weight, "weight", torch.float32, o.device)
    H, dv = o.shape[-2], o.shape[-1]
    NT = o.numel() // (H * dv) if o.numel() else 0
    y = out if out is not None else torch.empty_like(o)
    _need(y, "out", o.dtype, o.device)
    with torch.cuda.device(o.device):
        _check(lib.kda_output_gate(_ptr(o), _dtype_code(o), _ptr(gate), _ptr(weight), float(eps),
                                   _ptr(y), NT, H, dv, _stream(o.device)))
    return y


def gate_softplus(z: torch.Tensor, A: torch.Tensor, *, out=None):
    """The unbounded gate g = -exp(A[h]) * Softplus(z), z [..., H, 128] (bf16/fp32);
    a prefill on it needs the ``UNBOUNDED_GATE`` flag.  Returns g (fp32)."""
    _need(z, "z")
    _need(A, "A", torch.float32, z.device)
    H, dk = z.shape[-2], z.shape[-1]
    NT = z.numel() // (H * dk) if z.numel() else 0
    g = out if out is not None else torch.empty(z.shape, dtype=torch.float32, device=z.device)
    _need(g, "out", torch.float32, z.device)
    with torch.cuda.device(z.device):
        _check(lib.kda_gate_softplus(_ptr(z), _dtype_code(z), _ptr(A), _ptr(g), NT, H, dk,
                                     _stream(z.device)))
    return g


def chunk_fwd_workspace_size(n_tokens: int, n_seqs: int, H: int, dtype=torch.bfloat16,
                             flags: int = 0) -> int:
    code = BF16 if dtype == torch.bfloat16 else F32
    return int(lib.kda_chunk_fwd_workspace_size_ex(int(n_tokens), int(n_seqs), int(H), code,
                                                   int(flags)))


def segment_chunks(n: int) -> int:
    """Flag bits forcing chain segments of n chunks (KDA_CHUNK_SEGMENT_CHUNKS)."""
    return (int(n) & 0xFFFF) << 16


def chunk_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, *, output_final_state=True,
              workspace=None, flags: int = 0, out=None, final_state_out=None):
    """KDA prefill over whole sequences.

    q, k: [B, T, H, 128] or packed [T, H, 128] (with ``cu_seqlens``), bf16 or fp32;
    v like q; g: same shape, fp32 log-decays in [-5, 0] (with ``flags`` holding
    ``SCALAR_GATE``: [..., H], one per token and head); beta: [..., H] (dtype of q);
    h0: [N, H, 128, 128] fp32 (the state stored transposed, [dv][dk]) or None;
    cu_seqlens: int32 [N+1] on the device, or None for B sequences of length T.
    Returns ``(o, hT)`` with o like v and hT [N, H, 128, 128] fp32 (None if not asked).
    """
    _need(g, "g", torch.float32, q.device)
    c = _chunk_setup(q, k, v, beta, h0, cu_seqlens, output_final_state, workspace, flags, out,
                     final_state_out)
    with torch.cuda.device(q.device):
        _check(lib.kda_chunk_fwd_ex(_ptr(q), _ptr(k), _ptr(v), c["dt"], _ptr(g), _ptr(beta),
                                    _ptr(h0), _ptr(cu_seqlens), c["N"], c["B"], c["T"], c["H"],
                                    c["dk"], c["dv"], _ptr(c["o"]), _ptr(c["hT"]),
                                    _ptr(c["ws"]), c["ws"].numel(), _stream(q.device),
                                    int(flags)))
    return c["o"], c["hT"]


def chunk_fwd_checkpointed(q, k, v, g, beta, h0=None, cu_seqlens=None, *,
                           ckpt_tokens: int = 512, ckpt_capacity=None, ckpt_out=None,
                           output_final_state=True, workspace=None, flags: int = 0, out=None,
                           final_state_out=None):
    """``chunk_fwd`` that also returns the state after every ``ckpt_tokens`` tokens of
    each sequence (bf16, tensor-core path).  Sequence n contributes
    floor(len_n / ckpt_tokens) checkpoints, stacked in sequence order into
    ``ckpt`` [n_ckpt, H, 128, 128] fp32 (layout of hT).  ``ckpt_capacity`` (slots to
    allocate) defaults to the exact count, read from ``cu_seqlens`` on the host.
    Returns ``(o, hT, ckpt)``."""
    _need(g, "g", torch.float32, q.device)
    c = _chunk_setup(q, k, v, beta, h0, cu_seqlens, output_final_state, workspace, flags, out,
                     final_state_out)
    if ckpt_capacity is None:
        if ckpt_out is not None:
            ckpt_capacity = ckpt_out.shape[0]
        elif cu_seqlens is None:
            ckpt_capacity = c["B"] * (c["T"] // int(ckpt_tokens))
        else:
            lens = torch.diff(cu_seqlens.to("cpu", torch.int64))
            ckpt_capacity = int((lens.clamp(min=0) // int(ckpt_tokens)).sum())
    ck = ckpt_out if ckpt_out is not None else torch.empty(
        (int(ckpt_capacity), c["H"], c["dv"], c["dk"]), dtype=torch.float32, device=q.device)
    _need(ck, "ckpt_out", torch.float32, q.device)
    if ck.shape[0] < int(ckpt_capacity):
        raise ValueError(f"ckpt_out holds {ck.shape[0]} < {ckpt_capacity} checkpoints")
    with torch.cuda.device(q.device):
        _check(lib.kda_chunk_fwd_checkpointed(
            _ptr(q), _ptr(k), _ptr(v), c["dt"], _ptr(g), _ptr(beta), _ptr(h0),
            _ptr(cu_seqlens), c["N"], c["B"], c["T"], c["H"], c["dk"], c["dv"], _ptr(c["o"]),
            _ptr(c["hT"]), _ptr(ck) if int(ckpt_capacity) > 0 else None, int(ckpt_tokens),
            int(ckpt_capacity), _ptr(c["ws"]), c["ws"].numel(), _stream(q.device), int(flags)))
    return c["o"], c["hT"], ck


def chunk_fwd_fused(q, k, v, beta, h0=None, cu_seqlens=None, *, g=None, z=None, A=None,
                    g_min: float = -5.0, qk_l2_eps=None, out_gate=None, out_norm_weight=None,
                    out_norm_eps: float = 1e-6, output_final_state=True, workspace=None,
                    flags: int = 0, out=None, final_state_out=None):
    """bf16 prefill with the prologue and epilogue fused: exactly one of ``g`` (fp32
    log-decays) and ``z`` + ``A`` (gate computed in-kernel); ``qk_l2_eps`` (None: q, k
    used as given) L2-normalises q and k per token and head; ``out_gate`` [..., H,
    128] (dtype of q) applies o <- Sigmoid(out_gate) * w * o / rms(o) per head, with
    ``out_norm_weight`` fp32 [128] (None: ones).  Returns ``(o, hT)``."""
    if (g is None) == (z is None):
        raise ValueError("give exactly one of g and z")
    if g is not None:
        _need(g, "g", torch.float32, q.device)
    else:
        _need(z, "z", q.dtype, q.device)
        _need(A, "A", torch.float32, q.device)
    if out_gate is not None:
        _need(out_gate, "out_gate", q.dtype, q.device)
        if tuple(out_gate.shape) != tuple(v.shape):
            raise ValueError(f"out_gate must have the shape of v {tuple(v.shape)}")
    if out_norm_weight is not None:
        _need(out_norm_weight, "out_norm_weight", torch.float32, q.device)
    c = _chunk_setup(q, k, v, beta, h0, cu_seqlens, output_final_state, workspace, flags, out,
                     final_state_out)
    with torch.cuda.device(q.device):
        _check(lib.kda_chunk_fwd_fused(
            _ptr(q), _ptr(k), _ptr(v), c["dt"], _ptr(g), _ptr(z), _ptr(A), float(g_min),
            _ptr(beta), _ptr(h0), _ptr(cu_seqlens), c["N"], c["B"], c["T"], c["H"], c["dk"],
            c["dv"], -1.0 if qk_l2_eps is None else float(qk_l2_eps), _ptr(out_gate),
            _ptr(out_norm_weight), float(out_norm_eps), _ptr(c["o"]), _ptr(c["hT"]),
            _ptr(c["ws"]), c["ws"].numel(), _stream(q.device), int(flags)))
    return c["o"], c["hT"]


def chunk_fwd_gated(q, k, v, z, A, beta, h0=None, cu_seqlens=None, *, g_min: float = -5.0,
                    output_final_state=True, workspace=None, out=None, final_state_out=None):
    """KDA prefill with the bounded gate g = g_min * Sigmoid(exp(A_h) z) evaluated
    inside the chunk kernels (g is never materialised).  bf16 only; z like k,
    A fp32 [H].  Everything else as ``chunk_fwd``."""
    _need(z, "z", q.dtype, q.device)
    _need(A, "A", torch.float32, q.device)
    c = _chunk_setup(q, k, v, beta, h0, cu_seqlens, output_final_state, workspace, 0, out,
                     final_state_out)
    with torch.cuda.device(q.device):
        _check(lib.kda_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), c["dt"], _ptr(z), _ptr(A),
                                       float(g_min), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
                                       c["N"], c["B"], c["T"], c["H"], c["dk"], c["dv"],
                                       _ptr(c["o"]), _ptr(c["hT"]), _ptr(c["ws"]),
                                       c["ws"].numel(), _stream(q.device)))
    return c["o"], c["hT"]


def _chunk_setup(q, k, v, beta, h0, cu_seqlens, output_final_state, workspace, flags, out,
                 final_state_out):
    """Checks the chunk inputs and allocates the outputs and the workspace."""
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _need(t, name, q.dtype, dev)
    dt = _dtype_code(q)
    H, dk, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        N = cu_seqlens.numel() - 1
        B, T = 1, q.numel() // (H * dk)
        if q.dim() == 4 and q.shape[0] != 1:
            raise ValueError("with cu_seqlens, q must be packed as [1, NT, H, D] or [NT, H, D]")
    else:
        if q.dim() != 4:
            raise ValueError("q must be [B, T, H, D] without cu_seqlens")
        B, T = q.shape[0], q.shape[1]
        N = B
    NT = B * T if cu_seqlens is None else T
    if h0 is not None:
        _need(h0, "h0", torch.float32, dev)
        if tuple(h0.shape) != (N, H, dv, dk):
            raise ValueError(f"h0 must be [{N}, {H}, {dv}, {dk}], got {tuple(h0.shape)}")
    o = out if out is not None else torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(o, "out", v.dtype, dev)
    hT = None
    if output_final_state:
        hT = final_state_out if final_state_out is not None else torch.empty(
            (N, H, dv, dk), dtype=torch.float32, device=dev)
        _need(hT, "final_state_out", torch.float32, dev)
    need = chunk_fwd_workspace_size(NT, N, H, q.dtype, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    return dict(dt=dt, N=N, B=B, T=T, H=H, dk=dk, dv=dv, o=o, hT=hT, ws=workspace)


def recurrent_step(q, k, v, g, beta, S, *, out=None):
    """One decode token: q, k, v [N, H, 128] (bf16/fp32), g [N, H, 128] fp32,
    beta [N, H], S [N, H, 128, 128] fp32 updated in place.  Returns o [N, H, 128]."""
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _need(t, name, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(S, "S", torch.float32, dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    o = out if out is not None else torch.empty(v.shape, dtype=v.dtype, device=dev)
    _need(o, "out", v.dtype, dev)
    with torch.cuda.device(dev):
        _check(lib.kda_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g),
                                      _ptr(beta), _ptr(S), _ptr(o), N, H, dk, dv, _stream(dev)))
    return o


def recurrent_multi_step(q, k, v, g, beta, S, n_advance=None, *, out=None,
                         return_outputs=True):
    """T tokens per sequence: q, k, v [N, T, H, 128] (bf16/fp32), g [N, T, H, 128]
    fp32, beta [N, T, H], S [N, H, 128, 128] fp32 advanced in place by n_advance[n]
    tokens (int32 [N] on the device; None = all T).  Returns o [N, T, H, 128] (the
    outputs of all T tokens), or None when return_outputs is False."""
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _need(t, name, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(S, "S", torch.float32, dev)
    if n_advance is not None:
        _need(n_advance, "n_advance", torch.int32, dev)
    N, T, H, dk = q.shape
    dv = v.shape[-1]
    o = None
    if return_outputs:
        o = out if out is not None else torch.empty(v.shape, dtype=v.dtype, device=dev)
        _need(o, "out", v.dtype, dev)
    with torch.cuda.device(dev):
        _check(lib.kda_recurrent_multi_step(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g),
                                            _ptr(beta), _ptr(S), _ptr(o), _ptr(n_advance), N, T,
                                            H, dk, dv, _stream(dev)))
    return o


def profile_enable(on: bool = True):
    """Start (clearing earlier records) or stop per-kernel CUDA-event timing."""
    lib.kda_profile_enable(1 if on else 0)


def profile_collect() -> dict:
    """Waits for the recorded events; returns {kernel: (launches, total_ms)}."""
    n = lib.kda_profile_collect()
    if n < 0:
        raise KdaError(6, "profile collection failed")
    out = {}
    for i in range(n):
        name = ctypes.c_char_p()
        launches = ctypes.c_int()
        total = ctypes.c_double()
        lib.kda_profile_get(i, ctypes.byref(name), ctypes.byref(launches), ctypes.byref(total))
        out[name.value.decode()] = (launches.value, total.value)
    return out


def selftest_wait_timeout(timeout_us: int = 1000, device=None) -> int:
    """Runs the library's bounded-wait self-test (a kernel whose waits nothing
    signals gives up after ``timeout_us``); synchronizes and returns how many of
    its four waiting warps saw the wait end unsatisfied.  The device error flag is
    left set to KDA_ERR_DEVICE_TIMEOUT for :func:`get_device_error`."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    n = ctypes.c_int(-1)
    with torch.cuda.device(device):
        _check(lib.kda_selftest_wait_timeout(int(timeout_us), ctypes.byref(n), _stream(device)))
    return n.value


def get_device_error(device=None):
    """Raise KdaError if a kernel recorded a device-side error (syncs the stream)."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        _check(lib.kda_get_device_error(_stream(device)))
