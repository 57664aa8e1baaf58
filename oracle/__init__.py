"""fp64 CPU oracle for the KDA forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never links, loads or calls it, and the two share no code.

Functions and the passages they follow:

* :func:`gate` -- bounded log-decay ``g = g_min * Sigmoid(exp(A_h) z)``
  ("Kimi K3 technical report review" (devpress/CSDN), section 3.2, Eq. 5).
* :func:`recurrence` -- the token-by-token KDA recurrence
  ``S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T``, ``o_t = S_t^T q_t``
  (same review, section 3.1, Eq. 1; "Kimi K3: architecture, training and
  inference systems" (weigao.cc), section 3.1, product and delta forms).
  Implemented in C (``kda_oracle.c``), double precision, threads over
  (sequence, head) units.
* :func:`explicit_product_form` -- the same recurrence with the transition
  matrix ``(I - b k k^T) Diag(alpha)`` formed explicitly (numpy, tiny sizes).
* :func:`chunked` -- the chunkwise WY/UT form for a chunk size ``C``
  ("Kimi K3 notes" (s1mplewind blog), section "Chunkwise form": M, W, U, the
  state update and the inter/intra-chunk output split), evaluated with explicit
  cumulative decays in fp64 and a library linear solve; tiny sizes only.
* :func:`decode_step` -- one token of the recurrence for many independent
  (sequence, head) states, the decode form.
* :func:`l2_normalize` -- ``x / sqrt(|x|^2 + eps)`` per token and head, the
  L2Norm applied to q and k before the recurrence ("Kimi K3: architecture,
  training and inference systems", section 3.2, the q / k branches; done inside
  the FlashKDA prepare kernel, "Kimi K3 notes", section "FlashKDA", K1).
* :func:`gate_softplus` -- the unbounded gate ``g = -exp(A_h) Softplus(z)`` that
  the bounded one replaced ("Kimi K3 technical report review", section 3.2).
* :func:`output_gate` -- the head-wise RMSNorm of the KDA output times the
  full-rank Sigmoid gate ("Kimi K3 technical report review", section 3.3, Eq. 6;
  the same systems page, section 3.3), without the W_o / W_g projections.

Pins: ``tests/test_oracle.py`` checks these against closed forms, special
cases and invariants the pages fix (see that file's docstring).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")

_lib_cache: dict = {}


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle into a shared library (plain gcc, -O2, IEEE fp)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", src,
                           "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle library at ``path``."""
    path = path or compile_oracle()
    if path in _lib_cache:
        return _lib_cache[path]
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kda_oracle_gate.argtypes = [dp, dp, ctypes.c_double, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_int, dp]
    lib.kda_oracle_gate.restype = None
    lib.kda_oracle_recurrence.argtypes = [dp, dp, dp, dp, dp, dp,
                                          ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, dp, dp, ctypes.c_int]
    lib.kda_oracle_recurrence.restype = ctypes.c_int
    _lib_cache[path] = lib
    return lib


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact widening to fp64 on the host
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def gate(z, A, g_min: float = -5.0, lib=None) -> np.ndarray:
    """g[t, h, c] = g_min * Sigmoid(exp(A[h]) * z[t, h, c]) in fp64."""
    lib = lib or load()
    z = _f64(z)
    A = _f64(A)
    NT, H, dk = z.shape
    g = np.empty_like(z)
    lib.kda_oracle_gate(_ptr(z), _ptr(A), float(g_min), NT, H, dk, _ptr(g))
    return g


def recurrence(q, k, v, g, beta, h0=None, cu_seqlens=None, form: int = 0,
               n_threads: Optional[int] = None, lib=None):
    """Token-by-token KDA forward.  Returns ``(o, hT)`` as fp64 arrays.

    q, k, g: [NT, H, dk]; v: [NT, H, dv]; beta: [NT, H]; h0: [N, H, dv, dk] or
    None; cu_seqlens: [N+1] (default: one sequence of NT tokens).
    ``form`` 0 = product form, 1 = delta form.
    """
    lib = lib or load()
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    NT, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu = np.array([0, NT], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    if h0 is not None:
        assert h0.shape == (N, H, dv, dk), h0.shape
    o = np.zeros((NT, H, dv), dtype=np.float64)
    hT = np.zeros((N, H, dv, dk), dtype=np.float64)
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    rc = lib.kda_oracle_recurrence(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                   cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, dk,
                                   dv, int(form), _ptr(o), _ptr(hT), int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, hT


def decode_step(q, k, v, g, beta, S, n_threads: Optional[int] = None, lib=None):
    """One decode token for N independent sequences.

    q, k, g: [N, H, dk]; v: [N, H, dv]; beta: [N, H]; S: [N, H, dv, dk].
    Returns ``(o [N, H, dv], S_new [N, H, dv, dk])``.
    """
    q = _f64(q)
    N = q.shape[0]
    cu = np.arange(N + 1, dtype=np.int64)
    return recurrence(q, k, v, g, beta, h0=S, cu_seqlens=cu, n_threads=n_threads, lib=lib)


def explicit_product_form(q, k, v, g, beta, h0=None):
    """KDA with the transition matrix formed explicitly (one sequence).

    For each token: ``M_t = (I - b k k^T) @ Diag(exp(g))`` (a dk x dk matrix),
    ``S = M_t @ S + b * outer(k, v)``, ``o_t = S^T q``.  Tiny sizes only.
    Returns ``(o [T, H, dv], hT [H, dv, dk])``.
    """
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    T, H, dk = q.shape
    dv = v.shape[2]
    o = np.zeros((T, H, dv))
    hT = np.zeros((H, dv, dk))
    eye = np.eye(dk)
    for h in range(H):
        S = np.zeros((dk, dv)) if h0 is None else h0[h].T.copy()
        for t in range(T):
            kt = k[t, h]
            M = (eye - beta[t, h] * np.outer(kt, kt)) @ np.diag(np.exp(g[t, h]))
            S = M @ S + beta[t, h] * np.outer(kt, v[t, h])
            o[t, h] = S.T @ q[t, h]
        hT[h] = S.T
    return o, hT


def chunked(q, k, v, g, beta, h0=None, cu_seqlens=None, C: int = 64):
    """Chunkwise WY/UT evaluation of KDA in fp64 (brute force, tiny sizes).

    Per chunk [t] of length L <= C, with G the inclusive cumulative sum of g
    inside the chunk and Gamma = exp(G) (row r holds gamma_r = prod_{j<=r} alpha_j):
        A   = StrictTril(Diag(beta) (Gamma*K) (K/Gamma)^T)
        M   = (I + A)^{-1} Diag(beta)
        W   = M (Gamma*K),   U = M V
        Vt  = U - W S                       (the "pseudo-value" term)
        O   = (Gamma*Q) S + Tril((Gamma*Q) (K/Gamma)^T) Vt
        S'  = Diag(gamma_C) S + ((gamma_C/Gamma)*K)^T Vt
    following "Kimi K3 notes" (s1mplewind blog), section "Chunkwise form".
    fp64 holds exp(+-5C) for C <= 64, so no tile references are needed here.
    """
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    NT, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu = [0, NT]
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    o = np.zeros((NT, H, dv))
    hT = np.zeros((N, H, dv, dk))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[n, h].T.copy()
            for s in range(cu[n], cu[n + 1], C):
                e = min(s + C, cu[n + 1])
                L = e - s
                K = k[s:e, h]
                Q = q[s:e, h]
                V = v[s:e, h]
                b = beta[s:e, h]
                G = np.cumsum(g[s:e, h], axis=0)
                Gam = np.exp(G)
                Kg, Kn, Qg = Gam * K, K / Gam, Gam * Q
                A = np.tril(np.diag(b) @ Kg @ Kn.T, -1)
                M = np.linalg.solve(np.eye(L) + A, np.diag(b))
                W, U = M @ Kg, M @ V
                Vt = U - W @ S
                o[s:e, h] = Qg @ S + np.tril(Qg @ Kn.T) @ Vt
                gC = Gam[-1]
                S = gC[:, None] * S + (np.exp(G[-1][None, :] - G) * K).T @ Vt
            hT[n, h] = S.T
    return o, hT


def chunk_cumsum(g, cu_seqlens=None, C: int = 64) -> np.ndarray:
    """Running sum of g inside each C-token chunk of each sequence (chunks start
    at cu[n] + C m): the log of the in-chunk cumulative decay Gamma of the
    chunkwise form ("Kimi K3 notes", section "Chunkwise form")."""
    g = _f64(g)
    NT = g.shape[0]
    if cu_seqlens is None:
        cu = [0, NT]
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = [int(x) for x in cu_seqlens]
    out = np.zeros_like(g)
    for n in range(len(cu) - 1):
        for s in range(cu[n], cu[n + 1], C):
            e = min(s + C, cu[n + 1])
            out[s:e] = np.cumsum(g[s:e], axis=0)
    return out


def l2_normalize(x, eps: float) -> np.ndarray:
    """``x / sqrt(sum_c x_c^2 + eps)`` over the last axis (one head's channels) in
    fp64.  The pages name the L2Norm without an epsilon; ``eps`` is the caller's."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def output_gate(o, x, w=None, eps: float = 1e-6) -> np.ndarray:
    """``Sigmoid(x) * w * o / sqrt(mean_c(o_c^2) + eps)`` over the last axis (the dv
    channels of one head) in fp64: the head-wise RMSNorm of the recurrent output
    and the input-dependent full-rank gate, ``x`` being the gate logits W_g x_t.
    ``w`` is the RMSNorm weight over the channels (None: ones)."""
    o, x = _f64(o), _f64(x)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    y = o / rms / (1.0 + np.exp(-x))
    if w is not None:
        y = y * _f64(w)
    return y


def gate_softplus(z, A) -> np.ndarray:
    """``g[t, h, c] = -exp(A[h]) * log(1 + exp(z[t, h, c]))`` in fp64 (Softplus as
    ``logaddexp(0, z)``, exact for large |z|)."""
    z, A = _f64(z), _f64(A)
    return -np.exp(A)[None, :, None] * np.logaddexp(0.0, z)
