"""Seeded synthetic inputs for the KDA forward.

This module is shared by the tests, the benchmark and the CPU oracle harness.
It holds only input recipes (shapes, distributions, seeds); none of the KDA
arithmetic lives here.  In particular the bounded gate
``g = g_min * sigmoid(exp(A_h) * z)`` is part of the method, so the recipes
return the gate's inputs ``z`` and ``A`` and leave ``g`` to whoever runs the
method (the CUDA library or the oracle).  For tests of the chunk kernels in
isolation, :func:`uniform_decay` draws ``g`` directly from a plain uniform
distribution on ``[g_min, 0]`` instead.

Distributions follow the workload descriptions of the KDA pages (Kimi K3
report, KDA layer: q and k are L2-normalised per token and head, beta is a
sigmoid of a Gaussian logit, the decay logit z is Gaussian).  ``N(mu, s)``
reads ``s`` as a standard deviation.

Layouts (token-major, one packed batch):
  q, k : [NT, H, dk]   v : [NT, H, dv]   z : [NT, H, dk]   beta : [NT, H]
  A    : [H] fp32      h0 : [N, H, dv, dk] fp32 (the state S stored transposed)
  cu_seqlens : [N + 1] int32, sequence n owns tokens cu[n] .. cu[n+1]-1
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import torch

G_MIN = -5.0  # lower bound of the log-decay (Kimi K3 report, Eq. 5)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic KDA workload."""

    name: str
    seq_lens: tuple  # length of every packed sequence
    H: int
    dk: int = 128
    dv: int = 128
    dtype: torch.dtype = torch.bfloat16
    z_std: float = 1.0
    A_range: float = 1.0  # A_h ~ U(-A_range, A_range); 0 means A = 0
    h0_std: Optional[float] = None  # None: zero initial state
    seed: int = 0

    @property
    def n_tokens(self) -> int:
        return int(sum(self.seq_lens))

    @property
    def n_seqs(self) -> int:
        return len(self.seq_lens)


def _varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator().manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


def tiny(seed: int = 1001) -> Workload:
    """B=1, H=2, T=256, fp32 inputs, A=0, zero initial state."""
    return Workload("kda_fwd_tiny_B1_H2_T256_fp32", (256,), H=2, dtype=torch.float32,
                    A_range=0.0, h0_std=None, seed=seed)


def prefill(seed: int = 1002) -> Workload:
    """One K3 layer: B=1, T=8192, H=96, bf16, A_h~U(-1,1), h0~N(0,0.02)."""
    return Workload("kda_prefill_B1_T8192_H96_bf16", (8192,), H=96, dtype=torch.bfloat16,
                    A_range=1.0, h0_std=0.02, seed=seed)


def varlen(seed: int = 1003) -> Workload:
    """32 sequences, lengths ~U[512, 16384], packed; H=96, bf16, zero h0."""
    lens = _varlen_lengths(32, 512, 16384, seed)
    return Workload(f"kda_varlen_32seq_{sum(lens)}tok_H96_bf16", lens, H=96,
                    dtype=torch.bfloat16, A_range=1.0, h0_std=None, seed=seed)


def long_context(T: int = 1 << 20, seed: int = 1004) -> Workload:
    """B=1, T=1,048,576, H=16, bf16, z~N(0,2) (near-bound decays), zero h0."""
    return Workload(f"kda_long_B1_T{T}_H16_bf16", (T,), H=16, dtype=torch.bfloat16,
                    z_std=2.0, A_range=1.0, h0_std=None, seed=seed)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    N: int
    H: int
    dk: int = 128
    dv: int = 128
    dtype: torch.dtype = torch.bfloat16
    state_std: float = 0.02
    steps: int = 100
    seed: int = 1005


def decode(seed: int = 1005) -> DecodeWorkload:
    """512 sequences x 96 heads, one token per step, fp32 state, 100 steps."""
    return DecodeWorkload("kda_decode_N512_H96_bf16_fp32state", N=512, H=96, seed=seed)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    """L2-normalise the last dimension in fp32 (the q/k producers' L2Norm)."""
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


BLOCK_TOKENS = 4096  # per-token draws are made block by block (see make_inputs)


def _block_seed(seed: int, tensor: int, block: int) -> int:
    """Seed of one token block of one tensor: a fixed mix of (workload seed,
    tensor index, block index), so a block's values depend on nothing else."""
    x = (seed * 0x9E3779B1 + tensor * 0x85EBCA77 + block * 0xC2B2AE3D) & ((1 << 62) - 1)
    return x ^ (x >> 29)


def _per_token(gen_dev, seed, tensor, NT, shape, draw):
    """Concatenates ``draw(generator, n, shape)`` over token blocks of BLOCK_TOKENS,
    each block from its own seeded generator."""
    parts = []
    for b, a in enumerate(range(0, NT, BLOCK_TOKENS)):
        n = min(BLOCK_TOKENS, NT - a)
        parts.append(draw(_gen(gen_dev, _block_seed(seed, tensor, b)), n, shape))
    if not parts:
        return draw(_gen(gen_dev, _block_seed(seed, tensor, 0)), 0, shape)
    return torch.cat(parts) if len(parts) > 1 else parts[0]


def make_inputs(w: Workload, device="cpu", tokens: Optional[int] = None) -> dict:
    """Draw every input of ``w`` from generators seeded with ``w.seed``.

    Per-token tensors (q, k, v, z, beta) are drawn in blocks of BLOCK_TOKENS tokens,
    each block from its own generator seeded by (``w.seed``, tensor, block index):
    the first n tokens of a workload are the same whatever its length, so
    ``tokens=n`` (single-sequence workloads only) generates exactly the first n
    tokens of the full instance.  A and h0 come from a generator seeded with
    ``w.seed``.  Generation happens in fp32 on ``device``; q/k/v/beta are then cast
    to ``w.dtype``.  The returned dict also carries ``cu_seqlens`` (int32).
    """
    dev = torch.device(device)
    NT, H, dk, dv = w.n_tokens, w.H, w.dk, w.dv
    seq_lens = w.seq_lens
    if tokens is not None:
        if w.n_seqs != 1 or not 0 <= tokens <= NT:
            raise ValueError("a prefix is defined for one-sequence workloads, 0 <= tokens <= T")
        NT, seq_lens = int(tokens), (int(tokens),)
    f32 = torch.float32

    def normal(g, n, shp):
        return torch.randn(n, *shp, generator=g, device=dev, dtype=f32)

    q = _unit_rows(_per_token(dev, w.seed, 0, NT, (H, dk), normal))
    k = _unit_rows(_per_token(dev, w.seed, 1, NT, (H, dk), normal))
    v = _per_token(dev, w.seed, 2, NT, (H, dv), normal)
    z = _per_token(dev, w.seed, 3, NT, (H, dk), normal) * w.z_std
    beta = torch.sigmoid(_per_token(dev, w.seed, 4, NT, (H,), normal))
    gen = _gen(dev, w.seed)
    if w.A_range > 0:
        A = (torch.rand(H, generator=gen, device=dev, dtype=f32) * 2 - 1) * w.A_range
    else:
        A = torch.zeros(H, device=dev, dtype=f32)
    if w.h0_std is not None:
        h0 = torch.randn(w.n_seqs, H, dv, dk, generator=gen, device=dev, dtype=f32) * w.h0_std
    else:
        h0 = None
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(seq_lens, dtype=torch.int64), 0)
    dt = w.dtype
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), z=z.to(dt), beta=beta.to(dt), A=A,
                h0=h0, cu_seqlens=cu.to(torch.int32).to(dev))


def uniform_decay(shape, device="cpu", seed: int = 7, lo: float = G_MIN, hi: float = 0.0):
    """Log-decays drawn uniformly from [lo, hi] (fp32), for kernel tests that
    feed ``g`` directly rather than through the gate."""
    gen = _gen(torch.device(device), seed)
    return torch.rand(*shape, generator=gen, device=device, dtype=torch.float32) * (hi - lo) + lo


def make_decode_state(w: DecodeWorkload, device="cpu") -> torch.Tensor:
    gen = _gen(torch.device(device), w.seed)
    return torch.randn(w.N, w.H, w.dv, w.dk, generator=gen, device=device,
                       dtype=torch.float32) * w.state_std


def make_decode_step(w: DecodeWorkload, step: int, device="cpu") -> dict:
    """Inputs of decode step ``step`` (fresh draws each step, seeded per step)."""
    dev = torch.device(device)
    gen = _gen(dev, w.seed * 1000 + 1 + step)
    N, H, dk, dv = w.N, w.H, w.dk, w.dv
    f32 = torch.float32
    q = _unit_rows(torch.randn(N, H, dk, generator=gen, device=dev, dtype=f32))
    k = _unit_rows(torch.randn(N, H, dk, generator=gen, device=dev, dtype=f32))
    v = torch.randn(N, H, dv, generator=gen, device=dev, dtype=f32)
    z = torch.randn(N, H, dk, generator=gen, device=dev, dtype=f32)
    beta = torch.sigmoid(torch.randn(N, H, generator=gen, device=dev, dtype=f32))
    A = (torch.rand(H, generator=_gen(dev, w.seed), device=dev, dtype=f32) * 2 - 1)
    dt = w.dtype
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), z=z.to(dt), beta=beta.to(dt), A=A)


def custom(seq_lens, H=2, dk=128, dv=128, dtype=torch.float32, z_std=1.0, A_range=1.0,
           h0_std=None, seed=11, name="custom") -> Workload:
    return Workload(name, tuple(int(x) for x in seq_lens), H=H, dk=dk, dv=dv, dtype=dtype,
                    z_std=z_std, A_range=A_range, h0_std=h0_std, seed=seed)
