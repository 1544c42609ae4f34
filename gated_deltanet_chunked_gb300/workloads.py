"""Seeded synthetic inputs for the Gated DeltaNet forward.

This module only draws random numbers and casts them. It holds none of the
method's arithmetic, so both the CUDA path (tests, benchmark) and the CPU
oracle can be fed from it.

Shapes follow the Qwen3.5-style GDN layers described on the pages: head
dimension d_k = d_v = 128, grouped q/k heads shared by several v-heads.
Recipe (numpy PCG64, seed = 1000 + workload index):
  q, k  ~ N(0, 1), each head row L2-normalised in float64, then cast
  v     ~ N(0, 1)
  g     = -softplus(N(mu_g, 1))   (per-token log-decay, float32)
  beta  = sigmoid(N(0, 1))         (float32)
  S0    ~ N(0, sigma_s^2)          (float32, sigma_s = 0.1 or 0.05)
Varlen lengths are drawn from the same generator, uniform in [100, 8000].
Decode front-end inputs (raw projections, nothing normalised):
  q, k  ~ N(0, 1), cast          a, b ~ N(0, 1) (float32, [N, Hv])
  A_log = log U[1, 16]           dt_bias ~ U[-6.9, -2.25]   (float32, [Hv])
Output gate: z ~ N(0, 1) (io dtype, like v), RMSNorm weight ~ U[0.5, 1.5]
  (float32, [128]); a stand-alone read-out o ~ N(0, 0.05^2).
Short convolution: x ~ N(0, 1) (io dtype, [T, (2 Hq + Hv) 128]), weight
  ~ U[-0.5, 0.5] (float32, [C, 4]), bias ~ N(0, 0.1^2), conv state ~ N(0, 1)
  (io dtype, [slots, 3, C]).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

DK = 128
DV = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    kind: str  # "prefill" or "decode"
    io_dtype: torch.dtype
    hq: int
    hv: int
    seqlen: int = 0  # dense single sequence length (prefill)
    num_seqs: int = 1  # varlen sequences or decode batch
    varlen: bool = False
    g_mu: float = 0.0
    s0_sigma: Optional[float] = None  # None: zero initial state
    steps: int = 1  # decode: consecutive steps
    description: str = ""

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_f32_T200", 0, "prefill", torch.float32, hq=2, hv=2, seqlen=200, s0_sigma=0.1,
                 description="B=1, T=200 (3 full chunks + 8-token tail), Hq=Hv=2, f32 everywhere, S0~N(0,0.1^2)"),
        Workload("prefill_T4096_hq16_hv32", 1, "prefill", torch.bfloat16, hq=16, hv=32, seqlen=4096,
                 description="B=1, T=4096, Hq=16, Hv=32, d=128, bf16 q/k/v, f32 g/beta, zero S0"),
        Workload("varlen_8seq_hq16_hv32", 2, "prefill", torch.bfloat16, hq=16, hv=32, num_seqs=8, varlen=True,
                 s0_sigma=0.05,
                 description="8 packed sequences, lengths U[100,8000], Hq=16, Hv=32, bf16, S0~N(0,0.05^2)"),
        Workload("long_T65536_hq16_hv32", 3, "prefill", torch.bfloat16, hq=16, hv=32, seqlen=65536, g_mu=-2.0,
                 description="B=1, T=65536, Hq=16, Hv=32, bf16, g=-softplus(N(-2,1)), zero S0"),
        Workload("decode_N256_hq16_hv32", 4, "decode", torch.bfloat16, hq=16, hv=32, num_seqs=256, s0_sigma=0.05,
                 steps=100,
                 description="256 sequences x 1 token, Hq=16, Hv=32, f32 state [256,32,128,128], 100 steps"),
    ]
}


def _normal(rng, shape, mu=0.0, sigma=1.0):
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma) + np.float32(mu)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    x64 = x.astype(np.float64)
    x64 /= np.sqrt(np.sum(x64 * x64, axis=-1, keepdims=True))
    return x64


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x.astype(np.float64))


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x.astype(np.float64)))


def varlen_lengths(rng: np.random.Generator, n: int, lo: int = 100, hi: int = 8000) -> np.ndarray:
    return rng.integers(lo, hi + 1, size=n)


def make_token_inputs(rng, T, hq, hv, io_dtype, g_mu=0.0, dk=DK, dv=DV):
    """q, k, v, g, beta for T tokens (packed [T, H, d] / [T, H])."""
    q = torch.from_numpy(_unit_rows(_normal(rng, (T, hq, dk)))).to(io_dtype)
    k = torch.from_numpy(_unit_rows(_normal(rng, (T, hq, dk)))).to(io_dtype)
    v = torch.from_numpy(_normal(rng, (T, hv, dv))).to(io_dtype)
    g = torch.from_numpy(-_softplus(_normal(rng, (T, hv), mu=g_mu))).to(torch.float32)
    beta = torch.from_numpy(_sigmoid(_normal(rng, (T, hv)))).to(torch.float32)
    return q, k, v, g, beta


def make_prefill(w: Workload, seed: Optional[int] = None):
    """Inputs of a prefill workload as CPU torch tensors.

    Returns a dict with q, k [T_total, Hq, 128], v [T_total, Hv, 128],
    g, beta [T_total, Hv] f32, initial_state [N, Hv, 128, 128] f32 or None,
    cu_seqlens int32 [N+1] or None (dense single sequence), scale.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    if w.varlen:
        lens = varlen_lengths(rng, w.num_seqs)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T, N = int(cu[-1]), w.num_seqs
    else:
        cu, T, N = None, w.seqlen, 1
    q, k, v, g, beta = make_token_inputs(rng, T, w.hq, w.hv, w.io_dtype, g_mu=w.g_mu)
    s0 = None
    if w.s0_sigma is not None:
        s0 = torch.from_numpy(_normal(rng, (N, w.hv, DK, DV), sigma=w.s0_sigma))
    return dict(q=q, k=k, v=v, g=g, beta=beta, initial_state=s0,
                cu_seqlens=None if cu is None else torch.from_numpy(cu),
                scale=1.0 / math.sqrt(DK), num_seqs=N, total_tokens=T)


def make_decode_state(w: Workload, seed: Optional[int] = None):
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    return torch.from_numpy(_normal(rng, (w.num_seqs, w.hv, DK, DV), sigma=w.s0_sigma))


def make_decode_step(w: Workload, step: int):
    """Fresh seeded inputs of decode step ``step`` (one token per sequence)."""
    rng = np.random.Generator(np.random.PCG64([w.seed, 1 + step]))
    q, k, v, g, beta = make_token_inputs(rng, w.num_seqs, w.hq, w.hv, w.io_dtype, g_mu=w.g_mu)
    return dict(q=q, k=k, v=v, g=g, beta=beta, scale=1.0 / math.sqrt(DK))


def make_custom_prefill(seed, lengths, hq, hv, io_dtype=torch.float32, s0_sigma=None, g_mu=0.0,
                        dk=DK, dv=DV, packed=True):
    """Prefill inputs of arbitrary small shape for parity tests.

    ``lengths``: list of sequence lengths. Always packed [T_total, H, d]
    with int32 cu_seqlens (dense callers pass a single length and may drop it).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    cu = np.concatenate([[0], np.cumsum(np.asarray(lengths, np.int64))]).astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    q, k, v, g, beta = make_token_inputs(rng, T, hq, hv, io_dtype, g_mu=g_mu, dk=dk, dv=dv)
    s0 = None
    if s0_sigma is not None:
        s0 = torch.from_numpy(_normal(rng, (N, hv, dk, dv), sigma=s0_sigma))
    return dict(q=q, k=k, v=v, g=g, beta=beta, initial_state=s0, cu_seqlens=torch.from_numpy(cu),
                scale=1.0 / math.sqrt(dk), num_seqs=N, total_tokens=T)


def make_decode_gate_params(w: Workload, seed: Optional[int] = None):
    """Per-v-head parameters of the decode front-end: A_log, dt_bias [Hv] f32."""
    rng = np.random.Generator(np.random.PCG64([w.seed if seed is None else seed, 0]))
    A_log = np.log(rng.uniform(1.0, 16.0, size=w.hv)).astype(np.float32)
    dt_bias = rng.uniform(-6.9, -2.25, size=w.hv).astype(np.float32)
    return torch.from_numpy(A_log), torch.from_numpy(dt_bias)


def make_decode_step_gated(w: Workload, step: int, a_sigma: float = 1.0):
    """Raw inputs of gated decode step ``step``: q, k [N, Hq, 128] and v
    [N, Hv, 128] in the io dtype, gate projections a, b [N, Hv] f32."""
    rng = np.random.Generator(np.random.PCG64([w.seed, 1 + step, 1]))
    N = w.num_seqs
    q = torch.from_numpy(_normal(rng, (N, w.hq, DK))).to(w.io_dtype)
    k = torch.from_numpy(_normal(rng, (N, w.hq, DK))).to(w.io_dtype)
    v = torch.from_numpy(_normal(rng, (N, w.hv, DV))).to(w.io_dtype)
    a = torch.from_numpy(_normal(rng, (N, w.hv), sigma=a_sigma))
    b = torch.from_numpy(_normal(rng, (N, w.hv)))
    return dict(q=q, k=k, v=v, a=a, b=b, scale=1.0 / math.sqrt(DK))


def make_output_gate(seed: int, tokens: int, hv: int, io_dtype, with_o: bool = False):
    """z [tokens, Hv, 128] (io dtype) and the RMSNorm weight [128] f32 of the
    output gate; with ``with_o`` also a stand-alone read-out o of z's shape."""
    rng = np.random.Generator(np.random.PCG64([seed, 2]))
    z = torch.from_numpy(_normal(rng, (tokens, hv, DV))).to(io_dtype)
    weight = torch.from_numpy(rng.uniform(0.5, 1.5, size=DV).astype(np.float32))
    if not with_o:
        return z, weight
    o = torch.from_numpy(_normal(rng, (tokens, hv, DV), sigma=0.05)).to(io_dtype)
    return z, weight, o


def make_conv_inputs(seed: int, tokens: int, hq: int, hv: int, io_dtype, slots: int = 0, bias: bool = True):
    """Inputs of the short convolution: x [tokens, C], weight [C, 4], bias [C]
    (or None) and a conv state [slots, 3, C] (None for slots = 0), with
    C = (2 hq + hv) * 128."""
    rng = np.random.Generator(np.random.PCG64([seed, 3]))
    C = (2 * hq + hv) * DK
    x = torch.from_numpy(_normal(rng, (tokens, C))).to(io_dtype)
    weight = torch.from_numpy(rng.uniform(-0.5, 0.5, size=(C, 4)).astype(np.float32))
    b = torch.from_numpy(_normal(rng, (C,), sigma=0.1)) if bias else None
    state = torch.from_numpy(_normal(rng, (slots, 3, C))).to(io_dtype) if slots else None
    return x, weight, b, state
