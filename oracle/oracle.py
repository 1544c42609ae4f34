"""Python face of the CPU oracle for the Gated DeltaNet forward.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark are the only callers. The product library never imports this
module, and this module imports nothing from the product package.

The arithmetic lives in ``gdn_oracle.c`` (plain C, float64, OpenMP over the
independent (sequence, v-head) pairs). This file only builds that C file with
gcc, converts arrays to contiguous float64 and calls it.

Two independent routines (both from the "Lab3 GDN Prefill" page):
  * ``recurrent`` -- the gated delta rule one token at a time (section
    "Linear Attention 与 Gated DeltaNet").
  * ``chunked``  -- the chunk form with any chunk size C (section
    "计算过程描述"), including the tail chunk of length l_c = min(C, L - cC).

On top of them, in float64 numpy, the decode front-end (gates from the
projections, q/k L2 norm, optional bf16 rounding of beta) feeding the
one-token step; see the block above ``softplus``.

Layouts accepted: packed ``[T_total, H, d]`` with ``cu_seqlens`` (int [N+1]),
or dense ``[B, T, H, d]`` with ``cu_seqlens=None``. Outputs come back in the
layout of the inputs, as float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into _build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime on this host: build the same code single-threaded.
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            lib.gdn_oracle_recurrent.argtypes = [i64, ip, i64, i64, i64, i64, dp, dp, dp, dp, dp,
                                                 ctypes.c_double, dp, dp, dp]
            lib.gdn_oracle_recurrent.restype = None
            lib.gdn_oracle_chunked.argtypes = [i64, ip, i64, i64, i64, i64, i64, dp, dp, dp, dp, dp,
                                               ctypes.c_double, dp, dp, dp]
            lib.gdn_oracle_chunked.restype = None
            lib.gdn_oracle_max_threads.argtypes = []
            lib.gdn_oracle_max_threads.restype = ctypes.c_int
            lib.gdn_oracle_set_threads.argtypes = [ctypes.c_int]
            lib.gdn_oracle_set_threads.restype = ctypes.c_int
            lib.gdn_oracle_num_procs.argtypes = []
            lib.gdn_oracle_num_procs.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle will use (1 if built without OpenMP)."""
    return int(_load().gdn_oracle_max_threads())


def set_threads(n: int) -> int:
    """Sets the OpenMP threads of later calls (for timing; results do not
    depend on it) and returns the count in effect."""
    return int(_load().gdn_oracle_set_threads(int(n)))


def num_procs() -> int:
    """Processors the oracle's OpenMP runtime sees on this host."""
    return int(_load().gdn_oracle_num_procs())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a torch tensor; widen exactly on the CPU
        import torch

        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _prepare(q, k, v, g, beta, initial_state, cu_seqlens):
    q, k, v, g, beta, s0 = (_f64(x) for x in (q, k, v, g, beta, initial_state))
    dense = cu_seqlens is None
    if dense:
        if q.ndim != 4:
            raise ValueError("dense layout wants q of shape [B, T, Hq, dk]")
        B, T = q.shape[:2]
        cu = np.arange(B + 1, dtype=np.int64) * T
        q, k, v = (x.reshape(B * T, *x.shape[2:]) for x in (q, k, v))
        g, beta = (x.reshape(B * T, x.shape[2]) for x in (g, beta))
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        B, T = None, None
    Ttot, Hq, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = cu.shape[0] - 1
    if Hv % Hq:
        raise ValueError("Hv must be a multiple of Hq")
    if cu[0] != 0 or cu[-1] != Ttot or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, be non-decreasing and end at T_total")
    if s0 is not None:
        s0 = np.ascontiguousarray(s0.reshape(N, Hv, dk, dv))
    shapes = dict(N=N, Hq=Hq, Hv=Hv, dk=dk, dv=dv, Ttot=Ttot, dense=dense, B=B, T=T)
    return q, k, v, g, beta, s0, cu, shapes


def _finish(out, fin, sh):
    if sh["dense"]:
        out = out.reshape(sh["B"], sh["T"], sh["Hv"], sh["dv"])
    return out, fin


def recurrent(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None):
    """Token-by-token gated delta rule. Returns (o, final_state) in float64."""
    q, k, v, g, beta, s0, cu, sh = _prepare(q, k, v, g, beta, initial_state, cu_seqlens)
    out = np.zeros((sh["Ttot"], sh["Hv"], sh["dv"]), np.float64)
    fin = np.zeros((sh["N"], sh["Hv"], sh["dk"], sh["dv"]), np.float64)
    _load().gdn_oracle_recurrent(sh["N"], cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 sh["Hq"], sh["Hv"], sh["dk"], sh["dv"], _ptr(q), _ptr(k), _ptr(v),
                                 _ptr(g), _ptr(beta), float(scale), _ptr(s0), _ptr(out), _ptr(fin))
    return _finish(out, fin, sh)


def chunked(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None, chunk_size=64):
    """Chunk form with chunk size C = ``chunk_size``. Returns (o, final_state)."""
    if chunk_size < 1:
        raise ValueError("chunk_size must be >= 1")
    q, k, v, g, beta, s0, cu, sh = _prepare(q, k, v, g, beta, initial_state, cu_seqlens)
    out = np.zeros((sh["Ttot"], sh["Hv"], sh["dv"]), np.float64)
    fin = np.zeros((sh["N"], sh["Hv"], sh["dk"], sh["dv"]), np.float64)
    _load().gdn_oracle_chunked(sh["N"], cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                               sh["Hq"], sh["Hv"], sh["dk"], sh["dv"], int(chunk_size), _ptr(q), _ptr(k),
                               _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(s0), _ptr(out), _ptr(fin))
    return _finish(out, fin, sh)


def recurrent_step(q, k, v, g, beta, scale, state, state_indices=None, beta_bf16=False, state_bf16=False):
    """One decode step for N sequences, each with one token.

    q, k: [N, Hq, dk]; v: [N, Hv, dv]; g, beta: [N, Hv]; state: [slots, Hv, dk, dv].
    Sequence n reads and writes slot ``state_indices[n]`` (identity when None);
    a negative index skips the sequence (its output row stays zero). Returns
    (o [N, Hv, dv], new_state [slots, Hv, dk, dv]) without touching ``state``.
    The precision options of the packed SGLang decode kernel: ``beta_bf16``
    rounds beta to the nearest bf16 first; ``state_bf16`` rounds the updated
    slots to the nearest bf16 (a bf16 state cache).
    """
    if beta_bf16:
        beta = round_to_bf16(_f64(beta))
    out, st = _recurrent_step_f64(q, k, v, g, beta, scale, state, state_indices)
    if state_bf16:
        st = round_to_bf16(st)
    return out, st


def _recurrent_step_f64(q, k, v, g, beta, scale, state, state_indices):
    st = _f64(state).copy()
    N = int(_f64(q).shape[0])
    idx = np.arange(N) if state_indices is None else np.asarray(
        state_indices.detach().cpu().numpy() if hasattr(state_indices, "detach") else state_indices, np.int64)
    live = np.nonzero(idx >= 0)[0]
    Hv, dv = _f64(v).shape[1:]
    out = np.zeros((N, Hv, dv), np.float64)
    if live.size == 0:
        return out, st
    sel = lambda x: _f64(x)[live]
    o, fin = recurrent(sel(q), sel(k), sel(v), sel(g), sel(beta), scale,
                       initial_state=st[idx[live]], cu_seqlens=np.arange(live.size + 1))
    out[live] = o
    st[idx[live]] = fin
    return out, st


# ---------------------------------------------------------------------------
# Decode front-end: gates from the projections and the q/k L2 norm.
#
# Written out in float64 numpy from two pages:
#  * "sgl-qwen3-5-moe" page, decode node 7
#    (gdn_packed_recurrent_qk_norm_gating_state_update), steps one and two:
#      k_bar = k / sqrt(sum_j k_j^2 + 1e-6)
#      q_bar = (1 / sqrt(d_k)) * q / sqrt(sum_j q_j^2 + 1e-6)
#      g     = -exp(A_log) * softplus(a + dt_bias),  alpha = exp(g)
#      beta  = sigmoid(b)
#    and steps three and four, the gated delta rule, which ``recurrent_step``
#    already computes.
#  * "Kestrel_VLLM-24" page, gating row of its CPU-versus-kernel table and the
#    k_gdn_beta_g kernel it prints: softplus is linear above 20 and exp below
#    -20; in_proj_b feeds beta and in_proj_a feeds the gate; q and k are
#    normalised per k-head (q also scaled) before the v-heads are expanded.
# The page's bf16 rounding of beta belongs to the packed SGLang kernel's
# precision, not to the method; it is the ``beta_bf16`` option below.
# ---------------------------------------------------------------------------

SOFTPLUS_THRESHOLD = 20.0
QK_NORM_EPS = 1e-6


def softplus(x):
    """softplus(x) = log(1 + e^x) with the two overflow branches: x above 20
    returns x, x below -20 returns e^x (both within e^-20 of the exact value)."""
    x = np.asarray(x, dtype=np.float64)
    mid = np.clip(x, -SOFTPLUS_THRESHOLD, SOFTPLUS_THRESHOLD)
    return np.where(x > SOFTPLUS_THRESHOLD, x,
                    np.where(x < -SOFTPLUS_THRESHOLD, np.exp(np.minimum(x, 0.0)), np.log1p(np.exp(mid))))


def decode_gates(a, b, A_log, dt_bias):
    """Per-token log-decay g and write strength beta from the gate projections.

    a, b: [N, Hv]; A_log, dt_bias: [Hv]. Returns (g, beta), both [N, Hv]:
    g = -exp(A_log) * softplus(a + dt_bias) (the decay in the log domain, so
    alpha = exp(g) is in (0, 1]) and beta = 1 / (1 + exp(-b)).
    """
    a, b, A_log, dt_bias = (_f64(x) for x in (a, b, A_log, dt_bias))
    g = -np.exp(A_log)[None, :] * softplus(a + dt_bias[None, :])
    with np.errstate(over="ignore"):
        beta = 1.0 / (1.0 + np.exp(-b))
    return g, beta


def l2_normalise(x, eps=QK_NORM_EPS):
    """x / sqrt(sum of squares over the last axis + eps): a sum, not a mean."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def recurrent_step_gated(q, k, v, a, b, A_log, dt_bias, scale, state, state_indices=None,
                         beta_bf16=False, state_bf16=False):
    """One decode step from raw projections, in the order of decode node 7.

    q, k: [N, Hq, dk] raw (not normalised); v: [N, Hv, dv]; a, b: [N, Hv];
    A_log, dt_bias: [Hv]; ``scale`` is the query scale (1/sqrt(d_k) on the
    pages), applied once, to q_bar. With ``beta_bf16`` the write strength is
    rounded to the nearest bf16 (ties to even) before use. Everything else as
    ``recurrent_step`` (``state_bf16`` included); returns (o, new_state).
    """
    k_bar = l2_normalise(k)
    q_bar = float(scale) * l2_normalise(q)
    g, beta = decode_gates(a, b, A_log, dt_bias)
    return recurrent_step(q_bar, k_bar, v, g, beta, 1.0, state, state_indices, beta_bf16=beta_bf16,
                          state_bf16=state_bf16)


def round_to_bf16(x):
    """Nearest bfloat16 value (ties to even) of float64 ``x``, as float64.

    bfloat16 keeps 8 significant bits: x = m * 2^e with 2^7 <= |m| < 2^8 is
    rounded to an integer m by numpy's round-half-to-even. Below the smallest
    normal (2^-126) the quantum stays 2^-133 (subnormals)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    e = np.maximum(np.floor(np.log2(np.abs(x[nz]))) - 7, -133.0)
    out[nz] = np.round(x[nz] / np.exp2(e)) * np.exp2(e)
    out[~nz] = x[~nz]
    return out


# ---------------------------------------------------------------------------
# Output gate: head-wise RMSNorm of the read-out, then the SiLU gate of z
# ("sgl-qwen3-5-moe" page, node output_rmsnorm_silu_gate; "Kestrel_VLLM-24"
# page, the gated-RMSNorm row: rsqrt scale, then the weight, then silu(z)).
#   y = (o / sqrt(mean_j o_j^2 + eps)) * weight * silu(z),  over one head's d_v
# The norm comes before the gate (norm_before_gate); the weight multiplies
# directly (no 1 + w parameterisation). The page leaves eps as a symbol; the
# callers pass it.
# ---------------------------------------------------------------------------

def silu(x):
    """x * sigmoid(x) = x / (1 + e^-x)."""
    x = _f64(x)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def gated_rmsnorm(o, z, weight, eps):
    """o, z: [..., d_v]; weight: [d_v]. Returns y of o's shape in float64."""
    o, z, weight = _f64(o), _f64(z), _f64(weight)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + float(eps))
    return (o / rms) * weight * silu(z)


# ---------------------------------------------------------------------------
# Short causal convolution with its state ("Kestrel_VLLM-24" page, the
# conv+SiLU row and kernel: window [s0, s1, s2, x_t] oldest first, the
# history holding the convolution's INPUTS; "sgl-qwen3-5-moe" page, node 6:
# x~_{t,c} = SiLU(sum_l w_{c,l} x_{t-l,c} + b_c), a per-channel convolution,
# b_c = 0 without bias).
# Weights are stored oldest first, w[c, j] multiplying x_{t-(K-1-j), c}, so the
# second page's lag-l weight is w[c, K-1-l]. The state of a sequence is its
# last K-1 inputs, oldest first: [K-1, C].
# ---------------------------------------------------------------------------

def causal_conv1d_silu(x, weight, bias=None, conv_state=None, cu_seqlens=None, state_indices=None):
    """x: [T_total, C] packed tokens of the sequences cu_seqlens delimits
    (one sequence when None); weight: [C, K]; bias: [C] or None;
    conv_state: [slots, K-1, C] (zeros when None); sequence n uses slot
    state_indices[n] (n when None; negative: no state in or out, zero history).
    Returns (out [T_total, C] = SiLU of the convolution, new_state of
    conv_state's shape, the slots of the sequences replaced by their last K-1
    inputs)."""
    x, weight = _f64(x), _f64(weight)
    T, C = x.shape
    K = weight.shape[1]
    b = np.zeros(C) if bias is None else _f64(bias)
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(
        cu_seqlens.detach().cpu().numpy() if hasattr(cu_seqlens, "detach") else cu_seqlens, np.int64)
    N = len(cu) - 1
    idx = np.arange(N) if state_indices is None else np.asarray(
        state_indices.detach().cpu().numpy() if hasattr(state_indices, "detach") else state_indices, np.int64)
    st = None if conv_state is None else _f64(conv_state).copy()
    out = np.zeros((T, C))
    for n in range(N):
        s, e = int(cu[n]), int(cu[n + 1])
        hist = st[idx[n]] if (st is not None and idx[n] >= 0) else np.zeros((K - 1, C))
        ext = np.concatenate([hist, x[s:e]], axis=0)  # [K-1 + L, C], oldest first
        for t in range(e - s):
            window = ext[t:t + K]  # x_{t-K+1} .. x_t
            out[s + t] = silu(np.sum(window * weight.T, axis=0) + b)
        if st is not None and idx[n] >= 0:
            st[idx[n]] = ext[ext.shape[0] - (K - 1):]
    return out, st
