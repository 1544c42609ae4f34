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
            _lib = lib
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle will use (1 if built without OpenMP)."""
    return int(_load().gdn_oracle_max_threads())


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


def recurrent_step(q, k, v, g, beta, scale, state, state_indices=None):
    """One decode step for N sequences, each with one token.

    q, k: [N, Hq, dk]; v: [N, Hv, dv]; g, beta: [N, Hv]; state: [slots, Hv, dk, dv].
    Sequence n reads and writes slot ``state_indices[n]`` (identity when None);
    a negative index skips the sequence (its output row stays zero). Returns
    (o [N, Hv, dv], new_state [slots, Hv, dk, dv]) without touching ``state``.
    """
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
