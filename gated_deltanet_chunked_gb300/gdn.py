"""Thin ctypes binding of libgdn.so (include/gdn.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. There is
no fallback: if libgdn.so cannot be built or loaded, ``load()`` raises.

The entry points keep the C names:
  gdn_chunk_fwd, gdn_chunk_fwd_workspace_size, gdn_recurrent_step,
  gdn_recurrent_step_gated, gdn_gated_rmsnorm, gdn_causal_conv1d_silu,
  gdn_causal_conv1d_silu_step, gdn_gating,
  gdn_read_device_status, gdn_status_string, gdn_version.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional

import torch

from . import build as _build

GDN_OK, GDN_EINVAL, GDN_EUNSUPPORTED, GDN_ECUDA, GDN_ETIMEOUT, GDN_EDEVICE_INPUT, GDN_ETOOBIG = range(7)
GDN_NOALLOC_SCRATCH_BYTES = 32 << 20
GDN_DT_F32, GDN_DT_BF16 = 0, 1
GDN_FLAG_BETA_BF16, GDN_FLAG_STATE_BF16 = 1 << 1, 1 << 2

SYMBOLS = ("gdn_chunk_fwd", "gdn_chunk_fwd_workspace_size", "gdn_recurrent_step", "gdn_read_device_status",
           "gdn_status_string", "gdn_version", "gdn_profile_enable", "gdn_profile_collect", "gdn_kernel_name",
           "gdn_chunk_fwd_noalloc", "gdn_recurrent_step_gated", "gdn_gated_rmsnorm", "gdn_causal_conv1d_silu",
           "gdn_gating", "gdn_causal_conv1d_silu_step", "gdn_chunk_fwd_gated")
GDN_K_COUNT = 11


class GdnProblem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seqlen", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("total_tokens", ctypes.c_int32), ("hq", ctypes.c_int32), ("hv", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("num_state_slots", ctypes.c_int32)]


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gdn_status_string(status)}")


_lib = None
_lock = threading.Lock()
_vp, _fp, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p


def load(path: Optional[str] = None):
    """Build (if stale) and load libgdn.so; raises if either step fails."""
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(path or _build.build())
            P = ctypes.POINTER(GdnProblem)
            lib.gdn_chunk_fwd.argtypes = [P, _vp, _vp, _vp, _fp, _fp, ctypes.c_float, _fp, _ip, _vp, _fp, _vp,
                                          ctypes.c_size_t, _vp]
            lib.gdn_chunk_fwd.restype = ctypes.c_int
            lib.gdn_chunk_fwd_gated.argtypes = [P, _vp, _vp, _vp, _fp, _fp, ctypes.c_float, _fp, _ip, _vp, _fp,
                                                ctypes.c_float, _vp, _fp, _vp, ctypes.c_size_t, _vp]
            lib.gdn_chunk_fwd_gated.restype = ctypes.c_int
            lib.gdn_chunk_fwd_workspace_size.argtypes = [P]
            lib.gdn_chunk_fwd_workspace_size.restype = ctypes.c_size_t
            lib.gdn_recurrent_step.argtypes = [P, _vp, _vp, _vp, _fp, _fp, ctypes.c_float, _fp, _ip, _vp, _vp]
            lib.gdn_recurrent_step.restype = ctypes.c_int
            lib.gdn_recurrent_step_gated.argtypes = [P, _vp, _vp, _vp, _fp, _fp, _fp, _fp, ctypes.c_float, _fp,
                                                     _ip, _vp, _fp, ctypes.c_float, _vp, _vp]
            lib.gdn_gated_rmsnorm.argtypes = [P, _vp, _vp, _fp, ctypes.c_float, _vp, _vp]
            lib.gdn_gated_rmsnorm.restype = ctypes.c_int
            lib.gdn_causal_conv1d_silu.argtypes = [P, _vp, _fp, _fp, _vp, _ip, _ip, ctypes.c_int, _vp, _vp, _vp, _vp]
            lib.gdn_causal_conv1d_silu.restype = ctypes.c_int
            lib.gdn_causal_conv1d_silu_step.argtypes = [P, _vp, _fp, _fp, _vp, _ip, ctypes.c_int, _vp, _vp, _vp,
                                                        _vp]
            lib.gdn_causal_conv1d_silu_step.restype = ctypes.c_int
            lib.gdn_gating.argtypes = [P, _fp, _fp, _fp, _fp, _fp, _fp, _vp]
            lib.gdn_gating.restype = ctypes.c_int
            lib.gdn_recurrent_step_gated.restype = ctypes.c_int
            lib.gdn_read_device_status.argtypes = [_vp, ctypes.c_int]
            lib.gdn_read_device_status.restype = ctypes.c_int
            lib.gdn_status_string.argtypes = [ctypes.c_int]
            lib.gdn_status_string.restype = ctypes.c_char_p
            lib.gdn_version.argtypes = []
            lib.gdn_version.restype = ctypes.c_int
            lib.gdn_profile_enable.argtypes = [ctypes.c_int]
            lib.gdn_profile_enable.restype = ctypes.c_int
            lib.gdn_profile_collect.argtypes = [_vp, _vp, _vp, ctypes.c_int, ctypes.c_int]
            lib.gdn_profile_collect.restype = ctypes.c_int
            lib.gdn_chunk_fwd_noalloc.argtypes = [P, _vp, _vp, _vp, _fp, _fp, ctypes.c_float, _fp, _ip, _vp, _fp,
                                                  _vp]
            lib.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
            lib.gdn_kernel_name.argtypes = [ctypes.c_int]
            lib.gdn_kernel_name.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def lib():
    return load()


def gdn_status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def gdn_version() -> int:
    return int(load().gdn_version())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libgdn wants contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _io_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GDN_DT_F32
    if t.dtype == torch.bfloat16:
        return GDN_DT_BF16
    raise ValueError(f"unsupported io dtype {t.dtype}")


def _want(dtype, **tensors):
    """Raises ValueError unless every given (non-None) tensor has ``dtype``."""
    for name, t in tensors.items():
        if t is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def prefill_problem(q: torch.Tensor, v: torch.Tensor, num_seqs: int, packed: bool) -> GdnProblem:
    """Descriptor for q [T_total, Hq, dk] (packed) or [B, T, Hq, dk] (dense)."""
    if packed:
        Ttot, hq, dk = q.shape
        batch, seqlen = 1, 0
    else:
        batch, seqlen, hq, dk = q.shape
        Ttot = batch * seqlen
        num_seqs = batch
    return GdnProblem(batch, seqlen, num_seqs, Ttot, hq, v.shape[-2], dk, v.shape[-1], _io_dtype(q), 0, 0)


def gdn_chunk_fwd_workspace_size(problem: GdnProblem) -> int:
    return int(load().gdn_chunk_fwd_workspace_size(ctypes.byref(problem)))


def gdn_chunk_fwd(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None, out=None,
                  final_state=None, output_final_state=True, workspace=None, stream=None,
                  z=None, norm_weight=None, norm_eps=1e-6):
    """Chunked prefill. Packed when ``cu_seqlens`` (int32 device [N+1]) is given.

    Returns (out, final_state). ``workspace`` (uint8 device tensor) is
    allocated with PyTorch when not supplied. With ``z`` (like v) and
    ``norm_weight`` [128] f32, out holds the output gate applied to the
    read-out (gdn_chunk_fwd_gated).
    """
    packed = cu_seqlens is not None
    num_seqs = cu_seqlens.numel() - 1 if packed else q.shape[0]
    _want(q.dtype, k=k, v=v, out=out, z=z)
    _want(torch.float32, g=g, beta=beta, initial_state=initial_state, final_state=final_state,
          norm_weight=norm_weight)
    _want(torch.int32, cu_seqlens=cu_seqlens)
    prob = prefill_problem(q, v, num_seqs, packed)
    if out is None:
        out = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((prob.num_seqs, prob.hv, prob.dk, prob.dv), dtype=torch.float32, device=v.device)
    need = gdn_chunk_fwd_workspace_size(prob)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=v.device)
    if z is None:
        st = load().gdn_chunk_fwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                  _ptr(final_state), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                  _stream(stream))
        where = "gdn_chunk_fwd"
    else:
        st = load().gdn_chunk_fwd_gated(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(z),
                                        _ptr(norm_weight), ctypes.c_float(norm_eps), _ptr(out), _ptr(final_state),
                                        _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream))
        where = "gdn_chunk_fwd_gated"
    if st != GDN_OK:
        raise GdnError(st, where)
    return out, final_state


def gdn_chunk_fwd_noalloc(q, k, v, g, beta, scale, out, final_state=None, initial_state=None, cu_seqlens=None,
                          stream=None):
    """gdn_chunk_fwd without a workspace, for callers that cannot allocate:
    the library uses its fixed device scratch array (GDN_NOALLOC_SCRATCH_BYTES)
    and allocates nothing. ``out`` (and ``final_state`` if wanted) must be
    supplied. Raises GdnError(GDN_ETOOBIG) for problems above that size."""
    packed = cu_seqlens is not None
    num_seqs = cu_seqlens.numel() - 1 if packed else q.shape[0]
    _want(q.dtype, k=k, v=v, out=out)
    _want(torch.float32, g=g, beta=beta, initial_state=initial_state, final_state=final_state)
    _want(torch.int32, cu_seqlens=cu_seqlens)
    prob = prefill_problem(q, v, num_seqs, packed)
    st = load().gdn_chunk_fwd_noalloc(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                      ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                      _ptr(final_state), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_chunk_fwd_noalloc")
    return out, final_state


def _decode_flags(state, beta_bf16):
    return (GDN_FLAG_STATE_BF16 if state.dtype == torch.bfloat16 else 0) | (GDN_FLAG_BETA_BF16 if beta_bf16 else 0)


def gdn_recurrent_step(q, k, v, g, beta, scale, state, state_indices=None, out=None, stream=None,
                       beta_bf16=False):
    """One decode step; ``state`` [slots, Hv, 128, 128] (f32, or bf16 for a
    bf16 state cache) is updated in place. ``beta_bf16`` rounds beta to bf16."""
    N, hq, dk = q.shape
    _want(q.dtype, k=k, v=v, out=out)
    _want(torch.float32, g=g, beta=beta)
    _want(torch.int32, state_indices=state_indices)
    if state.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"state must be float32 or bfloat16, got {state.dtype}")
    prob = GdnProblem(N, 1, N, N, hq, v.shape[1], dk, v.shape[2], _io_dtype(q), _decode_flags(state, beta_bf16),
                      state.shape[0])
    if out is None:
        out = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    st = load().gdn_recurrent_step(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   ctypes.c_float(scale), _ptr(state), _ptr(state_indices), _ptr(out),
                                   _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_recurrent_step")
    return out


def gdn_recurrent_step_gated(q, k, v, a, b, A_log, dt_bias, scale, state, state_indices=None, out=None,
                             stream=None, z=None, norm_weight=None, norm_eps=1e-6, beta_bf16=False):
    """Decode step from raw q/k and the gate projections a, b [N, Hv] with
    per-head A_log, dt_bias [Hv] (all f32); ``state`` is updated in place.
    With ``z`` [N, Hv, 128] and ``norm_weight`` [128] f32 the output gate
    (head-wise RMSNorm, then silu(z)) is applied before the store. A bf16
    ``state`` is a bf16 state cache; ``beta_bf16`` rounds beta to bf16."""
    N, hq, dk = q.shape
    _want(q.dtype, k=k, v=v, out=out, z=z)
    _want(torch.float32, a=a, b=b, A_log=A_log, dt_bias=dt_bias, norm_weight=norm_weight)
    _want(torch.int32, state_indices=state_indices)
    if state.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"state must be float32 or bfloat16, got {state.dtype}")
    prob = GdnProblem(N, 1, N, N, hq, v.shape[1], dk, v.shape[2], _io_dtype(q), _decode_flags(state, beta_bf16),
                      state.shape[0])
    if out is None:
        out = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    st = load().gdn_recurrent_step_gated(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                         _ptr(A_log), _ptr(dt_bias), ctypes.c_float(scale), _ptr(state),
                                         _ptr(state_indices), _ptr(z), _ptr(norm_weight),
                                         ctypes.c_float(norm_eps), _ptr(out), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_recurrent_step_gated")
    return out


def gdn_gated_rmsnorm(o, z, weight, eps, out=None, stream=None):
    """y = o / sqrt(mean(o^2) + eps) * weight * silu(z) per (token, head) row
    of o, z [T, Hv, 128] (io dtype) with weight [128] f32. ``out`` may be o."""
    T, hv, dv = o.shape
    _want(o.dtype, z=z, out=out)
    _want(torch.float32, weight=weight)
    prob = GdnProblem(1, 0, 1, T, 1, hv, dv, dv, _io_dtype(o), 0, 0)
    if out is None:
        out = torch.empty_like(o)
    st = load().gdn_gated_rmsnorm(ctypes.byref(prob), _ptr(o), _ptr(z), _ptr(weight), ctypes.c_float(eps),
                                  _ptr(out), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_gated_rmsnorm")
    return out


def gdn_causal_conv1d_silu(x, weight, hq, hv, bias=None, conv_state=None, state_indices=None, cu_seqlens=None,
                           norm_qk=False, q=None, k=None, v=None, stream=None):
    """Short causal convolution (4 taps, weight [C, 4] f32 oldest first) + SiLU
    over packed tokens x [T, C] (C = (2 hq + hv) * 128), split into q, k
    [T, hq, 128] and v [T, hv, 128]; ``conv_state`` [slots, 3, C] is read and
    updated in place. ``norm_qk`` L2-normalises every q and k head row."""
    T, C = x.shape
    if C != (2 * hq + hv) * 128:
        raise ValueError("x must have (2 hq + hv) * 128 channels")
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _want(x.dtype, conv_state=conv_state, q=q, k=k, v=v)
    _want(torch.float32, weight=weight, bias=bias)
    _want(torch.int32, state_indices=state_indices, cu_seqlens=cu_seqlens)
    slots = 0 if conv_state is None else conv_state.shape[0]
    prob = GdnProblem(1, 0, N, T, hq, hv, 128, 128, _io_dtype(x), 0, slots)
    q = torch.empty((T, hq, 128), dtype=x.dtype, device=x.device) if q is None else q
    k = torch.empty((T, hq, 128), dtype=x.dtype, device=x.device) if k is None else k
    v = torch.empty((T, hv, 128), dtype=x.dtype, device=x.device) if v is None else v
    st = load().gdn_causal_conv1d_silu(ctypes.byref(prob), _ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state),
                                       _ptr(state_indices), _ptr(cu_seqlens), int(bool(norm_qk)), _ptr(q), _ptr(k),
                                       _ptr(v), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_causal_conv1d_silu")
    return q, k, v


def gdn_causal_conv1d_silu_step(x, weight, hq, hv, bias=None, conv_state=None, state_indices=None, norm_qk=False,
                                q=None, k=None, v=None, stream=None):
    """gdn_causal_conv1d_silu for one token per sequence: x [N, C]."""
    N, C = x.shape
    if C != (2 * hq + hv) * 128:
        raise ValueError("x must have (2 hq + hv) * 128 channels")
    _want(x.dtype, conv_state=conv_state, q=q, k=k, v=v)
    _want(torch.float32, weight=weight, bias=bias)
    _want(torch.int32, state_indices=state_indices)
    slots = 0 if conv_state is None else conv_state.shape[0]
    prob = GdnProblem(N, 1, N, N, hq, hv, 128, 128, _io_dtype(x), 0, slots)
    q = torch.empty((N, hq, 128), dtype=x.dtype, device=x.device) if q is None else q
    k = torch.empty((N, hq, 128), dtype=x.dtype, device=x.device) if k is None else k
    v = torch.empty((N, hv, 128), dtype=x.dtype, device=x.device) if v is None else v
    st = load().gdn_causal_conv1d_silu_step(ctypes.byref(prob), _ptr(x), _ptr(weight), _ptr(bias),
                                            _ptr(conv_state), _ptr(state_indices), int(bool(norm_qk)), _ptr(q),
                                            _ptr(k), _ptr(v), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_causal_conv1d_silu_step")
    return q, k, v


def gdn_gating(a, b, A_log, dt_bias, g=None, beta=None, stream=None):
    """g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b), a, b [T, Hv] f32."""
    T, hv = a.shape
    _want(torch.float32, a=a, b=b, A_log=A_log, dt_bias=dt_bias, g=g, beta=beta)
    prob = GdnProblem(1, 0, 1, T, 1, hv, 128, 128, GDN_DT_F32, 0, 0)
    g = torch.empty_like(a) if g is None else g
    beta = torch.empty_like(a) if beta is None else beta
    st = load().gdn_gating(ctypes.byref(prob), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(g), _ptr(beta),
                           _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_gating")
    return g, beta


def gdn_read_device_status(stream=None, clear: bool = True) -> int:
    return int(load().gdn_read_device_status(_stream(stream), int(clear)))


def gdn_profile_enable(enable: bool = True) -> None:
    load().gdn_profile_enable(int(enable))


def gdn_kernel_name(kernel: int) -> str:
    return load().gdn_kernel_name(int(kernel)).decode()


def gdn_profile_collect(reset: bool = True) -> dict:
    """{kernel name: (launches, summed event ms, timed launches)} for kernels that ran."""
    n = GDN_K_COUNT
    launches = (ctypes.c_longlong * n)()
    ms = (ctypes.c_double * n)()
    timed = (ctypes.c_longlong * n)()
    st = load().gdn_profile_collect(ctypes.cast(launches, _vp), ctypes.cast(ms, _vp), ctypes.cast(timed, _vp), n,
                                    int(reset))
    if st != GDN_OK:
        raise GdnError(st, "gdn_profile_collect")
    return {gdn_kernel_name(i): (int(launches[i]), float(ms[i]), int(timed[i])) for i in range(n) if launches[i]}
