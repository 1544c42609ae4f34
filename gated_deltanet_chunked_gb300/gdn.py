"""Thin ctypes binding of libgdn.so (include/gdn.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. There is
no fallback: if libgdn.so cannot be built or loaded, ``load()`` raises.

The entry points keep the C names:
  gdn_chunk_fwd, gdn_chunk_fwd_workspace_size, gdn_recurrent_step,
  gdn_recurrent_step_gated, gdn_gated_rmsnorm, gdn_causal_conv1d_silu,
  gdn_causal_conv1d_silu_step, gdn_gating,
  gdn_read_device_status, gdn_get_device_status, gdn_status_string, gdn_version.
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
           "gdn_gating", "gdn_causal_conv1d_silu_step", "gdn_chunk_fwd_gated", "gdn_get_device_status",
           "gdn_set_wait_limit_ns")
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
            lib.gdn_get_device_status.argtypes = [_vp]
            lib.gdn_get_device_status.restype = ctypes.c_int
            lib.gdn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
            lib.gdn_set_wait_limit_ns.restype = ctypes.c_int
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


def _stream(stream, device=None) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _on_device(dev: torch.device, **tensors):
    """Raises ValueError unless every given (non-None) tensor is a CUDA tensor
    on ``dev``. The library reads its device status word and its no-alloc
    scratch on the current device, and the kernels dereference the pointers
    they are given, so a host tensor or a tensor on another GPU must never
    reach it."""
    if dev.type != "cuda":
        raise ValueError(f"libgdn wants CUDA tensors, got a tensor on {dev}")
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, expected {dev} (the device of the first input)")


def _shape(name, t, *shape):
    """Raises ValueError unless tensor ``t`` (if given) has exactly ``shape``."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


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


def _prefill_checks(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, z=None, norm_weight=None,
                    workspace=None):
    """Device, dtype and shape checks shared by the prefill wrappers; returns
    (problem, device)."""
    packed = cu_seqlens is not None
    if q.dim() != (3 if packed else 4):
        raise ValueError("q must be [T, Hq, dk] with cu_seqlens, else [B, T, Hq, dk]")
    num_seqs = cu_seqlens.numel() - 1 if packed else q.shape[0]
    dev = q.device
    _want(q.dtype, k=k, v=v, out=out, z=z)
    _want(torch.float32, g=g, beta=beta, initial_state=initial_state, final_state=final_state,
          norm_weight=norm_weight)
    _want(torch.int32, cu_seqlens=cu_seqlens)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")
    prob = prefill_problem(q, v, num_seqs, packed)
    lead = q.shape[:-2]  # (T,) packed or (B, T) dense
    _shape("k", k, *q.shape)
    _shape("v", v, *lead, prob.hv, prob.dv)
    _shape("g", g, *lead, prob.hv)
    _shape("beta", beta, *lead, prob.hv)
    _shape("out", out, *v.shape)
    _shape("z", z, *v.shape)
    _shape("norm_weight", norm_weight, prob.dv)
    _shape("initial_state", initial_state, prob.num_seqs, prob.hv, prob.dk, prob.dv)
    _shape("final_state", final_state, prob.num_seqs, prob.hv, prob.dk, prob.dv)
    if packed and cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor [N + 1]")
    _on_device(dev, k=k, v=v, g=g, beta=beta, initial_state=initial_state, cu_seqlens=cu_seqlens, out=out,
               final_state=final_state, z=z, norm_weight=norm_weight, workspace=workspace)
    return prob, dev


def gdn_chunk_fwd(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None, out=None,
                  final_state=None, output_final_state=True, workspace=None, stream=None,
                  z=None, norm_weight=None, norm_eps=1e-6):
    """Chunked prefill. Packed when ``cu_seqlens`` (int32 device [N+1]) is given.

    Returns (out, final_state). ``workspace`` (uint8 device tensor) is
    allocated with PyTorch when not supplied. With ``z`` (like v) and
    ``norm_weight`` [128] f32, out holds the output gate applied to the
    read-out (gdn_chunk_fwd_gated). Every tensor must sit on q's device; the
    call runs with that device current, on its current stream unless
    ``stream`` is given.
    """
    prob, dev = _prefill_checks(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, z, norm_weight,
                                workspace)
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty(v.shape, dtype=v.dtype, device=dev)
        if final_state is None and output_final_state:
            final_state = torch.empty((prob.num_seqs, prob.hv, prob.dk, prob.dv), dtype=torch.float32, device=dev)
        need = gdn_chunk_fwd_workspace_size(prob)
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        if z is None:
            st = load().gdn_chunk_fwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                      ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                      _ptr(final_state), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                      _stream(stream, dev))
            where = "gdn_chunk_fwd"
        else:
            if norm_weight is None:
                raise ValueError("the output gate needs norm_weight")
            st = load().gdn_chunk_fwd_gated(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                            ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(z),
                                            _ptr(norm_weight), ctypes.c_float(norm_eps), _ptr(out),
                                            _ptr(final_state), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                            _stream(stream, dev))
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
    if out is None:
        raise ValueError("gdn_chunk_fwd_noalloc writes into a caller-supplied out")
    prob, dev = _prefill_checks(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state)
    with torch.cuda.device(dev):
        st = load().gdn_chunk_fwd_noalloc(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                          ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out),
                                          _ptr(final_state), _stream(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_chunk_fwd_noalloc")
    return out, final_state


def _decode_flags(state, beta_bf16):
    return (GDN_FLAG_STATE_BF16 if state.dtype == torch.bfloat16 else 0) | (GDN_FLAG_BETA_BF16 if beta_bf16 else 0)


def _decode_checks(q, v, state, state_indices, out, z=None):
    """Shape checks shared by the decode wrappers: q, k [N, Hq, 128],
    v, out, z [N, Hv, 128], state [slots, Hv, 128, 128], state_indices [N]."""
    if q.dim() != 3 or v.dim() != 3 or v.shape[0] != q.shape[0]:
        raise ValueError("q must be [N, Hq, dk] and v [N, Hv, dv] with the same N")
    if state.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"state must be float32 or bfloat16, got {state.dtype}")
    N, hv, dv = v.shape
    if state.dim() != 4 or tuple(state.shape[1:]) != (hv, q.shape[2], dv):
        raise ValueError(f"state must be [slots, {hv}, {q.shape[2]}, {dv}], got {tuple(state.shape)}")
    _shape("out", out, *v.shape)
    _shape("z", z, *v.shape)
    _shape("state_indices", state_indices, N)


def gdn_recurrent_step(q, k, v, g, beta, scale, state, state_indices=None, out=None, stream=None,
                       beta_bf16=False):
    """One decode step; ``state`` [slots, Hv, 128, 128] (f32, or bf16 for a
    bf16 state cache) is updated in place. ``beta_bf16`` rounds beta to bf16."""
    dev = q.device
    _want(q.dtype, k=k, v=v, out=out)
    _want(torch.float32, g=g, beta=beta)
    _want(torch.int32, state_indices=state_indices)
    _decode_checks(q, v, state, state_indices, out)
    N, hq, dk = q.shape
    _shape("k", k, *q.shape)
    _shape("g", g, N, v.shape[1])
    _shape("beta", beta, N, v.shape[1])
    _on_device(dev, k=k, v=v, g=g, beta=beta, state=state, state_indices=state_indices, out=out)
    prob = GdnProblem(N, 1, N, N, hq, v.shape[1], dk, v.shape[2], _io_dtype(q), _decode_flags(state, beta_bf16),
                      state.shape[0])
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty(v.shape, dtype=v.dtype, device=dev)
        st = load().gdn_recurrent_step(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                       ctypes.c_float(scale), _ptr(state), _ptr(state_indices), _ptr(out),
                                       _stream(stream, dev))
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
    dev = q.device
    _want(q.dtype, k=k, v=v, out=out, z=z)
    _want(torch.float32, a=a, b=b, A_log=A_log, dt_bias=dt_bias, norm_weight=norm_weight)
    _want(torch.int32, state_indices=state_indices)
    _decode_checks(q, v, state, state_indices, out, z)
    N, hq, dk = q.shape
    hv = v.shape[1]
    _shape("k", k, *q.shape)
    _shape("a", a, N, hv)
    _shape("b", b, N, hv)
    _shape("A_log", A_log, hv)
    _shape("dt_bias", dt_bias, hv)
    _shape("norm_weight", norm_weight, v.shape[2])
    if z is not None and norm_weight is None:
        raise ValueError("the output gate needs norm_weight")
    _on_device(dev, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, state=state, state_indices=state_indices,
               out=out, z=z, norm_weight=norm_weight)
    prob = GdnProblem(N, 1, N, N, hq, hv, dk, v.shape[2], _io_dtype(q), _decode_flags(state, beta_bf16),
                      state.shape[0])
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty(v.shape, dtype=v.dtype, device=dev)
        st = load().gdn_recurrent_step_gated(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                             _ptr(A_log), _ptr(dt_bias), ctypes.c_float(scale), _ptr(state),
                                             _ptr(state_indices), _ptr(z), _ptr(norm_weight),
                                             ctypes.c_float(norm_eps), _ptr(out), _stream(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_recurrent_step_gated")
    return out


def gdn_gated_rmsnorm(o, z, weight, eps, out=None, stream=None):
    """y = o / sqrt(mean(o^2) + eps) * weight * silu(z) per (token, head) row
    of o, z [T, Hv, 128] (io dtype) with weight [128] f32. ``out`` may be o."""
    dev = o.device
    if o.dim() != 3:
        raise ValueError("o must be [T, Hv, 128]")
    T, hv, dv = o.shape
    _want(o.dtype, z=z, out=out)
    _want(torch.float32, weight=weight)
    _shape("z", z, *o.shape)
    _shape("out", out, *o.shape)
    _shape("weight", weight, dv)
    _on_device(dev, z=z, weight=weight, out=out)
    prob = GdnProblem(1, 0, 1, T, 1, hv, dv, dv, _io_dtype(o), 0, 0)
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty_like(o)
        st = load().gdn_gated_rmsnorm(ctypes.byref(prob), _ptr(o), _ptr(z), _ptr(weight), ctypes.c_float(eps),
                                      _ptr(out), _stream(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_gated_rmsnorm")
    return out


def _conv_checks(x, weight, bias, conv_state, state_indices, cu_seqlens, q, k, v, hq, hv, N):
    dev = x.device
    if x.dim() != 2:
        raise ValueError("x must be [T, C]")
    T, C = x.shape
    if C != (2 * hq + hv) * 128:
        raise ValueError("x must have (2 hq + hv) * 128 channels")
    _want(x.dtype, conv_state=conv_state, q=q, k=k, v=v)
    _want(torch.float32, weight=weight, bias=bias)
    _want(torch.int32, state_indices=state_indices, cu_seqlens=cu_seqlens)
    _shape("weight", weight, C, 4)
    _shape("bias", bias, C)
    _shape("state_indices", state_indices, N)
    _shape("cu_seqlens", cu_seqlens, N + 1)
    _shape("q", q, T, hq, 128)
    _shape("k", k, T, hq, 128)
    _shape("v", v, T, hv, 128)
    if conv_state is not None and (conv_state.dim() != 3 or tuple(conv_state.shape[1:]) != (3, C)):
        raise ValueError(f"conv_state must be [slots, 3, {C}], got {tuple(conv_state.shape)}")
    _on_device(dev, weight=weight, bias=bias, conv_state=conv_state, state_indices=state_indices,
               cu_seqlens=cu_seqlens, q=q, k=k, v=v)
    return dev


def gdn_causal_conv1d_silu(x, weight, hq, hv, bias=None, conv_state=None, state_indices=None, cu_seqlens=None,
                           norm_qk=False, q=None, k=None, v=None, stream=None):
    """Short causal convolution (4 taps, weight [C, 4] f32 oldest first) + SiLU
    over packed tokens x [T, C] (C = (2 hq + hv) * 128), split into q, k
    [T, hq, 128] and v [T, hv, 128]; ``conv_state`` [slots, 3, C] is read and
    updated in place. ``norm_qk`` L2-normalises every q and k head row."""
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = _conv_checks(x, weight, bias, conv_state, state_indices, cu_seqlens, q, k, v, hq, hv, N)
    T = x.shape[0]
    slots = 0 if conv_state is None else conv_state.shape[0]
    prob = GdnProblem(1, 0, N, T, hq, hv, 128, 128, _io_dtype(x), 0, slots)
    with torch.cuda.device(dev):
        q = torch.empty((T, hq, 128), dtype=x.dtype, device=dev) if q is None else q
        k = torch.empty((T, hq, 128), dtype=x.dtype, device=dev) if k is None else k
        v = torch.empty((T, hv, 128), dtype=x.dtype, device=dev) if v is None else v
        st = load().gdn_causal_conv1d_silu(ctypes.byref(prob), _ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state),
                                           _ptr(state_indices), _ptr(cu_seqlens), int(bool(norm_qk)), _ptr(q),
                                           _ptr(k), _ptr(v), _stream(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_causal_conv1d_silu")
    return q, k, v


def gdn_causal_conv1d_silu_step(x, weight, hq, hv, bias=None, conv_state=None, state_indices=None, norm_qk=False,
                                q=None, k=None, v=None, stream=None):
    """gdn_causal_conv1d_silu for one token per sequence: x [N, C]."""
    N = x.shape[0]
    dev = _conv_checks(x, weight, bias, conv_state, state_indices, None, q, k, v, hq, hv, N)
    slots = 0 if conv_state is None else conv_state.shape[0]
    prob = GdnProblem(N, 1, N, N, hq, hv, 128, 128, _io_dtype(x), 0, slots)
    with torch.cuda.device(dev):
        q = torch.empty((N, hq, 128), dtype=x.dtype, device=dev) if q is None else q
        k = torch.empty((N, hq, 128), dtype=x.dtype, device=dev) if k is None else k
        v = torch.empty((N, hv, 128), dtype=x.dtype, device=dev) if v is None else v
        st = load().gdn_causal_conv1d_silu_step(ctypes.byref(prob), _ptr(x), _ptr(weight), _ptr(bias),
                                                _ptr(conv_state), _ptr(state_indices), int(bool(norm_qk)), _ptr(q),
                                                _ptr(k), _ptr(v), _stream(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_causal_conv1d_silu_step")
    return q, k, v


def gdn_gating(a, b, A_log, dt_bias, g=None, beta=None, stream=None):
    """g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b), a, b [T, Hv] f32."""
    dev = a.device
    if a.dim() != 2:
        raise ValueError("a must be [T, Hv]")
    T, hv = a.shape
    _want(torch.float32, a=a, b=b, A_log=A_log, dt_bias=dt_bias, g=g, beta=beta)
    for name, t in (("b", b), ("g", g), ("beta", beta)):
        _shape(name, t, T, hv)
    _shape("A_log", A_log, hv)
    _shape("dt_bias", dt_bias, hv)
    _on_device(dev, b=b, A_log=A_log, dt_bias=dt_bias, g=g, beta=beta)
    prob = GdnProblem(1, 0, 1, T, 1, hv, 128, 128, GDN_DT_F32, 0, 0)
    with torch.cuda.device(dev):
        g = torch.empty_like(a) if g is None else g
        beta = torch.empty_like(a) if beta is None else beta
        st = load().gdn_gating(ctypes.byref(prob), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(g),
                               _ptr(beta), _stream(stream, dev))
    if st != GDN_OK:
        raise GdnError(st, "gdn_gating")
    return g, beta


def gdn_read_device_status(stream=None, clear: bool = True) -> int:
    """Synchronises ``stream`` (the current device's current stream when
    None) and returns the device status word, clearing it when ``clear``."""
    return int(load().gdn_read_device_status(_stream(stream), int(clear)))


def gdn_get_device_status(stream=None) -> int:
    """gdn_read_device_status with clear: returns the first device-side error
    recorded since the last read and resets the word (cudaGetLastError-like)."""
    return int(load().gdn_get_device_status(_stream(stream)))


def gdn_set_wait_limit_ns(ns: int) -> None:
    """Limit of the prefill kernels' bounded device-side waits for later
    launches (0 restores the default 2 s); for tests of the timeout path."""
    load().gdn_set_wait_limit_ns(int(ns))


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
