"""Host-side checks of libgdn.so that need no GPU.

* The library builds, loads and exports every function include/gdn.h declares.
* Argument checks reject bad problems before any CUDA call (so they can be
  exercised on a machine without a GPU): wrong head counts, unsupported head
  dims, bad dtype, flags, misaligned pointers, short workspace.
* The workspace size query depends only on the problem descriptor.
"""
import ctypes
import os
import re

import pytest

from gated_deltanet_chunked_gb300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_symbols():
    assert set(header_functions()) == set(gdn.SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = gdn.load()
    for name in header_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings():
    assert gdn.gdn_version() >= 100
    for s in range(7):
        assert gdn.gdn_status_string(s).startswith("GDN_")
    assert "unknown" in gdn.gdn_status_string(99)


def problem(**kw):
    base = dict(batch=1, seqlen=256, num_seqs=1, total_tokens=256, hq=16, hv=32, dk=128, dv=128,
                io_dtype=gdn.GDN_DT_BF16, flags=0, num_state_slots=0)
    base.update(kw)
    return gdn.GdnProblem(**base)


FAKE = 1 << 20  # a 16-byte aligned non-null address: never dereferenced by the checks


def call_fwd(p, ws_bytes=1 << 40, ptr=FAKE, ws=FAKE << 8, cu=None):
    lib = gdn.load()
    P = ctypes.c_void_p
    return lib.gdn_chunk_fwd(ctypes.byref(p), P(ptr), P(ptr), P(ptr), P(ptr), P(ptr), ctypes.c_float(0.1), None,
                             None if cu is None else P(cu), P(ptr), None, P(ws), ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("kw,code", [
    (dict(hv=33), gdn.GDN_EINVAL),           # hv % hq != 0
    (dict(hq=0), gdn.GDN_EINVAL),
    (dict(dk=64, dv=64), gdn.GDN_EUNSUPPORTED),
    (dict(dk=0), gdn.GDN_EINVAL),
    (dict(io_dtype=7), gdn.GDN_EINVAL),
    (dict(flags=1), gdn.GDN_EUNSUPPORTED),
    (dict(total_tokens=255), gdn.GDN_EINVAL),  # dense: B*T != total
    (dict(num_seqs=2), gdn.GDN_EINVAL),        # dense: num_seqs != batch
    (dict(num_seqs=0), gdn.GDN_EINVAL),
])
def test_chunk_fwd_rejects_bad_problems(kw, code):
    assert call_fwd(problem(**kw)) == code


def test_chunk_fwd_rejects_bad_pointers_and_workspace():
    p = problem()
    need = gdn.gdn_chunk_fwd_workspace_size(p)
    assert need > 0
    assert call_fwd(p, ptr=FAKE + 4) == gdn.GDN_EINVAL           # misaligned tensor
    assert call_fwd(p, ptr=0) == gdn.GDN_EINVAL                  # NULL tensor
    assert call_fwd(p, ws_bytes=need - 1) == gdn.GDN_EINVAL      # short workspace
    assert call_fwd(p, ws=(FAKE << 8) + 16) == gdn.GDN_EINVAL    # workspace not 256-aligned
    assert call_fwd(p, cu=FAKE + 8) == gdn.GDN_EINVAL            # misaligned cu_seqlens


def test_workspace_size_query():
    p = problem()
    a = gdn.gdn_chunk_fwd_workspace_size(p)
    b = gdn.gdn_chunk_fwd_workspace_size(problem(batch=1, seqlen=0, num_seqs=1))  # packed descriptor
    assert a == b > 0
    assert gdn.gdn_chunk_fwd_workspace_size(problem(hv=33)) == 0
    # grows with tokens and with sequences (chunk upper bound T/64 + N)
    assert gdn.gdn_chunk_fwd_workspace_size(problem(seqlen=0, total_tokens=4096)) > a
    assert (gdn.gdn_chunk_fwd_workspace_size(problem(seqlen=0, num_seqs=8)) >
            gdn.gdn_chunk_fwd_workspace_size(problem(seqlen=0, num_seqs=1)))


def test_recurrent_step_rejects_bad_problems():
    lib = gdn.load()
    P = ctypes.c_void_p

    def step(p, idx=None, ptr=FAKE):
        return lib.gdn_recurrent_step(ctypes.byref(p), P(ptr), P(ptr), P(ptr), P(ptr), P(ptr), ctypes.c_float(1.0),
                                      P(ptr), None if idx is None else P(idx), P(ptr), None)

    ok = dict(batch=4, seqlen=1, num_seqs=4, total_tokens=4, num_state_slots=4)
    assert step(problem(**{**ok, "num_state_slots": 3})) == gdn.GDN_EINVAL  # identity map needs N slots
    assert step(problem(**{**ok, "total_tokens": 5})) == gdn.GDN_EINVAL
    assert step(problem(**{**ok, "dk": 96})) == gdn.GDN_EUNSUPPORTED
    assert step(problem(**{**ok, "flags": 16})) == gdn.GDN_EUNSUPPORTED
    assert step(problem(**ok), ptr=FAKE + 2) == gdn.GDN_EINVAL
    assert step(problem(**ok), idx=FAKE + 4) == gdn.GDN_EINVAL



def test_recurrent_step_gated_rejects_bad_problems():
    lib = gdn.load()
    P = ctypes.c_void_p

    def step(p, idx=None, ptr=FAKE, gate=FAKE, b=FAKE, z=None, w=FAKE, eps=1e-6):
        return lib.gdn_recurrent_step_gated(ctypes.byref(p), P(ptr), P(ptr), P(ptr), P(gate), P(b), P(gate),
                                            P(gate), ctypes.c_float(1.0), P(ptr), None if idx is None else P(idx),
                                            None if z is None else P(z), P(w), ctypes.c_float(eps), P(ptr), None)

    ok = dict(batch=4, seqlen=1, num_seqs=4, total_tokens=4, num_state_slots=4)
    assert step(problem(**{**ok, "num_state_slots": 3})) == gdn.GDN_EINVAL
    assert step(problem(**{**ok, "total_tokens": 5})) == gdn.GDN_EINVAL
    assert step(problem(**{**ok, "dv": 64})) == gdn.GDN_EUNSUPPORTED
    assert step(problem(**{**ok, "flags": 1})) == gdn.GDN_EUNSUPPORTED  # bit 0 is no decode option
    assert step(problem(**{**ok, "flags": 8})) == gdn.GDN_EUNSUPPORTED
    assert step(problem(**ok), ptr=FAKE + 4) == gdn.GDN_EINVAL  # tensors want 16-byte alignment
    assert step(problem(**ok), gate=FAKE + 2) == gdn.GDN_EINVAL  # gate inputs want 4-byte alignment
    assert step(problem(**ok), b=0) == gdn.GDN_EINVAL
    assert step(problem(**ok), idx=FAKE + 4) == gdn.GDN_EINVAL
    assert step(problem(**ok), z=FAKE, w=0) == gdn.GDN_EINVAL        # output gate without its weight
    assert step(problem(**ok), z=FAKE + 2) == gdn.GDN_EINVAL         # misaligned z
    assert step(problem(**ok), z=FAKE, w=FAKE + 4) == gdn.GDN_EINVAL
    assert step(problem(**ok), z=FAKE, eps=-1.0) == gdn.GDN_EINVAL
    assert step(problem(**ok), z=FAKE, eps=float("nan")) == gdn.GDN_EINVAL


def test_gated_rmsnorm_rejects_bad_arguments():
    lib = gdn.load()
    P = ctypes.c_void_p

    def norm(p, o=FAKE, z=FAKE, w=FAKE, y=FAKE, eps=1e-6):
        return lib.gdn_gated_rmsnorm(ctypes.byref(p), P(o), P(z), P(w), ctypes.c_float(eps), P(y), None)

    ok = dict(total_tokens=64)
    assert norm(problem(**{**ok, "dv": 64})) == gdn.GDN_EUNSUPPORTED
    assert norm(problem(**{**ok, "hv": 0})) == gdn.GDN_EINVAL
    assert norm(problem(**{**ok, "io_dtype": 5})) == gdn.GDN_EINVAL
    assert norm(problem(**ok), z=0) == gdn.GDN_EINVAL
    assert norm(problem(**ok), y=FAKE + 8) == gdn.GDN_EINVAL
    assert norm(problem(**ok), w=FAKE + 4) == gdn.GDN_EINVAL
    assert norm(problem(**ok), eps=-1e-3) == gdn.GDN_EINVAL


def test_conv_and_gating_reject_bad_arguments():
    lib = gdn.load()
    P = ctypes.c_void_p

    def conv(p, x=FAKE, w=FAKE, b=None, st=None, idx=None, cu=FAKE, out=FAKE):
        return lib.gdn_causal_conv1d_silu(ctypes.byref(p), P(x), P(w), None if b is None else P(b),
                                          None if st is None else P(st), None if idx is None else P(idx),
                                          None if cu is None else P(cu), 0, P(out), P(out), P(out), None)

    ok = dict(batch=1, seqlen=0, num_seqs=2, total_tokens=64, hq=1, hv=2, num_state_slots=2)
    assert conv(problem(**{**ok, "dk": 64, "dv": 64})) == gdn.GDN_EUNSUPPORTED
    assert conv(problem(**{**ok, "num_seqs": 0})) == gdn.GDN_EINVAL
    assert conv(problem(**ok), cu=None) == gdn.GDN_EINVAL            # two sequences need offsets
    assert conv(problem(**{**ok, "num_state_slots": 1}), st=FAKE) == gdn.GDN_EINVAL  # identity slots
    assert conv(problem(**ok), w=0) == gdn.GDN_EINVAL
    assert conv(problem(**ok), w=FAKE + 4) == gdn.GDN_EINVAL
    assert conv(problem(**ok), b=FAKE + 8) == gdn.GDN_EINVAL
    assert conv(problem(**ok), x=FAKE + 2) == gdn.GDN_EINVAL
    assert conv(problem(**ok), cu=FAKE + 2) == gdn.GDN_EINVAL

    def gating(p, a=FAKE, g=FAKE):
        return lib.gdn_gating(ctypes.byref(p), P(a), P(a), P(a), P(a), P(g), P(g), None)

    assert gating(problem(hv=0)) == gdn.GDN_EINVAL
    assert gating(problem(), a=0) == gdn.GDN_EINVAL
    assert gating(problem(), g=FAKE + 2) == gdn.GDN_EINVAL


def test_binding_rejects_wrong_dtypes():
    """The binding checks dtypes before any call (no GPU needed)."""
    import torch

    bf = torch.bfloat16
    q = torch.zeros((2, 1, 128), dtype=bf)
    v = torch.zeros((2, 2, 128), dtype=bf)
    g = torch.zeros((2, 2))
    with pytest.raises(ValueError):
        gdn.gdn_recurrent_step(q, q, v, g, g.double(), 0.1, torch.zeros((2, 2, 128, 128)))
    with pytest.raises(ValueError):
        gdn.gdn_recurrent_step(q, q, v, g, g, 0.1, torch.zeros((2, 2, 128, 128), dtype=torch.float16))
    with pytest.raises(ValueError):
        gdn.gdn_chunk_fwd(q, q, v.float(), g, g, 0.1)
    with pytest.raises(ValueError):
        gdn.gdn_gated_rmsnorm(v, v.float(), torch.ones(128), 1e-6)
    with pytest.raises(ValueError):
        gdn.gdn_causal_conv1d_silu(torch.zeros((2, 512), dtype=bf), torch.zeros((512, 4), dtype=bf), 1, 2)
    with pytest.raises(ValueError):
        gdn.gdn_gating(g, g, torch.zeros(2, dtype=torch.float64), torch.zeros(2))


def test_binding_rejects_wrong_shapes_before_any_call():
    """Shapes are checked against the problem descriptor in the binding: a
    wrong final_state, state or gate shape never reaches the library (where it
    would be an out-of-bounds write)."""
    import torch

    bf = torch.bfloat16
    T, hq, hv = 70, 1, 2
    q = torch.zeros((T, hq, 128), dtype=bf)
    v = torch.zeros((T, hv, 128), dtype=bf)
    g = torch.zeros((T, hv))
    cu = torch.tensor([0, T], dtype=torch.int32)
    with pytest.raises(ValueError, match="final_state"):
        gdn.gdn_chunk_fwd(q, q, v, g, g, 0.1, cu_seqlens=cu, final_state=torch.zeros((1, hv, 128, 64)))
    with pytest.raises(ValueError, match="initial_state"):
        gdn.gdn_chunk_fwd(q, q, v, g, g, 0.1, cu_seqlens=cu, initial_state=torch.zeros((2, hv, 128, 128)))
    with pytest.raises(ValueError, match="beta"):
        gdn.gdn_chunk_fwd(q, q, v, g, g[:, :1].contiguous(), 0.1, cu_seqlens=cu)
    with pytest.raises(ValueError, match="out"):
        gdn.gdn_chunk_fwd(q, q, v, g, g, 0.1, cu_seqlens=cu, out=torch.zeros((T, hv, 64), dtype=bf))
    with pytest.raises(ValueError, match="state"):
        gdn.gdn_recurrent_step(q[:4], q[:4], v[:4], g[:4], g[:4], 0.1, torch.zeros((4, hv, 128, 64)))
    with pytest.raises(ValueError, match="state_indices"):
        gdn.gdn_recurrent_step(q[:4], q[:4], v[:4], g[:4], g[:4], 0.1, torch.zeros((4, hv, 128, 128)),
                               state_indices=torch.zeros(3, dtype=torch.int32))
    with pytest.raises(ValueError, match="weight"):
        gdn.gdn_gated_rmsnorm(v, v, torch.ones(64), 1e-6)


def test_binding_rejects_host_tensors():
    """Correctly shaped tensors that are not on a CUDA device are refused in
    the binding (the kernels would dereference their host addresses)."""
    import torch

    bf = torch.bfloat16
    T, hq, hv = 70, 1, 2
    q = torch.zeros((T, hq, 128), dtype=bf)
    v = torch.zeros((T, hv, 128), dtype=bf)
    g = torch.zeros((T, hv))
    with pytest.raises(ValueError, match="CUDA"):
        gdn.gdn_chunk_fwd(q, q, v, g, g, 0.1, cu_seqlens=torch.tensor([0, T], dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        gdn.gdn_recurrent_step(q[:4], q[:4], v[:4], g[:4], g[:4], 0.1, torch.zeros((4, hv, 128, 128)))
    with pytest.raises(ValueError, match="CUDA"):
        gdn.gdn_gated_rmsnorm(v, v, torch.ones(128), 1e-6)


def test_boundary_names_of_the_specification():
    """The boundary's specified names resolve in the library: the two prefill
    entry points, the workspace query, the decode step, the status word
    (gdn_get_device_status) and the status strings."""
    lib = gdn.load()
    for name in ("gdn_chunk_fwd", "gdn_chunk_fwd_workspace_size", "gdn_recurrent_step", "gdn_get_device_status",
                 "gdn_status_string"):
        assert hasattr(lib, name), name
