"""gdn_chunk_fwd_noalloc: the prefill entry point for callers that cannot allocate.

Callers that may not call cudaMalloc (allocator hooks, host callbacks,
runtimes that freeze their memory footprint after start-up) cannot provide
a workspace; this entry point runs the same forward on the library's fixed
device scratch array instead. The GPU tests call it through the C ABI twice
in a row, on two different problems: the same kernels run on the same inputs
as the regular gdn_chunk_fwd (which uses a caller workspace) and the path is
deterministic, so the results must be bit-identical to it; each call is also
checked against the CPU oracle. A problem just under the scratch size runs,
one just over it is refused. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, oracle_prefill


def _call_noalloc(d, out, fin):
    lib = gdn.load()
    prob = gdn.prefill_problem(d["q"], d["v"], d["cu_seqlens"].numel() - 1, packed=True)
    P = ctypes.c_void_p
    ptr = lambda t: None if t is None else P(t.data_ptr())
    return lib.gdn_chunk_fwd_noalloc(ctypes.byref(prob), ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]),
                                     ptr(d["beta"]), ctypes.c_float(d["scale"]), ptr(d["initial_state"]),
                                     ptr(d["cu_seqlens"]), ptr(out), ptr(fin),
                                     P(torch.cuda.current_stream().cuda_stream))


def _largest_tokens(hq, hv, io_dtype):
    """Largest single-sequence token count whose workspace fits the scratch."""
    lo, hi = 0, 1 << 20
    while lo < hi:
        m = (lo + hi + 1) // 2
        need = gdn.gdn_chunk_fwd_workspace_size(gdn.GdnProblem(1, 0, 1, m, hq, hv, 128, 128, io_dtype, 0, 0))
        lo, hi = (m, hi) if need <= gdn.GDN_NOALLOC_SCRATCH_BYTES else (lo, m - 1)
    return lo


def _run_and_compare(inp, cuda):
    d = {k: (v.to(cuda) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty_like(d["v"])
    fin = torch.empty((d["cu_seqlens"].numel() - 1, d["v"].shape[1], 128, 128), device=cuda)
    assert _call_noalloc(d, out, fin) == gdn.GDN_OK
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    o_ws, S_ws = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                   initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(out, o_ws), "noalloc o differs from gdn_chunk_fwd"
    assert torch.equal(fin, S_ws), "noalloc final_state differs from gdn_chunk_fwd"
    o_ref, S_ref = oracle_prefill(inp)
    check(out, o_ref, inp["q"].dtype, "noalloc o")
    check(fin, S_ref, inp["q"].dtype, "noalloc final_state")


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_twice(cuda):
    cases = [
        W.make_custom_prefill(201, [130, 1, 64], 2, 4, torch.bfloat16, s0_sigma=0.05),
        W.make_custom_prefill(202, [77, 200], 1, 2, torch.float32, s0_sigma=0.1),
    ]
    for inp in cases:  # two calls in a row share (and reuse) the scratch array
        _run_and_compare(inp, cuda)


@pytest.mark.gpu
def test_noalloc_largest_problem_that_fits(cuda):
    """The Qwen3.5-style layer shape (hq = 16, hv = 32) at the largest token
    count whose workspace fits the scratch runs and matches."""
    T = _largest_tokens(16, 32, gdn.GDN_DT_BF16)
    assert T > 0
    _run_and_compare(W.make_custom_prefill(203, [T], 16, 32, torch.bfloat16), cuda)


def test_noalloc_rejects_problems_above_the_scratch_size():
    """Checked on the host before any CUDA call, so it also runs without a GPU."""
    lib = gdn.load()
    fake = ctypes.c_void_p(1 << 20)
    for dt in (gdn.GDN_DT_BF16, gdn.GDN_DT_F32):
        T = _largest_tokens(16, 32, dt)
        fits = gdn.GdnProblem(1, 0, 1, T, 16, 32, 128, 128, dt, 0, 0)
        over = gdn.GdnProblem(1, 0, 1, T + 1, 16, 32, 128, 128, dt, 0, 0)
        assert gdn.gdn_chunk_fwd_workspace_size(fits) <= gdn.GDN_NOALLOC_SCRATCH_BYTES
        assert gdn.gdn_chunk_fwd_workspace_size(over) > gdn.GDN_NOALLOC_SCRATCH_BYTES
        st = lib.gdn_chunk_fwd_noalloc(ctypes.byref(over), fake, fake, fake, fake, fake, ctypes.c_float(1.0), None,
                                       fake, fake, None, None)
        assert st == gdn.GDN_ETOOBIG
    big = gdn.GdnProblem(1, 0, 1, 1 << 16, 16, 32, 128, 128, gdn.GDN_DT_BF16, 0, 0)
    st = lib.gdn_chunk_fwd_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, ctypes.c_float(1.0), None, fake,
                                   fake, None, None)
    assert st == gdn.GDN_ETOOBIG
    bad = gdn.GdnProblem(1, 0, 1, 64, 16, 33, 128, 128, gdn.GDN_DT_BF16, 0, 0)  # hv % hq != 0
    st = lib.gdn_chunk_fwd_noalloc(ctypes.byref(bad), fake, fake, fake, fake, fake, ctypes.c_float(1.0), None, fake,
                                   fake, None, None)
    assert st == gdn.GDN_EINVAL
