"""gdn_chunk_fwd_noalloc: the prefill entry point for callers that cannot allocate.

Callers that may not call cudaMalloc (allocator hooks, host callbacks,
runtimes that freeze their memory footprint after start-up) cannot provide
a workspace; this entry point runs the same forward on the library's fixed
device scratch array instead. The GPU test calls it through the C ABI twice
in a row, on two different problems, and compares each result with the
regular gdn_chunk_fwd (which uses a caller workspace) within the bf16/f32
tolerances of the parity tests. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check


def _call_noalloc(d, out, fin):
    lib = gdn.load()
    prob = gdn.prefill_problem(d["q"], d["v"], d["cu_seqlens"].numel() - 1, packed=True)
    P = ctypes.c_void_p
    ptr = lambda t: None if t is None else P(t.data_ptr())
    return lib.gdn_chunk_fwd_noalloc(ctypes.byref(prob), ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]),
                                     ptr(d["beta"]), ctypes.c_float(d["scale"]), ptr(d["initial_state"]),
                                     ptr(d["cu_seqlens"]), ptr(out), ptr(fin),
                                     P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_twice(cuda):
    cases = [
        W.make_custom_prefill(201, [130, 1, 64], 2, 4, torch.bfloat16, s0_sigma=0.05),
        W.make_custom_prefill(202, [77, 200], 1, 2, torch.float32, s0_sigma=0.1),
    ]
    for inp in cases:  # two calls in a row share (and reuse) the scratch array
        d = {k: (v.to(cuda) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        out = torch.empty_like(d["v"])
        fin = torch.empty((d["cu_seqlens"].numel() - 1, d["v"].shape[1], 128, 128), device=cuda)
        assert _call_noalloc(d, out, fin) == gdn.GDN_OK
        torch.cuda.synchronize()
        assert gdn.gdn_read_device_status() == gdn.GDN_OK
        o_ref, S_ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                         initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"])
        torch.cuda.synchronize()
        check(out, o_ref.double().cpu().numpy(), inp["q"].dtype, "noalloc o")
        check(fin, S_ref.double().cpu().numpy(), inp["q"].dtype, "noalloc final_state")


def test_noalloc_rejects_problems_above_the_scratch_size():
    """Checked on the host before any CUDA call, so it also runs without a GPU."""
    lib = gdn.load()
    big = gdn.GdnProblem(1, 0, 1, 1 << 16, 16, 32, 128, 128, gdn.GDN_DT_BF16, 0, 0)
    assert gdn.gdn_chunk_fwd_workspace_size(big) > gdn.GDN_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    st = lib.gdn_chunk_fwd_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, ctypes.c_float(1.0), None, fake,
                                   fake, None, None)
    assert st == gdn.GDN_ETOOBIG
    bad = gdn.GdnProblem(1, 0, 1, 64, 16, 33, 128, 128, gdn.GDN_DT_BF16, 0, 0)  # hv % hq != 0
    st = lib.gdn_chunk_fwd_noalloc(ctypes.byref(bad), fake, fake, fake, fake, fake, ctypes.c_float(1.0), None, fake,
                                   fake, None, None)
    assert st == gdn.GDN_EINVAL
