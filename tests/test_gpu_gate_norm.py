"""Parity of gdn_gated_rmsnorm (CUDA, through the C ABI) with the oracle's
head-wise gated RMSNorm, stand-alone and after a prefill.

Covers both io dtypes, a row count that leaves a ragged last block, the
in-place form (y = o), zero rows (y = 0 through eps), saturated gates, the
T=4096 x 32-head tensor of the prefill workload, prefill followed by the
output gate, and the gate fused into the prefill (gdn_chunk_fwd_gated), each
against the oracle's chunk form followed by its gated RMSNorm.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, head_slice, oracle_prefill, run_gpu_prefill

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gate_norm_small_ragged(cuda, dtype):
    z, w, o = W.make_output_gate(51, 37, 3, dtype, with_o=True)  # 111 rows
    o[5, 1] = 0  # a zero row: y = 0
    z[7, 2, :16] = 40.0  # silu saturates to the identity ...
    z[8, 0, :16] = -40.0  # ... and to zero
    y = gdn.gdn_gated_rmsnorm(o.to(cuda), z.to(cuda), w.to(cuda), EPS)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(o, z, w, EPS)
    check(y, ref, dtype, "y")
    assert torch.all(y[5, 1] == 0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gate_norm_in_place(cuda, dtype):
    z, w, o = W.make_output_gate(52, 300, 4, dtype, with_o=True)
    od = o.to(cuda)
    y = gdn.gdn_gated_rmsnorm(od, z.to(cuda), w.to(cuda), 1e-5, out=od)
    torch.cuda.synchronize()
    assert y.data_ptr() == od.data_ptr()
    check(od, oracle.gated_rmsnorm(o, z, w, 1e-5), dtype, "y in place")


def test_gate_norm_prefill_tensor_size(cuda):
    """The T=4096 x 32-head read-out tensor of the prefill workload (bf16)."""
    w = W.WORKLOADS["prefill_T4096_hq16_hv32"]
    z, weight, o = W.make_output_gate(w.seed, w.seqlen, w.hv, w.io_dtype, with_o=True)
    y = gdn.gdn_gated_rmsnorm(o.to(cuda), z.to(cuda), weight.to(cuda), EPS)
    torch.cuda.synchronize()
    check(y, oracle.gated_rmsnorm(o, z, weight, EPS), torch.bfloat16, "y")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_then_output_gate(cuda, dtype):
    inp = W.make_custom_prefill(53, [150, 64, 9], 2, 4, dtype, s0_sigma=0.05)
    o, _ = run_gpu_prefill(inp, cuda)
    z, weight = W.make_output_gate(53, inp["total_tokens"], 4, dtype)
    y = gdn.gdn_gated_rmsnorm(o, z.to(cuda), weight.to(cuda), EPS)
    torch.cuda.synchronize()
    o_ref, _ = oracle_prefill(inp, routine="chunked")
    check(y, oracle.gated_rmsnorm(o_ref, z, weight, EPS), dtype, "y")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_fused_gated_prefill_packed(cuda, dtype):
    """gdn_chunk_fwd_gated (the gate inside the fused kernel on the bf16 path)
    on packed sequences with an empty and a one-token one, against the
    oracle's chunk form followed by its gated RMSNorm."""
    lengths = [150, 64, 9, 0, 1, 130]
    inp = W.make_custom_prefill(54, lengths, 2, 4, dtype, s0_sigma=0.05)
    z, weight = W.make_output_gate(54, inp["total_tokens"], 4, dtype)
    d = {k: (v.to(cuda) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], initial_state=d["initial_state"],
                             cu_seqlens=d["cu_seqlens"], z=z.to(cuda), norm_weight=weight.to(cuda), norm_eps=EPS)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    o_ref, S_ref = oracle_prefill(inp, routine="chunked")
    check(y, oracle.gated_rmsnorm(o_ref, z, weight, EPS), dtype, "y")
    check(S, S_ref, dtype, "final state")


def test_fused_gated_prefill_full_size(cuda):
    """T=4096, Hq=16, Hv=32 bf16 through gdn_chunk_fwd_gated: two sampled
    q/k head groups against the oracle; the final state is the ungated
    call's, bit for bit."""
    w = W.WORKLOADS["prefill_T4096_hq16_hv32"]
    inp = W.make_prefill(w)
    z, weight = W.make_output_gate(w.seed, w.seqlen, w.hv, w.io_dtype)
    d = {k: (v.to(cuda) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu = torch.tensor([0, w.seqlen], dtype=torch.int32, device=cuda)
    y, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], cu_seqlens=cu, z=z.to(cuda),
                             norm_weight=weight.to(cuda), norm_eps=EPS)
    _, S_plain = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], cu_seqlens=cu)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    assert torch.equal(S, S_plain)
    group = w.hv // w.hq
    for hk in (3, 14):
        sub = head_slice(inp, hk, group)
        o_ref, _ = oracle_prefill(sub, routine="chunked")
        hv = slice(hk * group, (hk + 1) * group)
        check(y[:, hv], oracle.gated_rmsnorm(o_ref, z[:, hv], weight, EPS), torch.bfloat16, f"y heads of k-head {hk}")
