"""Parity of gdn_gated_rmsnorm (CUDA, through the C ABI) with the oracle's
head-wise gated RMSNorm, stand-alone and after a prefill.

Covers both io dtypes, a row count that leaves a ragged last block, the
in-place form (y = o), zero rows (y = 0 through eps), saturated gates, the
T=4096 x 32-head tensor of the prefill workload, and prefill followed by the
output gate against the oracle's chunk form followed by its gated RMSNorm.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, oracle_prefill, run_gpu_prefill

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
