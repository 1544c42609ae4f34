"""Degenerate sizes on the GPU: every entry point with no tokens or no
sequences returns GDN_OK, launches nothing that writes, and leaves its
outputs untouched; zero-length sequences inside a packed batch keep their
states (prefill and convolution)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check

pytestmark = pytest.mark.gpu


def test_decode_entry_points_with_no_sequences(cuda):
    bf = torch.bfloat16
    q = torch.empty((0, 2, 128), dtype=bf, device=cuda)
    v = torch.empty((0, 4, 128), dtype=bf, device=cuda)
    g = torch.empty((0, 4), device=cuda)
    state = torch.randn((3, 4, 128, 128), device=cuda)
    before = state.clone()
    gdn.gdn_recurrent_step(q, q, v, g, g, 0.1, state)
    A_log, dt_bias = torch.zeros(4, device=cuda), torch.zeros(4, device=cuda)
    gdn.gdn_recurrent_step_gated(q, q, v, g, g, A_log, dt_bias, 0.1, state)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    assert torch.equal(state, before)


def test_front_end_entry_points_with_no_tokens(cuda):
    bf = torch.bfloat16
    x = torch.empty((0, 1024), dtype=bf, device=cuda)
    w = torch.zeros((1024, 4), device=cuda)
    cst = torch.randn((2, 3, 1024), device=cuda).to(bf)
    before = cst.clone()
    gdn.gdn_causal_conv1d_silu_step(x, w, 2, 4, conv_state=cst)
    gdn.gdn_causal_conv1d_silu(x, w, 2, 4, conv_state=cst, cu_seqlens=torch.zeros(2, dtype=torch.int32, device=cuda))
    g, beta = gdn.gdn_gating(torch.empty((0, 4), device=cuda), torch.empty((0, 4), device=cuda),
                             torch.zeros(4, device=cuda), torch.zeros(4, device=cuda))
    o = torch.empty((0, 4, 128), dtype=bf, device=cuda)
    y = gdn.gdn_gated_rmsnorm(o, o, torch.ones(128, device=cuda), 1e-6)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    assert torch.equal(cst, before) and y.numel() == 0 and g.numel() == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_all_sequences_empty(cuda, dtype):
    """Packed batch of three empty sequences: no tokens, final state = S0."""
    hq, hv = 1, 2
    q = torch.empty((0, hq, 128), dtype=dtype, device=cuda)
    v = torch.empty((0, hv, 128), dtype=dtype, device=cuda)
    g = torch.empty((0, hv), device=cuda)
    S0 = torch.randn((3, hv, 128, 128), device=cuda)
    cu = torch.zeros(4, dtype=torch.int32, device=cuda)
    o, S = gdn.gdn_chunk_fwd(q, q, v, g, g, 0.1, initial_state=S0, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    assert o.numel() == 0 and torch.equal(S, S0)


def test_conv_empty_sequences_between_others(cuda):
    """Zero-length sequences in a packed batch keep their conv state."""
    hq, hv = 1, 2
    lengths = [0, 5, 0, 0, 2, 0]
    T = sum(lengths)
    x, w, b, st0 = W.make_conv_inputs(90, T, hq, hv, torch.float32, slots=6)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    st = st0.to(cuda)
    q, k, v = gdn.gdn_causal_conv1d_silu(x.to(cuda), w.to(cuda), hq, hv, bias=b.to(cuda), conv_state=st,
                                         cu_seqlens=cu.to(cuda))
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    y_ref, st_ref = oracle.causal_conv1d_silu(x, w, b, st0, cu)
    check(torch.cat([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], 1), y_ref, torch.float32, "y")
    check(st, st_ref, torch.float32, "conv state")
    assert torch.equal(st[[0, 2, 3, 5]], st0[[0, 2, 3, 5]].to(cuda))
