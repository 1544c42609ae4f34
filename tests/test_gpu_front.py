"""Parity of the front-end kernels (CUDA, through the C ABI) with the oracle:
the short causal convolution + SiLU with its state and the q/k/v split
(gdn_causal_conv1d_silu), the gates of every token (gdn_gating), and the
prefill layer core from raw projections to the gated output
(conv -> gating -> chunk form -> output gate).

Convolution cases: packed sequences of lengths 0 to 150 (shorter than the
window, empty, spanning token tiles), slot indices with a padding slot, no
state, the fused q/k norm, 20 chained decode steps of 256 sequences, and one
4096-token sequence of 8192 channels.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, check_f32_state

pytestmark = pytest.mark.gpu


def split_ref(y, hq, hv):
    T = y.shape[0]
    q = y[:, :hq * 128].reshape(T, hq, 128)
    k = y[:, hq * 128:2 * hq * 128].reshape(T, hq, 128)
    v = y[:, 2 * hq * 128:].reshape(T, hv, 128)
    return q, k, v


def run_conv(dev, x, w, b, st, idx, cu, hq, hv, norm=False):
    d = lambda t: None if t is None else t.to(dev)
    out = gdn.gdn_causal_conv1d_silu(d(x), d(w), hq, hv, bias=d(b), conv_state=st, state_indices=d(idx),
                                     cu_seqlens=d(cu), norm_qk=norm)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("norm", [False, True], ids=["raw", "qknorm"])
def test_conv_packed_sequences_with_slots(cuda, dtype, norm):
    lengths = [150, 2, 0, 1, 70, 3, 33]
    hq, hv = 2, 4
    T = sum(lengths)
    x, w, b, st0 = W.make_conv_inputs(61, T, hq, hv, dtype, slots=8)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    idx = torch.tensor([4, 0, 7, -1, 2, 1, 6], dtype=torch.int32)
    st = st0.to(cuda)
    gdn.gdn_read_device_status(clear=True)
    q, k, v = run_conv(cuda, x, w, b, st, idx, cu, hq, hv, norm)
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    y_ref, st_ref = oracle.causal_conv1d_silu(x, w, b, st0, cu, idx)
    q_ref, k_ref, v_ref = split_ref(y_ref, hq, hv)
    if norm:
        q_ref, k_ref = oracle.l2_normalise(q_ref), oracle.l2_normalise(k_ref)
    for name, got, ref in (("q", q, q_ref), ("k", k, k_ref), ("v", v, v_ref)):
        check(got, ref, dtype, name)
    check(st, st_ref, dtype, "conv state")
    assert torch.equal(st[[3, 5]], st0[[3, 5]].to(cuda))  # slots nobody names


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_conv_without_state_one_sequence(cuda, dtype):
    x, w, b, _ = W.make_conv_inputs(62, 300, 1, 2, dtype)
    q, k, v = run_conv(cuda, x, w, None, None, None, None, 1, 2)
    y_ref, _ = oracle.causal_conv1d_silu(x, w)
    for got, ref in zip((q, k, v), split_ref(y_ref, 1, 2)):
        check(got, ref, dtype, "y")


def test_conv_decode_steps_chained(cuda):
    """256 sequences of one token each, 20 steps, state slots permuted."""
    hq, hv, N = 16, 32, 256
    _, w, b, st0 = W.make_conv_inputs(63, 1, hq, hv, torch.bfloat16, slots=N)
    idx = torch.from_numpy(np.random.default_rng(3).permutation(N).astype(np.int32))
    cu = torch.arange(N + 1, dtype=torch.int32)
    st = st0.to(cuda)
    st_ref = st0.double().numpy()
    for step in range(20):
        x, _, _, _ = W.make_conv_inputs(1000 + step, N, hq, hv, torch.bfloat16)
        q, k, v = run_conv(cuda, x, w, b, st, idx, cu, hq, hv)
        y_ref, st_ref = oracle.causal_conv1d_silu(x, w, b, st_ref, cu, idx)
        if step in (0, 19):
            for got, ref in zip((q, k, v), split_ref(y_ref, hq, hv)):
                check(got, ref, torch.bfloat16, f"y step {step}")
    check(st, st_ref, torch.bfloat16, "conv state after 20 steps")


def test_conv_prefill_size(cuda):
    """One 4096-token sequence, Hq = 16, Hv = 32 (8192 channels), bf16, with state."""
    hq, hv = 16, 32
    x, w, b, st0 = W.make_conv_inputs(64, 4096, hq, hv, torch.bfloat16, slots=1)
    st = st0.to(cuda)
    q, k, v = run_conv(cuda, x, w, b, st, None, torch.tensor([0, 4096], dtype=torch.int32), hq, hv, norm=True)
    y_ref, st_ref = oracle.causal_conv1d_silu(x, w, b, st0)
    q_ref, k_ref, v_ref = split_ref(y_ref, hq, hv)
    check(q, oracle.l2_normalise(q_ref), torch.bfloat16, "q")
    check(k, oracle.l2_normalise(k_ref), torch.bfloat16, "k")
    check(v, v_ref, torch.bfloat16, "v")
    check(st, st_ref, torch.bfloat16, "conv state")


def test_conv_bad_offsets_report_status(cuda):
    x, w, b, _ = W.make_conv_inputs(65, 10, 1, 2, torch.float32)
    cu = torch.tensor([0, 6, 4, 10], dtype=torch.int32)  # decreasing: rejected on the device
    gdn.gdn_read_device_status(clear=True)
    run_conv(cuda, x, w, b, None, None, cu, 1, 2)
    assert gdn.gdn_read_device_status(clear=True) == gdn.GDN_EDEVICE_INPUT


def test_gating_every_token(cuda):
    rng = np.random.default_rng(66)
    T, hv = 1000, 32
    a = torch.from_numpy((rng.standard_normal((T, hv)) * 15).astype(np.float32))  # both softplus branches
    b = torch.from_numpy((rng.standard_normal((T, hv)) * 30).astype(np.float32))
    w = W.WORKLOADS["decode_N256_hq16_hv32"]
    A_log, dt_bias = W.make_decode_gate_params(w)
    g, beta = gdn.gdn_gating(a.to(cuda), b.to(cuda), A_log.to(cuda), dt_bias.to(cuda))
    torch.cuda.synchronize()
    g_ref, beta_ref = oracle.decode_gates(a, b, A_log, dt_bias)
    check(g, g_ref, torch.float32, "g")
    check(beta, beta_ref, torch.float32, "beta")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_layer_core_from_projections(cuda, dtype):
    """conv (+ q/k norm) -> gates -> chunk form -> output gate, against the
    oracle's convolution, L2 norm, gates, chunk form and gated RMSNorm."""
    lengths, hq, hv = [100, 37, 64], 1, 2
    T = sum(lengths)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    x, w, b, st0 = W.make_conv_inputs(67, T, hq, hv, dtype, slots=3)
    rng = np.random.default_rng(68)
    a = torch.from_numpy(rng.standard_normal((T, hv)).astype(np.float32))
    bb = torch.from_numpy(rng.standard_normal((T, hv)).astype(np.float32))
    wl = W.Workload("layer", 68, "decode", dtype, hq=hq, hv=hv)
    A_log, dt_bias = W.make_decode_gate_params(wl)
    z, nw = W.make_output_gate(68, T, hv, dtype)
    scale = 128 ** -0.5
    # CUDA path
    st = st0.to(cuda)
    q, k, v = run_conv(cuda, x, w, b, st, None, cu, hq, hv, norm=True)
    g, beta = gdn.gdn_gating(a.to(cuda), bb.to(cuda), A_log.to(cuda), dt_bias.to(cuda))
    o, S = gdn.gdn_chunk_fwd(q, k, v, g, beta, scale, cu_seqlens=cu.to(cuda))
    y = gdn.gdn_gated_rmsnorm(o, z.to(cuda), nw.to(cuda), 1e-6)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    # oracle chain
    y_c, st_ref = oracle.causal_conv1d_silu(x, w, b, st0, cu)
    q_r, k_r, v_r = split_ref(y_c, hq, hv)
    g_r, beta_r = oracle.decode_gates(a, bb, A_log, dt_bias)
    o_r, S_r = oracle.chunked(oracle.l2_normalise(q_r), oracle.l2_normalise(k_r), v_r, g_r, beta_r, scale,
                              None, cu.numpy())
    check(y, oracle.gated_rmsnorm(o_r, z, nw, 1e-6), dtype, "y")
    check(S, S_r, dtype, "final state")
    check(st, st_ref, dtype, "conv state")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_conv_step_kernel_chained(cuda, dtype):
    """gdn_causal_conv1d_silu_step: 256 one-token sequences x 12 steps, q/k
    norm, a padding slot (-1: zero history, no write), against the oracle."""
    hq, hv, N = 16, 32, 256
    _, w, b, st0 = W.make_conv_inputs(69, 1, hq, hv, dtype, slots=N + 1)
    idx_np = np.random.default_rng(4).permutation(N + 1)[:N].astype(np.int32)
    idx_np[7] = -1
    idx = torch.from_numpy(idx_np)
    cu = torch.arange(N + 1, dtype=torch.int32)
    st = st0.to(cuda)
    st_ref = st0.double().numpy()
    for step in range(12):
        x, _, _, _ = W.make_conv_inputs(2000 + step, N, hq, hv, dtype)
        q, k, v = gdn.gdn_causal_conv1d_silu_step(x.to(cuda), w.to(cuda), hq, hv, bias=b.to(cuda), conv_state=st,
                                                  state_indices=idx.to(cuda), norm_qk=True)
        torch.cuda.synchronize()
        y_ref, st_ref = oracle.causal_conv1d_silu(x, w, b, st_ref, cu, idx_np)
        q_r, k_r, v_r = split_ref(y_ref, hq, hv)
        if step in (0, 11):
            check(q, oracle.l2_normalise(q_r), dtype, f"q step {step}")
            check(k, oracle.l2_normalise(k_r), dtype, f"k step {step}")
            check(v, v_r, dtype, f"v step {step}")
    check(st, st_ref, dtype, "conv state after 12 steps")


def test_conv_step_out_of_range_slot(cuda):
    _, w, b, st0 = W.make_conv_inputs(70, 1, 1, 2, torch.float32, slots=2)
    x, _, _, _ = W.make_conv_inputs(71, 2, 1, 2, torch.float32)
    st = st0.to(cuda)
    gdn.gdn_read_device_status(clear=True)
    gdn.gdn_causal_conv1d_silu_step(x.to(cuda), w.to(cuda), 1, 2, bias=b.to(cuda), conv_state=st,
                                    state_indices=torch.tensor([1, 5], dtype=torch.int32, device=cuda))
    assert gdn.gdn_read_device_status(clear=True) == gdn.GDN_EDEVICE_INPUT
    assert torch.equal(st[0], st0[0].to(cuda))  # slot 0 is nobody's


@pytest.mark.parametrize("state_bf16", [False, True], ids=["f32state", "bf16state"])
def test_decode_layer_core_from_projections(cuda, state_bf16):
    """Eight decode steps of the layer core from raw projections, as the
    SGLang decode path runs it: conv step (no norm) -> gated recurrent step
    (q/k norm, gates, output gate in one kernel), against the oracle's
    convolution, gated step and gated RMSNorm; optionally with the bf16 state
    cache and bf16 beta."""
    hq, hv, N = 2, 4, 5
    dtype = torch.bfloat16
    _, w, b, cst0 = W.make_conv_inputs(80, 1, hq, hv, dtype, slots=N)
    wl = W.Workload("dec_layer", 81, "decode", dtype, hq=hq, hv=hv, num_seqs=N, s0_sigma=0.05)
    A_log, dt_bias = W.make_decode_gate_params(wl)
    S0 = W.make_decode_state(wl)
    if state_bf16:
        S0 = S0.to(torch.bfloat16)
    idx = torch.tensor([3, 0, 4, 1, 2], dtype=torch.int32)
    cst, S = cst0.to(cuda), S0.to(cuda)
    cst_ref, S_ref = cst0.double().numpy(), S0.double().numpy()
    # the recurrent step alone, fed the q/k/v the GPU's conv step produced:
    # its f32 state is held to the f32 bar (the chain above it carries the
    # bf16 rounding of the conv outputs and is compared normwise)
    S_step = S0.double().numpy()
    cu = np.arange(N + 1)
    rng = np.random.default_rng(82)
    for step in range(8):
        x, _, _, _ = W.make_conv_inputs(900 + step, N, hq, hv, dtype)
        a = torch.from_numpy(rng.standard_normal((N, hv)).astype(np.float32))
        bb = torch.from_numpy(rng.standard_normal((N, hv)).astype(np.float32))
        z, nw = W.make_output_gate(900 + step, N, hv, dtype)
        q, k, v = gdn.gdn_causal_conv1d_silu_step(x.to(cuda), w.to(cuda), hq, hv, bias=b.to(cuda), conv_state=cst,
                                                  state_indices=idx.to(cuda))
        y = gdn.gdn_recurrent_step_gated(q, k, v, a.to(cuda), bb.to(cuda), A_log.to(cuda), dt_bias.to(cuda),
                                         128 ** -0.5, S, state_indices=idx.to(cuda), z=z.to(cuda),
                                         norm_weight=nw.to(cuda), norm_eps=1e-6, beta_bf16=state_bf16)
        torch.cuda.synchronize()
        y_c, cst_ref = oracle.causal_conv1d_silu(x, w, b, cst_ref, cu, idx.numpy())
        q_r, k_r, v_r = split_ref(y_c, hq, hv)
        o_r, S_ref = oracle.recurrent_step_gated(q_r, k_r, v_r, a, bb, A_log, dt_bias, 128 ** -0.5, S_ref, idx.numpy(),
                                                 beta_bf16=state_bf16, state_bf16=state_bf16)
        check(y, oracle.gated_rmsnorm(o_r, z, nw, 1e-6), dtype, f"y step {step}")
        _, S_step = oracle.recurrent_step_gated(q.cpu(), k.cpu(), v.cpu(), a, bb, A_log, dt_bias, 128 ** -0.5, S_step, idx.numpy(),
                                                beta_bf16=state_bf16, state_bf16=state_bf16)
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    check(S, S_ref, dtype, "recurrent state after 8 steps")
    if not state_bf16:
        check_f32_state(S, S_step, "recurrent state after 8 steps (step kernel alone)")
    check(cst, cst_ref, dtype, "conv state after 8 steps")
