"""Parity of gdn_recurrent_step (CUDA, through the C ABI) with the CPU oracle.

The 256-sequence x 32-head workload is checked in full on its first step and
over 100 consecutive steps (fresh seeded inputs each step) on a sample of
sequences; slot indirection, padding slots and out-of-range slots are
checked, and T single steps are compared with a T-token prefill.

The step does f32 arithmetic on exactly widened inputs, so its f32 state is
held to the f32 bar (max_rel <= 1e-4, element by element) whatever the io
dtype, and a bf16 output to its own rounding bound element by element.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, check_bf16_rounded, check_f32_state, oracle_prefill, run_gpu_prefill, to_dev

pytestmark = pytest.mark.gpu

DEC = W.WORKLOADS["decode_N256_hq16_hv32"]


def step_gpu(inp, state, dev, idx=None, out=None):
    d = to_dev(inp, dev)
    o = gdn.gdn_recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], state,
                               state_indices=idx, out=out)
    torch.cuda.synchronize()
    return o


def test_decode_first_step_full(cuda):
    state0 = W.make_decode_state(DEC)
    state = state0.to(cuda)
    inp = W.make_decode_step(DEC, 0)
    o = step_gpu(inp, state, cuda)
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    o_ref, st_ref = oracle.recurrent_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"], state0)
    check(o, o_ref, torch.bfloat16, "o")
    check_bf16_rounded(o, o_ref, "o")
    check_f32_state(state, st_ref, "state")


def test_decode_100_steps_sampled(cuda):
    state0 = W.make_decode_state(DEC)
    state = state0.to(cuda)
    sample = np.array([0, 17, 101, 255])
    st_ref = state0[sample].double().numpy()
    for step in range(DEC.steps):
        inp = W.make_decode_step(DEC, step)
        o = step_gpu(inp, state, cuda)
        sub = {k: v[sample] for k, v in inp.items() if isinstance(v, torch.Tensor)}
        o_ref, st_ref = oracle.recurrent_step(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], inp["scale"],
                                              st_ref)
        if step in (0, 9, 49, 99):
            check_bf16_rounded(o[sample], o_ref, f"o step {step}")
    check_f32_state(state[sample], st_ref, "state after 100 steps")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_slot_indices_and_padding(cuda, dtype):
    rng = np.random.default_rng(3)
    N, slots = 6, 9
    inp = W.make_custom_prefill(31, [1] * N, 2, 4, dtype)
    inp = {k: v for k, v in inp.items() if k in ("q", "k", "v", "g", "beta", "scale")}
    state0 = torch.from_numpy(rng.standard_normal((slots, 4, 128, 128)).astype(np.float32) * 0.05)
    idx = torch.tensor([8, -1, 0, 3, -1, 5], dtype=torch.int32)
    state = state0.to(cuda)
    out = torch.full(inp["v"].shape, 5.0, dtype=dtype, device=cuda)
    o = step_gpu(inp, state, cuda, idx=idx.to(cuda), out=out)
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    o_ref, st_ref = oracle.recurrent_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                          state0, idx.numpy())
    live = [0, 2, 3, 5]
    check(o[live], o_ref[live], dtype, "o")
    check_f32_state(state, st_ref, "state")
    assert torch.all(o[[1, 4]] == 5.0)  # padding rows untouched
    untouched = [1, 2, 4, 6, 7]
    assert torch.equal(state[untouched], state0[untouched].to(cuda))


def test_out_of_range_slot_reports_status(cuda):
    inp = W.make_custom_prefill(32, [1, 1], 1, 1, torch.float32)
    inp = {k: v for k, v in inp.items() if k in ("q", "k", "v", "g", "beta", "scale")}
    state = torch.zeros((2, 1, 128, 128), device=cuda)
    gdn.gdn_read_device_status(clear=True)
    step_gpu(inp, state, cuda, idx=torch.tensor([0, 2], dtype=torch.int32, device=cuda))
    assert gdn.gdn_read_device_status(clear=True) == gdn.GDN_EDEVICE_INPUT


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_steps_equal_prefill(cuda, dtype):
    """T single steps from S0 match one T-token prefill (and the oracle)."""
    T = 70
    inp = W.make_custom_prefill(33, [T], 2, 4, dtype, s0_sigma=0.05)
    o_pre, S_pre = run_gpu_prefill(inp, cuda)
    state = inp["initial_state"].clone().to(cuda)
    outs = []
    for t in range(T):
        tok = {k: inp[k][t:t + 1] for k in ("q", "k", "v", "g", "beta")}
        tok["scale"] = inp["scale"]
        outs.append(step_gpu(tok, state, cuda))
    o_steps = torch.cat(outs)
    o_ref, S_ref = oracle_prefill(inp, routine="recurrent")
    check(o_steps, o_ref, dtype, "o (steps)")
    if dtype == torch.bfloat16:
        check_bf16_rounded(o_steps, o_ref, "o (steps)")
    check_f32_state(state, S_ref, "state (steps)")
    check(o_pre, o_ref, dtype, "o (prefill)")
    check(S_pre, S_ref, dtype, "final state (prefill)")
