"""Parity of gdn_recurrent_step_gated (CUDA, through the C ABI) with the
CPU oracle's decode front-end (gates from the projections, q/k L2 norm).

The 256-sequence x 32-head workload is checked in full on its first step and
over 100 consecutive steps on a sample of sequences; small cases cover both
io dtypes, slot indirection with padding slots, gate inputs on both sides of
the +-20 softplus branches, saturated sigmoids and zero q/k rows.

The kernel's arithmetic is f32 throughout, so an f32 state is held to the f32
bar (max_rel <= 1e-4, element by element) whatever the io dtype; bf16 outputs
are held to their rounding bound element by element. Only the bf16 state
cache of the SGLang precision mode is compared normwise.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, check_bf16_rounded, check_f32_state, to_dev

pytestmark = pytest.mark.gpu

DEC = W.WORKLOADS["decode_N256_hq16_hv32"]


def step_gpu(inp, A_log, dt_bias, state, dev, idx=None, out=None):
    d = to_dev(inp, dev)
    o = gdn.gdn_recurrent_step_gated(d["q"], d["k"], d["v"], d["a"], d["b"], A_log.to(dev), dt_bias.to(dev),
                                     d["scale"], state, state_indices=idx, out=out)
    torch.cuda.synchronize()
    return o


def step_ref(inp, A_log, dt_bias, state, idx=None):
    return oracle.recurrent_step_gated(inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], A_log, dt_bias,
                                       inp["scale"], state, idx)


def test_gated_decode_first_step_full(cuda):
    A_log, dt_bias = W.make_decode_gate_params(DEC)
    state0 = W.make_decode_state(DEC)
    state = state0.to(cuda)
    inp = W.make_decode_step_gated(DEC, 0)
    o = step_gpu(inp, A_log, dt_bias, state, cuda)
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    o_ref, st_ref = step_ref(inp, A_log, dt_bias, state0)
    check(o, o_ref, torch.bfloat16, "o")
    check_bf16_rounded(o, o_ref, "o")
    check_f32_state(state, st_ref, "state")


def test_gated_decode_100_steps_sampled(cuda):
    A_log, dt_bias = W.make_decode_gate_params(DEC)
    state0 = W.make_decode_state(DEC)
    state = state0.to(cuda)
    sample = np.array([0, 31, 128, 255])
    st_ref = state0[sample].double().numpy()
    for step in range(DEC.steps):
        inp = W.make_decode_step_gated(DEC, step)
        o = step_gpu(inp, A_log, dt_bias, state, cuda)
        sub = {k: (v[sample] if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        o_ref, st_ref = step_ref(sub, A_log, dt_bias, st_ref)
        if step in (0, 9, 49, 99):
            check_bf16_rounded(o[sample], o_ref, f"o step {step}")
    check_f32_state(state[sample], st_ref, "state after 100 steps")


def _small_case(dtype, N=6, hq=2, hv=4, a_sigma=1.0, seed=41):
    w = W.Workload("small", seed, "decode", dtype, hq=hq, hv=hv, num_seqs=N, s0_sigma=0.05)
    inp = W.make_decode_step_gated(w, 0, a_sigma=a_sigma)
    A_log, dt_bias = W.make_decode_gate_params(w)
    return w, inp, A_log, dt_bias


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gated_slots_padding_and_softplus_branches(cuda, dtype):
    """a ~ N(0, 30^2): most gates fall in the linear or exponential softplus
    branch; b spans saturated sigmoids. Slot indirection with padding."""
    w, inp, A_log, dt_bias = _small_case(dtype, N=6, a_sigma=30.0)
    inp["b"] = torch.tensor(np.linspace(-60, 60, 24, dtype=np.float32).reshape(6, 4))
    a = inp["a"].numpy() + dt_bias.numpy()[None]
    assert np.any(a > 20) and np.any(a < -20) and np.any(np.abs(a) < 20)
    slots = 9
    rng = np.random.default_rng(5)
    state0 = torch.from_numpy(rng.standard_normal((slots, 4, 128, 128)).astype(np.float32) * 0.05)
    idx = torch.tensor([8, -1, 0, 3, -1, 5], dtype=torch.int32)
    state = state0.to(cuda)
    out = torch.full(inp["v"].shape, 5.0, dtype=dtype, device=cuda)
    o = step_gpu(inp, A_log, dt_bias, state, cuda, idx=idx.to(cuda), out=out)
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    o_ref, st_ref = step_ref(inp, A_log, dt_bias, state0, idx.numpy())
    live = [0, 2, 3, 5]
    check(o[live], o_ref[live], dtype, "o")
    check_f32_state(state, st_ref, "state")
    assert torch.all(o[[1, 4]] == 5.0)
    untouched = [1, 2, 4, 6, 7]
    assert torch.equal(state[untouched], state0[untouched].to(cuda))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gated_zero_rows(cuda, dtype):
    """A zero key writes nothing (state only decays); a zero query reads 0."""
    w, inp, A_log, dt_bias = _small_case(dtype, N=3, hq=1, hv=2, seed=43)
    inp["k"][0] = 0
    inp["q"][1] = 0
    state0 = W.make_decode_state(w)
    state = state0.to(cuda)
    o = step_gpu(inp, A_log, dt_bias, state, cuda)
    o_ref, st_ref = step_ref(inp, A_log, dt_bias, state0)
    assert torch.all(o[1] == 0)
    check(o[[0, 2]], o_ref[[0, 2]], dtype, "o")
    check_f32_state(state, st_ref, "state")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gated_many_steps_small(cuda, dtype):
    """40 steps of a GVA case (hv = 4 hq) against the oracle, full compare."""
    w = W.Workload("small_steps", 44, "decode", dtype, hq=2, hv=8, num_seqs=5, s0_sigma=0.05)
    A_log, dt_bias = W.make_decode_gate_params(w)
    state0 = W.make_decode_state(w)
    state = state0.to(cuda)
    st_ref = state0.double().numpy()
    for step in range(40):
        inp = W.make_decode_step_gated(w, step)
        o = step_gpu(inp, A_log, dt_bias, state, cuda)
        o_ref, st_ref = step_ref(inp, A_log, dt_bias, st_ref)
        check(o, o_ref, dtype, f"o step {step}")
        if dtype == torch.bfloat16:
            check_bf16_rounded(o, o_ref, f"o step {step}")
    check_f32_state(state, st_ref, "state after 40 steps")


def test_gated_invalid_arguments(cuda):
    w, inp, A_log, dt_bias = _small_case(torch.float32, N=2)
    d = to_dev(inp, cuda)
    state = torch.zeros((2, 4, 128, 128), device=cuda)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_recurrent_step_gated(d["q"], d["k"], d["v"], d["a"], None, A_log.to(cuda), dt_bias.to(cuda),
                                     d["scale"], state)
    assert e.value.status == gdn.GDN_EINVAL
    assert torch.all(state == 0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gated_decode_with_output_gate(cuda, dtype):
    """Front-end, step and output gate (RMSNorm over the head, silu(z)) in one
    kernel, against the oracle's step followed by its gated RMSNorm."""
    w, inp, A_log, dt_bias = _small_case(dtype, N=6, hq=2, hv=4, seed=45)
    z, weight = W.make_output_gate(45, 6, 4, dtype)
    idx = torch.tensor([3, 0, -1, 5, 1, 2], dtype=torch.int32)
    rng = np.random.default_rng(6)
    state0 = torch.from_numpy(rng.standard_normal((6, 4, 128, 128)).astype(np.float32) * 0.05)
    state = state0.to(cuda)
    d = to_dev(inp, cuda)
    out = torch.full(inp["v"].shape, 7.0, dtype=dtype, device=cuda)
    gdn.gdn_recurrent_step_gated(d["q"], d["k"], d["v"], d["a"], d["b"], A_log.to(cuda), dt_bias.to(cuda),
                                 d["scale"], state, state_indices=idx.to(cuda), out=out, z=z.to(cuda),
                                 norm_weight=weight.to(cuda), norm_eps=1e-6)
    torch.cuda.synchronize()
    o_ref, st_ref = step_ref(inp, A_log, dt_bias, state0, idx.numpy())
    y_ref = oracle.gated_rmsnorm(o_ref, z, weight, 1e-6)
    live = [0, 1, 3, 4, 5]
    check(out[live], y_ref[live], dtype, "y")
    if dtype == torch.bfloat16:
        check_bf16_rounded(out[live], y_ref[live], "y")
    check_f32_state(state, st_ref, "state")
    assert torch.all(out[2] == 7.0)


def test_gated_decode_full_with_output_gate(cuda):
    A_log, dt_bias = W.make_decode_gate_params(DEC)
    z, weight = W.make_output_gate(DEC.seed, DEC.num_seqs, DEC.hv, DEC.io_dtype)
    state0 = W.make_decode_state(DEC)
    state = state0.to(cuda)
    inp = W.make_decode_step_gated(DEC, 3)
    d = to_dev(inp, cuda)
    y = gdn.gdn_recurrent_step_gated(d["q"], d["k"], d["v"], d["a"], d["b"], A_log.to(cuda), dt_bias.to(cuda),
                                     d["scale"], state, z=z.to(cuda), norm_weight=weight.to(cuda), norm_eps=1e-6)
    torch.cuda.synchronize()
    o_ref, st_ref = step_ref(inp, A_log, dt_bias, state0)
    y_ref = oracle.gated_rmsnorm(o_ref, z, weight, 1e-6)
    check(y, y_ref, torch.bfloat16, "y")
    check_bf16_rounded(y, y_ref, "y")
    check_f32_state(state, st_ref, "state")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("gated", [False, True], ids=["plain", "gated"])
def test_sglang_precision_mode(cuda, dtype, gated):
    """bf16 state cache + bf16 beta, 30 chained steps with padding slots,
    against the oracle with the same two roundings. With a bf16 state the
    comparison is normwise whatever the io dtype (the state itself carries
    bf16 rounding; a 1-ulp tie difference between the f32 kernel and the f64
    oracle is 0.4% of that element)."""
    w = W.Workload("sgl", 72, "decode", dtype, hq=2, hv=4, num_seqs=6, s0_sigma=0.05)
    A_log, dt_bias = W.make_decode_gate_params(w)
    rng = np.random.default_rng(7)
    state0 = torch.from_numpy(rng.standard_normal((8, 4, 128, 128)).astype(np.float32) * 0.05).to(torch.bfloat16)
    idx = torch.tensor([5, -1, 0, 7, 2, -1], dtype=torch.int32)
    state = state0.to(cuda)
    st_ref = state0.double().numpy()
    for step in range(30):
        if gated:
            inp = W.make_decode_step_gated(w, step)
            d = to_dev(inp, cuda)
            o = gdn.gdn_recurrent_step_gated(d["q"], d["k"], d["v"], d["a"], d["b"], A_log.to(cuda),
                                             dt_bias.to(cuda), d["scale"], state, state_indices=idx.to(cuda),
                                             beta_bf16=True)
            o_ref, st_ref = oracle.recurrent_step_gated(inp["q"], inp["k"], inp["v"], inp["a"], inp["b"], A_log,
                                                        dt_bias, inp["scale"], st_ref, idx.numpy(), beta_bf16=True,
                                                        state_bf16=True)
        else:
            inp = W.make_decode_step(w, step)
            d = to_dev(inp, cuda)
            o = gdn.gdn_recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], state,
                                       state_indices=idx.to(cuda), beta_bf16=True)
            o_ref, st_ref = oracle.recurrent_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                                  st_ref, idx.numpy(), beta_bf16=True, state_bf16=True)
        torch.cuda.synchronize()
        live = [0, 2, 3, 4]
        if step in (0, 29):
            check(o[live], o_ref[live], torch.bfloat16, f"o step {step}")
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    check(state, st_ref, torch.bfloat16, "bf16 state after 30 steps")
    assert torch.equal(state[[1, 3, 4, 6]], state0[[1, 3, 4, 6]].to(cuda))  # nobody's slots
