"""Shared helpers of the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import oracle
from gated_deltanet_chunked_gb300 import gdn

# Tolerances fixed for the two arithmetic paths:
#  * f32 path: max|x - ref| / max|ref| <= 1e-4 (the criterion the decode page
#    applies to its f32 kernels against its CPU reference).
#  * bf16 path: ||x - ref||_2 / ||ref||_2 <= 2e-2 on o and on the final state.
F32_MAX_REL = 1e-4
BF16_NORMWISE = 2e-2


def max_rel(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def normwise(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30))


def check(x, ref, io_dtype, what):
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else x
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    if io_dtype == torch.float32:
        err = max_rel(x, ref)
        assert err <= F32_MAX_REL, f"{what}: max_rel {err:.3e} > {F32_MAX_REL}"
    else:
        err = normwise(x, ref)
        assert err <= BF16_NORMWISE, f"{what}: normwise {err:.3e} > {BF16_NORMWISE}"
    return err


def check_f32_state(x, ref, what):
    """An f32-arithmetic result (the decode step's f32 state, whatever the io
    dtype: bf16 inputs are widened exactly) at the f32 bar, element by
    element: max|x - ref| / max|ref| <= 1e-4."""
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else x
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    err = max_rel(x, ref)
    assert err <= F32_MAX_REL, f"{what}: max_rel {err:.3e} > {F32_MAX_REL}"
    return err


# round-to-nearest into bf16 (8 significant bits) moves a value by at most
# 2^-8 of its magnitude
BF16_HALF_ULP = 2.0 ** -8


def check_bf16_rounded(x, ref, what):
    """A bf16 output of f32 arithmetic, element by element: every element
    within its own rounding bound, |x - ref| <= 2^-8 |ref| plus the f32 bar
    (1e-4 of the largest magnitude) for the arithmetic before the rounding."""
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    bound = BF16_HALF_ULP * np.abs(ref) * (1 + 1e-3) + F32_MAX_REL * max(float(np.max(np.abs(ref))), 1e-30)
    excess = np.abs(x - ref) / bound
    worst = np.unravel_index(int(np.argmax(excess)), excess.shape)
    assert excess[worst] <= 1.0, (f"{what}: element {worst} off by {abs(x[worst] - ref[worst]):.3e} "
                                  f"(ref {ref[worst]:.3e}, bound {bound[worst]:.3e})")
    return float(excess[worst])


def check_per_head(x, ref, cu, io_dtype, what):
    """check() applied to every (sequence, head) slice of a packed [T, H, d]
    output (cu = offsets [N+1]) or of a [N, H, dk, dv] state (cu None), so
    that a wrong chunk of one sequence or one bad head is not diluted by the
    rest of the tensor. Returns the worst error."""
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    worst = 0.0
    if cu is None:
        for n in range(x.shape[0]):
            for h in range(x.shape[1]):
                worst = max(worst, check(x[n, h], ref[n, h], io_dtype, f"{what} [seq {n}, head {h}]"))
    else:
        cu = [int(c) for c in (cu.tolist() if hasattr(cu, "tolist") else cu)]
        for n in range(len(cu) - 1):
            if cu[n + 1] == cu[n]:
                continue
            for h in range(x.shape[1]):
                worst = max(worst, check(x[cu[n]:cu[n + 1], h], ref[cu[n]:cu[n + 1], h], io_dtype,
                                         f"{what} [seq {n}, head {h}]"))
    return worst


def to_dev(inp, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_gpu_prefill(inp, dev, packed=True, output_final_state=True):
    """Runs gdn_chunk_fwd on packed inputs; packed=False sends a single
    sequence through the dense [1, T, H, d] layout instead."""
    d = to_dev(inp, dev)
    cu = d["cu_seqlens"]
    if not packed:
        assert cu is None or cu.numel() == 2
        b = lambda x: x.unsqueeze(0)
        o, S = gdn.gdn_chunk_fwd(b(d["q"]), b(d["k"]), b(d["v"]), b(d["g"]), b(d["beta"]), d["scale"],
                                 initial_state=d["initial_state"], output_final_state=output_final_state)
        o = o[0]
    else:
        if cu is None:
            cu = torch.tensor([0, d["q"].shape[0]], dtype=torch.int32, device=dev)
        o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                 initial_state=d["initial_state"], cu_seqlens=cu,
                                 output_final_state=output_final_state)
    torch.cuda.synchronize()
    status = gdn.gdn_read_device_status()
    assert status == gdn.GDN_OK, gdn.gdn_status_string(status)
    return o, S


def head_slice(inp, hk, group):
    """Inputs restricted to q/k head hk and its `group` v-heads (for sampling)."""
    hv = slice(hk * group, (hk + 1) * group)
    out = dict(inp)
    out["q"], out["k"] = inp["q"][:, hk:hk + 1], inp["k"][:, hk:hk + 1]
    out["v"], out["g"], out["beta"] = inp["v"][:, hv], inp["g"][:, hv], inp["beta"][:, hv]
    if inp["initial_state"] is not None:
        out["initial_state"] = inp["initial_state"][:, hv]
    return out


def oracle_prefill(inp, routine="chunked"):
    cu = inp["cu_seqlens"]
    if cu is None:
        cu = np.array([0, inp["q"].shape[0]])
    fn = oracle.chunked if routine == "chunked" else oracle.recurrent
    return fn(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"], inp["initial_state"], cu)
