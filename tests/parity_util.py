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
