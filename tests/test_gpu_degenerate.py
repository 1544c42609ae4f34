"""The method's degenerate cases on the CUDA path, checked against their
closed forms rather than only against the oracle (the gated delta rule of the
"Lab3 GDN Prefill" page, section "Linear Attention 与 Gated DeltaNet", with
S_t = a_t (I - b_t k_t^T k_t) S_{t-1} + b_t k_t^T v_t and o_t = scale q_t S_t):

* beta = 0: nothing is ever written, so S_T = exp(sum of g) S0 and
  o_t = scale exp(G_t) q_t S0, with G_t the running sum of g over the
  sequence up to and including t (prefill and the decode step);
* g = 0, beta = 1 and orthonormal keys (at most d_k = 128 tokens), S0 = 0:
  every token overwrites its own key's direction, so k_j S_T = v_j for each
  token j of the sequence.

Both io dtypes; packed sequences with several chunks and tail chunks.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, run_gpu_prefill

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.bfloat16]
IDS = ["f32", "bf16"]


def _np(t):
    """The values the kernels see (bf16 inputs widened exactly)."""
    return t.double().numpy()


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_prefill_beta_zero_is_pure_decay(cuda, dtype):
    lengths, hq, hv = [150, 64, 9, 1], 2, 4
    inp = W.make_custom_prefill(71, lengths, hq, hv, dtype, s0_sigma=0.1, g_mu=-2.0)
    inp["beta"] = torch.zeros_like(inp["beta"])
    o, S = run_gpu_prefill(inp, cuda)
    q, g, s0, cu = _np(inp["q"]), _np(inp["g"]), _np(inp["initial_state"]), inp["cu_seqlens"].numpy()
    group, scale = hv // hq, inp["scale"]
    o_ref = np.zeros((q.shape[0], hv, 128))
    S_ref = np.zeros_like(s0)
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        G = np.cumsum(g[a:b], axis=0)  # [L, hv]
        for h in range(hv):
            o_ref[a:b, h] = scale * np.exp(G[:, h])[:, None] * (q[a:b, h // group] @ s0[n, h])
            S_ref[n, h] = np.exp(G[-1, h]) * s0[n, h]
    check(o, o_ref, dtype, "o (beta = 0)")
    check(S, S_ref, dtype, "final state (beta = 0)")


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_prefill_orthonormal_keys_overwrite(cuda, dtype):
    lengths, hq, hv = [128, 100, 37], 2, 4  # two full chunks; a full chunk + a tail; a tail
    inp = W.make_custom_prefill(72, lengths, hq, hv, dtype)  # no initial state: S0 = 0
    cu = inp["cu_seqlens"].numpy()
    rng = np.random.Generator(np.random.PCG64([72, 1]))
    k = np.zeros((int(cu[-1]), hq, 128))
    for n in range(len(lengths)):
        for h in range(hq):
            Q, _ = np.linalg.qr(rng.normal(size=(128, 128)))
            k[cu[n]:cu[n + 1], h] = Q[: lengths[n]]
    inp["k"] = torch.from_numpy(k).to(dtype)
    inp["g"] = torch.zeros_like(inp["g"])
    inp["beta"] = torch.ones_like(inp["beta"])
    _, S = run_gpu_prefill(inp, cuda)
    S = S.cpu().double().numpy()
    kd, v = _np(inp["k"]), _np(inp["v"])
    group = hv // hq
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        for h in range(hv):
            check(kd[a:b, h // group] @ S[n, h], v[a:b, h], dtype, f"k_j S_T against v_j (seq {n}, head {h})")


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_decode_step_beta_zero_is_pure_decay(cuda, dtype):
    N, hq, hv = 32, 2, 4
    rng = np.random.Generator(np.random.PCG64(73))
    q = torch.from_numpy(rng.normal(size=(N, hq, 128)) / np.sqrt(128)).to(dtype)
    k = torch.from_numpy(rng.normal(size=(N, hq, 128)) / np.sqrt(128)).to(dtype)
    v = torch.from_numpy(rng.normal(size=(N, hv, 128))).to(dtype)
    g = torch.from_numpy(-np.log1p(np.exp(rng.normal(size=(N, hv))))).float()
    beta = torch.zeros((N, hv), dtype=torch.float32)
    s0 = rng.normal(scale=0.1, size=(N, hv, 128, 128))
    state = torch.from_numpy(s0).float().to(cuda)
    scale = 1.0 / np.sqrt(128)
    o = gdn.gdn_recurrent_step(q.to(cuda), k.to(cuda), v.to(cuda), g.to(cuda), beta.to(cuda), scale, state)
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK
    s0 = torch.from_numpy(s0).float().double().numpy()  # the f32 state the kernel started from
    a = np.exp(g.double().numpy())
    S_ref = a[:, :, None, None] * s0
    qd = _np(q)
    o_ref = np.stack([scale * np.einsum("nd,nde->ne", qd[:, h // (hv // hq)], S_ref[:, h]) for h in range(hv)], 1)
    check(o, o_ref, dtype, "o (beta = 0)")
    check(state, S_ref, torch.float32, "state (beta = 0)")
