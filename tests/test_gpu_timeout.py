"""A bounded device-side wait that runs out, under test.

Every wait in the tensor-core prefill kernel (copies, MMA completion, the
ready flags between the prepare engines and the walks) is bounded; when one
runs out the kernel records GDN_ETIMEOUT in the device status word, drains
what it has in flight and returns. Here the limit is lowered to 5 us, far
below the ~10 us it takes to prepare the first chunk, so the walks' first
flag wait gives up. The test then checks the status, restores the default
limit and runs the same problem again on the same stream: the context is
still usable and the result matches the oracle.
"""
import pytest
import torch

from gated_deltanet_chunked_gb300 import gdn, workloads as W
from parity_util import check, check_per_head, oracle_prefill, to_dev

pytestmark = pytest.mark.gpu


def test_wait_limit_runs_out_then_normal_call_passes(cuda):
    inp = W.make_custom_prefill(301, [640], 1, 2, torch.bfloat16, s0_sigma=0.05)
    d = to_dev(inp, cuda)
    run = lambda: gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                    initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"])
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    try:
        gdn.gdn_set_wait_limit_ns(5000)
        run()
        torch.cuda.synchronize()
        assert gdn.gdn_get_device_status() == gdn.GDN_ETIMEOUT
    finally:
        gdn.gdn_set_wait_limit_ns(0)  # back to the default 2 s
    assert gdn.gdn_get_device_status() == gdn.GDN_OK  # read and reset above
    o, S = run()
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_status() == gdn.GDN_OK
    o_ref, S_ref = oracle_prefill(inp)
    check(o, o_ref, torch.bfloat16, "o after a timed-out call")
    check(S, S_ref, torch.bfloat16, "final_state after a timed-out call")
    check_per_head(o, o_ref, inp["cu_seqlens"], torch.bfloat16, "o after a timed-out call")
