"""The decode kernels' pipeline-timeout report, driven without a fault or a hang.

Every wait inside the kernels is bounded; when one gives up, the kernel stops,
frees its tensor memory, returns, and ORs MOE_W2_DEV_PIPELINE_TIMEOUT into the
device status word.  moe_w2_debug_force_pipeline_timeout makes the cross-CTA
dependency wait of the decode kernels (a down item waiting for the h it reads)
unsatisfiable with a limit of about 0.1 ms, so that wait gives up on purpose.
The test checks that the call returns, the bit is set, and the next normal call
on the same stream is correct again.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.helpers import assert_close_layer, from_dev_bf16, planes_to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 0x80000000


@pytest.mark.parametrize("I,T,kernel", [(512, 4, "decode_mma_kernel"), (512, 4, "decode_stream_kernel"),
                                        (512, 16, "decode_layer_kernel")])
def test_forced_dependency_timeout_is_reported_and_recovers(I, T, kernel):
    with moe_w2.decode_stream(kernel == "decode_stream_kernel"):
        _forced_timeout(I, T, kernel)


def _forced_timeout(I, T, kernel):
    assert moe_w2.decode_kernel(T, 2, 512, I) == kernel
    lay = inputs.small_layer_inputs(512, I, 8, 2, T, 60 + T)
    pd = planes_to_dev(lay.planes)
    x, ids, w = to_dev_bf16(lay.x), torch.from_numpy(lay.ids).cuda(), torch.from_numpy(lay.weights).cuda()
    L = moe_w2.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        assert L.moe_w2_debug_force_pipeline_timeout(1) == 0
        moe_w2.forward(x, ids, w, pd, status=st)
        torch.cuda.synchronize()              # the kernel returned: no hang
    finally:
        L.moe_w2_debug_force_pipeline_timeout(0)
    assert (int(st.item()) & 0xFFFFFFFF) & TIMEOUT_BIT, f"{kernel}: bit not set"

    st.zero_()
    y = moe_w2.forward(x, ids, w, pd, status=st)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes)
    assert int(st.item()) == rst == 0
    assert_close_layer(from_dev_bf16(y), ref, f"after a forced timeout, T={T}")
