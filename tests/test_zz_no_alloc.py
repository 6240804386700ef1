"""moe_w2_forward_noalloc against moe_w2_forward, through the C ABI.

The no-alloc entry point is for callers that cannot allocate device memory
where they run the layer (a fixed memory pool, memory already handed out in
full, or a point where an allocation would synchronise the device).  It runs
the same kernels as moe_w2_forward with its scratch in a device array the
library owns, so on the same inputs its output must be bitwise identical to
moe_w2_forward's, whatever earlier calls left in that array: two calls in a row
on different inputs (the second reuses scratch the first left behind), then
the first input again, each compared bit for bit (which also meets the layer
bar, rel L2 <= 1e-3, max abs <= 1e-2 * max|y|).  Sizes past the array's
capacity must be refused on the host.  This file is collected last so that it
also runs after every other test in the same process, and it passes on its own
in a fresh one.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.helpers import assert_close_layer, from_dev_bf16, planes_to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

MOE_W2_ERR_WORKSPACE = 3


def _dev_inputs(lay):
    return (to_dev_bf16(lay.x), torch.from_numpy(lay.ids).cuda(), torch.from_numpy(lay.weights).cuda())


def _call_noalloc(L, planes, x, ids, w, y, status, stream):
    return L.moe_w2_forward_noalloc(moe_w2._ptr(x), moe_w2._ptr(ids), moe_w2._ptr(w), ctypes.byref(planes),
                                    x.shape[0], ids.shape[1], moe_w2._ptr(y), moe_w2._ptr(status),
                                    ctypes.c_void_p(stream.cuda_stream))


def _call_forward(L, planes, x, ids, w, y, status, stream):
    need = moe_w2.workspace_size(x.shape[0], ids.shape[1], planes.num_experts, planes.hidden, planes.inter)
    work = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    st = L.moe_w2_forward(moe_w2._ptr(x), moe_w2._ptr(ids), moe_w2._ptr(w), ctypes.byref(planes), x.shape[0],
                          ids.shape[1], moe_w2._ptr(y), moe_w2._ptr(work), work.numel(), moe_w2._ptr(status),
                          ctypes.c_void_p(stream.cuda_stream))
    stream.synchronize()
    return st


@pytest.mark.parametrize("H,I,E,k,T_a,T_b,seed", [
    (512, 256, 8, 2, 4, 16, 21),        # decode path, both calls
    (1024, 512, 16, 4, 1, 80, 22),      # decode then prefill path
])
def test_two_calls_in_a_row_match_forward(H, I, E, k, T_a, T_b, seed):
    L = moe_w2.load()
    lay_a = inputs.small_layer_inputs(H, I, E, k, T_a, seed)
    lay_b = inputs.small_layer_inputs(H, I, E, k, T_b, seed)   # same seed: the same planes
    assert all(np.array_equal(lay_a.planes[n], lay_b.planes[n]) for n in lay_a.planes)
    pd = planes_to_dev(lay_a.planes)
    planes = moe_w2.make_planes(pd)
    stream = torch.cuda.current_stream()
    a, b = _dev_inputs(lay_a), _dev_inputs(lay_b)
    for T in (T_a, T_b):
        assert moe_w2.workspace_size(T, k, E, H, I) <= moe_w2.NOALLOC_WORKSPACE_BYTES

    st_na = torch.zeros(3, dtype=torch.int32, device="cuda")
    y_na = [torch.empty_like(a[0]), torch.empty_like(b[0]), torch.empty_like(a[0])]
    for i, inp in enumerate((a, b, a)):
        assert _call_noalloc(L, planes, *inp, y_na[i], st_na[i:i + 1], stream) == 0
    stream.synchronize()

    st_ref = torch.zeros(2, dtype=torch.int32, device="cuda")
    y_ref_a = torch.empty_like(a[0])
    y_ref_b = torch.empty_like(b[0])
    assert _call_forward(L, planes, *a, y_ref_a, st_ref[0:1], stream) == 0
    assert _call_forward(L, planes, *b, y_ref_b, st_ref[1:2], stream) == 0

    assert st_na.tolist() == [0, 0, 0] and st_ref.tolist() == [0, 0]
    # the same kernels on the same inputs: bit for bit, not just within tolerance
    assert torch.equal(y_na[0], y_ref_a), f"no-alloc first call T={T_a} differs from moe_w2_forward"
    assert torch.equal(y_na[1], y_ref_b), f"no-alloc second call T={T_b} differs from moe_w2_forward"
    assert torch.equal(y_na[2], y_ref_a), f"no-alloc third call T={T_a} differs from moe_w2_forward"
    assert_close_layer(from_dev_bf16(y_na[1]), from_dev_bf16(y_ref_b), f"no-alloc second call T={T_b}")


def test_sizes_past_the_static_workspace_are_refused():
    L = moe_w2.load()
    H, I, E, k = 6144, 2048, 256, 8
    fits = [T for T in range(1, 65) if moe_w2.workspace_size(T, k, E, H, I) <= moe_w2.NOALLOC_WORKSPACE_BYTES]
    t_max = max(fits)
    assert fits == list(range(1, t_max + 1)) and t_max >= 16   # a useful decode batch fits
    # the size check comes before any pointer is used: nothing is enqueued
    planes = moe_w2.Planes(None, None, None, None, E, H, I)
    st = L.moe_w2_forward_noalloc(None, None, None, ctypes.byref(planes), t_max + 1, k, None, None, None)
    assert st == MOE_W2_ERR_WORKSPACE
    assert moe_w2.status_string(st) == "workspace too small"
