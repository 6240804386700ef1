"""GPU parity of the MXFP4 loader (moe_w2_requant_mxfp4) and of zero-sign
balancing in both FP4 loaders, bit-exact against the CPU oracle.

Codes and UE8M0 bytes compared element by element on the same seeded inputs:
small tensors with a ragged last row block at scale bytes across the whole
range (0, 1, 2, 127, 253, 254, and 255 = NaN), blocks of +0 and -0, the
16-expert MXFP4 workload (gate/up 2 x [2048 x 6144] and down [6144 x 2048] per
expert) on every block, and an NVFP4 export whose exact zeros are all +0, with
and without balancing.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2

pytestmark = pytest.mark.gpu

BAL = moe_w2.REQUANT_BALANCE_ZERO_SIGNS


def _gpu_mx(t: inputs.Mxfp4Tensors, options=0):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    c, u = moe_w2.requant_mxfp4(torch.from_numpy(t.e2m1).cuda(), torch.from_numpy(t.scales).cuda(), status=st,
                                options=options)
    return c.cpu().numpy(), u.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("options", [0, BAL])
def test_small_tensors_every_kind_of_scale_byte(options):
    rng = np.random.default_rng(51)
    t = inputs.mxfp4_tensors(rng, 3, 200, 384, plus_zero_frac=0.15)
    flat = t.scales.reshape(-1)
    pick = rng.choice(flat.size, size=7 * 40, replace=False).reshape(7, 40)
    for s, idx in zip([0, 1, 2, 127, 253, 254, 255], pick):
        flat[idx] = s
    c, u, st = _gpu_mx(t, options)
    rc, ru, rst = oracle.requant_mxfp4(t.e2m1, t.scales, options=options)
    assert st == rst == oracle.BAD_NVFP4
    assert np.array_equal(u, ru) and np.array_equal(c, rc)


@pytest.mark.parametrize("options", [0, BAL])
def test_zero_blocks(options):
    e2m1 = np.zeros((4, 1, 16), np.uint8)
    e2m1[1] = 0x88            # all -0
    e2m1[2] = 0x80            # +0, -0 alternating
    e2m1[3, 0, :4] = 0x21     # a few small values among +0
    sc = np.array([127, 1, 254, 100], np.uint8).reshape(4, 1, 1)
    c, u, st = _gpu_mx(inputs.Mxfp4Tensors(e2m1, sc), options)
    rc, ru, rst = oracle.requant_mxfp4(e2m1, sc, options=options)
    assert st == rst == 0 and np.array_equal(u, ru) and np.array_equal(c, rc)


def test_mxfp4_workload_every_block():
    gu, dn = inputs.requant_mxfp4_inputs(experts=inputs.REQUANT_MXFP4_CASES["requant_mxfp4_16"])
    for t in (gu, dn):
        c, u, st = _gpu_mx(t)
        rc, ru, rst = oracle.requant_mxfp4(t.e2m1, t.scales, parallel=True)
        assert st == rst == 0
        assert np.array_equal(u, ru)
        assert np.array_equal(c, rc)


@pytest.mark.parametrize("options", [0, BAL])
def test_nvfp4_plus_zero_export(options):
    rng = np.random.default_rng(52)
    t = inputs.plus_zero_nvfp4(rng, 4, 300, 512, zero_frac=0.3)
    t.e4m3[1, 3, 5] = 0x00     # a zero e4m3 scale: the half-block is all exact zeros
    t.e4m3[2, 7, 0] = 0x80     # -0 scale
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    c, u = moe_w2.requant(torch.from_numpy(t.e2m1).cuda(), torch.from_numpy(t.e4m3).cuda(),
                          torch.from_numpy(t.scale_2).cuda(), status=st, options=options)
    rc, ru, rst = oracle.requant(t.e2m1, t.e4m3, t.scale_2, options=options)
    assert int(st.item()) == rst == 0
    assert np.array_equal(u.cpu().numpy(), ru) and np.array_equal(c.cpu().numpy(), rc)
