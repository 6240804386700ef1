"""GPU parity of the routing permutation and the NVFP4 re-quantizer (bit-exact).

Both run through the C ABI (moe_w2_permute, moe_w2_requant) and are compared
element by element with the CPU oracle on the same seeded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2

pytestmark = pytest.mark.gpu


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("T,k,E,seed", [(1, 8, 256, 0), (4, 2, 8, 1), (32, 8, 256, 2), (64, 16, 1024, 3),
                                        (8192, 8, 256, 4), (1000, 3, 17, 5), (3, 1, 1, 6), (20000, 16, 300, 7)])
def test_permute_bit_exact(T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    st = _status()
    s, inv, off = moe_w2.permute(torch.from_numpy(ids).cuda(), E, status=st)
    rs, rinv, roff, rst = oracle.permute(ids, E)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert int(st.item()) == rst == 0


@pytest.mark.parametrize("T,k,E", [(3, 8, 64), (4, 8, 256), (2, 16, 40), (33, 1, 5)])
def test_permute_small_steps_with_invalid_and_repeated_ids(T, k, E):
    # steps of at most 32 pairs take the one-warp path, 33 the CTA path
    rng = np.random.default_rng(T * 100 + k)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids.flat[1] = -1
    ids.flat[-1] = E
    ids.flat[2] = ids.flat[0]
    st = _status()
    s, inv, off = moe_w2.permute(torch.from_numpy(ids).cuda(), E, status=st)
    rs, rinv, roff, rst = oracle.permute(ids, E)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert int(st.item()) == rst == moe_w2.DEV_BAD_EXPERT_ID


def test_permute_invalid_ids_and_zipf_routing():
    rng = np.random.default_rng(9)
    ids, _ = inputs.routing_zipf(rng, 32, 256, 8)
    ids[3, 2] = -5
    ids[7, 0] = 256
    ids[31, 7] = 1 << 30
    st = _status()
    s, inv, off = moe_w2.permute(torch.from_numpy(ids).cuda(), 256, status=st)
    rs, rinv, roff, rst = oracle.permute(ids, 256)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(off.cpu().numpy(), roff)
    assert int(st.item()) == rst == moe_w2.DEV_BAD_EXPERT_ID


def _requant_gpu(t: inputs.Nvfp4Tensors):
    st = _status()
    c, s = moe_w2.requant(torch.from_numpy(t.e2m1).cuda(), torch.from_numpy(t.e4m3).cuda(),
                          torch.from_numpy(t.scale_2).cuda(), status=st)
    return c.cpu().numpy(), s.cpu().numpy(), int(st.item())


def test_requant_small_full_compare():
    t = inputs.nvfp4_tensors(np.random.default_rng(31), 6, 64, 512)
    t.scale_2[1] = np.float32(0.37)          # non power of two
    t.scale_2[2] = np.float32(3.0e38)        # top clamp
    t.scale_2[3] = np.float32(2.0 ** -149)   # subnormal scale_2
    t.e4m3[4, :8] = np.uint8(0x01)           # subnormal e4m3
    t.e4m3[4, 8:16] = np.uint8(0)            # zero scales
    t.e4m3[5, :, ::3] |= np.uint8(0x80)      # negative scales
    c, s, st = _requant_gpu(t)
    rc, rs, rst = oracle.requant(t.e2m1, t.e4m3, t.scale_2)
    assert np.array_equal(s, rs)
    assert np.array_equal(c, rc)
    assert st == rst == 0


def test_requant_adversarial_blocks():
    from tests.test_oracle_requant import ADVERSARIAL, _block_arrays
    n = len(ADVERSARIAL)
    e2m1 = np.zeros((n, 1, 16), np.uint8)
    e4m3 = np.zeros((n, 1, 2), np.uint8)
    s2 = np.zeros(n, np.float32)
    for i, (nib, sc, v) in enumerate(ADVERSARIAL):
        a, b = _block_arrays(nib, sc)
        e2m1[i], e4m3[i], s2[i] = a[0], b[0], np.float32(v)
    t = inputs.Nvfp4Tensors(e2m1, e4m3, s2)
    c, s, st = _requant_gpu(t)
    rc, rs, rst = oracle.requant(e2m1, e4m3, s2)
    assert np.array_equal(s, rs) and np.array_equal(c, rc)
    assert st == rst == moe_w2.DEV_BAD_NVFP4


def test_requant_random_scales_and_patterns():
    rng = np.random.default_rng(33)
    n, rows, K = 64, 8, 256
    e2m1 = inputs.random_bytes(rng, (n, rows, K // 2))
    e4m3 = rng.integers(0, 256, size=(n, rows, K // 16), dtype=np.uint8)
    e4m3[(e4m3 & 0x7F) == 0x7F] = 0x38         # no NaN here
    s2 = (rng.uniform(0.5, 2.0, n) * np.exp2(rng.integers(-60, 60, n))).astype(np.float32)
    t = inputs.Nvfp4Tensors(e2m1, e4m3, s2)
    c, s, st = _requant_gpu(t)
    rc, rs, rst = oracle.requant(e2m1, e4m3, s2)
    assert np.array_equal(s, rs) and np.array_equal(c, rc) and st == rst == 0


@pytest.fixture(scope="module")
def requant_workload():
    return inputs.requant_inputs()


def test_requant_full_workload_every_block(requant_workload):
    """All 256 experts (gate/up and down tensors, ~302 M blocks of 32) on the GPU,
    every code byte and scale byte compared with the OpenMP build of the oracle."""
    gu, dn = requant_workload
    for t in (gu, dn):
        c, s, st = _requant_gpu(t)
        assert st == 0
        rc, rs, rst = oracle.requant(t.e2m1, t.e4m3, t.scale_2, parallel=True)
        assert rst == 0
        assert np.array_equal(s, rs)
        assert np.array_equal(c, rc)
