"""GPU parity of the FP8 block-128 re-quantizer (moe_w2_requant_fp8), bit-exact.

Codes and UE8M0 bytes compared element by element with the CPU oracle on the
same seeded inputs: small tensors with a ragged last 128-row block, adversarial
blocks (NaN bytes, zero / negative / infinite / subnormal scales, extreme
spreads), and the 16-expert FP8 workload (gate/up 2 x [2048 x 6144] and down
[6144 x 2048] per expert) on every block through the OpenMP build.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.test_oracle_requant_fp8 import ADVERSARIAL

pytestmark = pytest.mark.gpu


def _gpu(t: inputs.Fp8Tensors):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    c, u = moe_w2.requant_fp8(torch.from_numpy(t.w8).cuda(), torch.from_numpy(t.scales).cuda(), status=st)
    return c.cpu().numpy(), u.cpu().numpy(), int(st.item())


def test_small_tensors_ragged_rows():
    t = inputs.fp8_tensors(np.random.default_rng(41), 3, 200, 384)
    t.scales[1, 1, 2] = np.float32(1e-40)       # a subnormal block scale
    t.scales[2, 0, 0] = np.float32(3.0e38)      # near the top of f32
    c, u, st = _gpu(t)
    rc, ru, rst = oracle.requant_fp8(t.w8, t.scales)
    assert np.array_equal(u, ru) and np.array_equal(c, rc) and st == rst == 0


def test_adversarial_blocks():
    n = len(ADVERSARIAL)
    w8 = np.zeros((n, 1, 32), np.uint8)
    sc = np.zeros((n, 1, 1), np.float32)
    for i, (byts, s) in enumerate(ADVERSARIAL):
        w8[i, 0] = byts
        sc[i, 0, 0] = np.float32(s)
    c, u, st = _gpu(inputs.Fp8Tensors(w8, sc))
    rc, ru, rst = oracle.requant_fp8(w8, sc)
    assert np.array_equal(u, ru) and np.array_equal(c, rc)
    assert st == rst == oracle.BAD_NVFP4


def test_random_bytes_any_scale():
    rng = np.random.default_rng(43)
    w8 = rng.integers(0, 256, size=(32, 128, 256), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x40
    sc = (rng.uniform(0.5, 2.0, (32, 1, 2)) * np.exp2(rng.integers(-60, 60, (32, 1, 2)))).astype(np.float32)
    c, u, st = _gpu(inputs.Fp8Tensors(w8, sc))
    rc, ru, rst = oracle.requant_fp8(w8, sc)
    assert np.array_equal(u, ru) and np.array_equal(c, rc) and st == rst == 0


def test_fp8_workload_every_block():
    gu, dn = inputs.requant_fp8_inputs(experts=inputs.REQUANT_FP8_CASES["requant_fp8_16"])
    for t in (gu, dn):
        c, u, st = _gpu(t)
        rc, ru, rst = oracle.requant_fp8(t.w8, t.scales, parallel=True)
        assert st == rst == 0
        assert np.array_equal(u, ru)
        assert np.array_equal(c, rc)
