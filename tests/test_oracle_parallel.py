"""The OpenMP build of the oracle against its single-threaded build.

Both libraries are compiled from the same ``oracle.c``; the parallel one runs the
loops over independent requant blocks and forward tokens on several threads.
Each block and token is still computed by one thread with the same operations,
so the outputs and status bits must be bitwise identical.  The full-size GPU
parity tests lean on the parallel build, so this pins it to the plain one.
"""
import numpy as np

import oracle
from bit_moe_expert_w2_gb300 import inputs


def test_parallel_build_uses_threads_and_serial_build_one():
    assert oracle.threads(parallel=False) == 1
    assert oracle.threads(parallel=True) >= 1


def test_requant_parallel_bitwise_equal():
    rng = np.random.default_rng(41)
    t = inputs.nvfp4_tensors(rng, 24, 32, 512)
    t.scale_2[1] = np.float32(0.37)            # non power of two: the exact-integer search
    t.scale_2[2] = np.float32(np.nan)          # invalid: codes 0, scale byte 0, status bit
    t.e4m3[3, :, ::5] = np.uint8(0x7F)         # e4m3 NaN blocks
    t.e4m3[4, :4] = np.uint8(0)                # zero blocks
    a = oracle.requant(t.e2m1, t.e4m3, t.scale_2, parallel=False)
    b = oracle.requant(t.e2m1, t.e4m3, t.scale_2, parallel=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2] == oracle.BAD_NVFP4
    ids = rng.integers(0, t.e4m3.size // 2, 5000)
    c = oracle.requant_blocks(t.e2m1, t.e4m3, t.scale_2, ids, parallel=False)
    d = oracle.requant_blocks(t.e2m1, t.e4m3, t.scale_2, ids, parallel=True)
    assert all(np.array_equal(u, v) for u, v in zip(c[:2], d[:2])) and c[2] == d[2]
    assert np.array_equal(c[0], a[0].reshape(-1, 8)[ids]) and np.array_equal(c[1], a[1].reshape(-1)[ids])


def test_forward_parallel_bitwise_equal():
    lay = inputs.small_layer_inputs(512, 256, 8, 4, 24, 42)
    ids, w = lay.ids.copy(), lay.weights.copy()
    ids[2, 1] = -3                             # invalid id: status bit, no contribution
    ids[5] = [1, 1, 6, 1]                      # duplicates
    w[7] = 0.0
    planes = {k: v.copy() for k, v in lay.planes.items()}
    planes["w2_scales"][1, 3, 0] = 255         # invalid scale byte
    a = oracle.forward_tokens(lay.x, ids, w, planes, want_h=True, parallel=False)
    b = oracle.forward_tokens(lay.x, ids, w, planes, want_h=True, parallel=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert a[2] == b[2] == (oracle.BAD_EXPERT_ID | oracle.BAD_SCALE)
    tok = np.array([23, 0, 7, 7, 11])
    c = oracle.forward_tokens(lay.x, ids, w, planes, tokens=tok, parallel=True)
    assert np.array_equal(c[0], a[0][tok])
