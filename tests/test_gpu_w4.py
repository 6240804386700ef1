"""GPU parity of the FP4 layer (moe_w4_forward) against the oracle.

The FP4 layer (page "vLLM-Moet wiki", "The kernels" and "FP4 recovery":
moe_w4_mm) is the MoE forward over NVFP4 experts.  Bar as for the 2-bit layer:
rel L2 <= 1e-3 and max abs <= 1e-2 max|oracle| on every compared token.
  * small shapes on the decode kernel (T <= 64) and the prefill kernels, every
    token, with several scale_2 per tensor;
  * the decode_t1 and decode_t32 layer shapes (H=6144, I=2048, top-8) over 64
    experts, every token; prefill at H=4096 I=2048 over 32 experts, T=1024,
    128 sampled tokens;
  * exactly representable experts with power-of-two scale_2: y bitwise equal
    to moe_w2_forward over the planes the NVFP4 re-quantizer writes for them
    (the same instruction sequence over the same bf16 weights), on both paths;
  * an e4m3 NaN scale: status bit 2 and the oracle's zeroed block;
  * repeated runs bitwise identical.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.helpers import assert_close_layer, from_dev_bf16, planes_to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _w4_dev(planes):
    return {n: torch.from_numpy(np.ascontiguousarray(v)).cuda() for n, v in planes.items()}


def _run(lay, pd=None, ids=None):
    pd = pd or _w4_dev(lay.planes)
    ids = lay.ids if ids is None else ids
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe_w2.forward_w4(to_dev_bf16(lay.x), torch.from_numpy(ids).cuda(), torch.from_numpy(lay.weights).cuda(),
                          pd, status=st)
    return from_dev_bf16(y), int(st.item())


def _layer(H, I, E, k, T, seed, routing="logits"):
    lay = inputs.w4_layer_inputs(inputs.LayerConfig(f"w4_{H}_{I}_{E}_{k}_{T}", H, I, E, k, T, -9, -6, routing, seed))
    rng = np.random.default_rng(seed)
    lay.planes["w13_scale_2"][:] = np.exp2(rng.uniform(-9, -7, size=(E, 2))).astype(np.float32)
    lay.planes["w2_scale_2"][:] = np.exp2(rng.uniform(-9, -7, size=E)).astype(np.float32)
    return lay


@pytest.mark.parametrize("H,I,E,k,T", [(256, 256, 8, 2, 1), (512, 256, 8, 4, 2), (256, 512, 6, 4, 16),
                                       (768, 512, 16, 8, 64), (512, 256, 8, 2, 80), (256, 768, 4, 4, 200)])
def test_small_shapes_every_token(H, I, E, k, T):
    lay = _layer(H, I, E, k, T, 10 + T)
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == 0
    assert_close_layer(y, ref, f"FP4 layer H{H} I{I} E{E} k{k} T{T}")


@pytest.mark.parametrize("T,E", [(1, 64), (32, 64)])
def test_decode_shapes_full_size(T, E):
    lay = inputs.w4_layer_inputs(inputs.LayerConfig(f"w4_decode_t{T}", 6144, 2048, E, 8, T, -10, -6, "zipf", 40 + T))
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, lay.planes, parallel=True)
    assert st == rst == 0
    assert_close_layer(y, ref, f"FP4 layer H6144 I2048 top-8 T{T} over {E} experts, all tokens")


def test_prefill_shape_sampled_tokens():
    lay = inputs.w4_layer_inputs(inputs.LayerConfig("w4_prefill_t1024_e32", 4096, 2048, 32, 8, 1024, -10, -6,
                                                    "logits", 50))
    y, st = _run(lay)
    tok = np.linspace(0, 1023, 128).astype(np.int64)
    ref, rst = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, lay.planes, tokens=tok, parallel=True)
    assert st == rst == 0
    assert_close_layer(y[tok], ref, "FP4 layer H4096 I2048 top-8 T1024 over 32 experts, 128 tokens")


def _representable(rng, E, H, I):
    def part(rows, K):
        nib = rng.choice(np.array([2, 6, 10, 14], np.uint8), size=(E, rows, K))
        e2m1 = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
        k32 = rng.integers(-4, 3, size=(E, rows, K // 32))
        return e2m1, np.repeat(((k32 + 7) << 3).astype(np.uint8), 2, axis=-1)
    a, b = part(2 * I, H)
    c, d = part(H, I)
    return {"w13_e2m1": a, "w13_e4m3": b, "w13_scale_2": np.exp2(rng.integers(-9, -6, size=(E, 2))).astype(np.float32),
            "w2_e2m1": c, "w2_e4m3": d, "w2_scale_2": np.exp2(rng.integers(-9, -6, size=E)).astype(np.float32)}


@pytest.mark.parametrize("T", [2, 80])
def test_representable_experts_bitwise_equal_to_the_2bit_layer(T):
    rng = np.random.default_rng(60 + T)
    E, H, I, k = 8, 512, 256, 2
    p4 = _representable(rng, E, H, I)
    gate = oracle.requant(p4["w13_e2m1"][:, :I], p4["w13_e4m3"][:, :I], p4["w13_scale_2"][:, 0])
    up = oracle.requant(p4["w13_e2m1"][:, I:], p4["w13_e4m3"][:, I:], p4["w13_scale_2"][:, 1])
    dn = oracle.requant(p4["w2_e2m1"], p4["w2_e4m3"], p4["w2_scale_2"])
    p2 = {"w13_codes": np.concatenate([gate[0], up[0]], axis=1),
          "w13_scales": np.concatenate([gate[1], up[1]], axis=1), "w2_codes": dn[0], "w2_scales": dn[1]}
    x = inputs.activations(rng, T, H)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
    xd, idd, wd = to_dev_bf16(x), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y4 = from_dev_bf16(moe_w2.forward_w4(xd, idd, wd, _w4_dev(p4), status=st))
    y2 = from_dev_bf16(moe_w2.forward(xd, idd, wd, planes_to_dev(p2), status=st))
    assert int(st.item()) == 0
    assert np.array_equal(y4, y2), f"T={T}: FP4 layer differs from the 2-bit layer on representable experts"


@pytest.mark.parametrize("T", [4, 96])
def test_nan_scale_is_flagged_and_zeroed(T):
    lay = _layer(256, 256, 4, 2, T, 70 + T)
    e = int(lay.ids[0, 0])
    lay.planes["w13_e4m3"][e, 3, 2] = 0x7F
    lay.planes["w2_e4m3"][e, 10, 5] = 0xFF
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == oracle.BAD_SCALE
    assert_close_layer(y, ref, f"FP4 layer with NaN scales, T={T}")


@pytest.mark.parametrize("T", [8, 100])
def test_repeat_runs_are_bitwise_identical(T):
    lay = _layer(512, 512, 8, 4, T, 80 + T)
    pd = _w4_dev(lay.planes)
    ys = [_run(lay, pd)[0] for _ in range(4)]
    assert all(np.array_equal(ys[0], v) for v in ys[1:])
