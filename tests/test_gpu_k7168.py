"""The K = 7168 shape family on the GPU (page "vLLM-Moet wiki", the Kimi-K2.7
paragraph: 384 experts, top-8, H = 7168, loaded through the NVFP4 re-quantizer
with a zero-sign balancing fix).

H = 7168 is 14 x 512, so both decode kernels and the prefill kernels take it:
  * decode T = 1 (mma.sync kernel and, selected, the stream-K kernel), T = 2
    (stream-K kernel), T = 4 and T = 16 (block-scaled kernel), every
    token against the oracle, and prefill T = 72 on sampled tokens; the layer has
    384 routed experts of I = 2048 behind an expert cache holding the step's
    experts plus a few others (moe_w2_forward_cached), as a 384-expert layer
    is served from a cache;
  * the NVFP4 loader on one expert's K = 7168 tensors (gate/up [2048 x 7168],
    down [7168 x 2048]) whose exact zeros are all +0, with and without zero-sign
    balancing, bit-exact on every block.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.helpers import assert_close_layer, from_dev_bf16, planes_to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

H, I, E, K_TOP = 7168, 2048, 384, 8


@pytest.mark.parametrize("T,path", [(1, moe_w2.PATH_DECODE_MMA), (1, moe_w2.PATH_DECODE_STREAM),
                                    (2, moe_w2.PATH_DECODE_STREAM), (4, moe_w2.PATH_DECODE_BLOCK_SCALED),
                                    (16, moe_w2.PATH_DECODE_BLOCK_SCALED), (72, moe_w2.PATH_PREFILL)])
def test_kimi_shaped_layer(T, path):
    with moe_w2.decode_stream(path == moe_w2.PATH_DECODE_STREAM):
        _kimi_shaped_layer(T, path)


def _kimi_shaped_layer(T, path):
    cfg = inputs.LayerConfig(f"k7168_t{T}", H, I, E, K_TOP, T, -10, -6, "zipf", 300 + T)
    lay = inputs.cached_layer_inputs(cfg, extra_slots=8)
    S = lay.planes["w13_codes"].shape[0]
    assert moe_w2.forward_path(T, K_TOP, S, H, I) == path
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    miss = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe_w2.forward_cached(to_dev_bf16(lay.x), torch.from_numpy(lay.ids).cuda(),
                              torch.from_numpy(lay.weights).cuda(), planes_to_dev(lay.planes),
                              torch.from_numpy(lay.slot_of).cuda(), misses=miss, status=st)
    tokens = np.arange(T) if T <= 16 else np.linspace(0, T - 1, 12).astype(np.int64)
    ref, rst, rm = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, lay.planes, lay.slot_of,
                                                tokens=tokens, parallel=True)
    assert int(st.item()) == rst == 0 and int(miss.item()) == rm == 0
    assert_close_layer(from_dev_bf16(y)[tokens], ref, f"K=7168 layer (E=384 top-8, I=2048), T={T}")


@pytest.mark.parametrize("balance", [0, moe_w2.REQUANT_BALANCE_ZERO_SIGNS])
def test_nvfp4_loader_k7168_plus_zero_export(balance):
    rng = np.random.default_rng(71)
    for t in (inputs.plus_zero_nvfp4(rng, 2, I, H), inputs.plus_zero_nvfp4(rng, 1, H, I)):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        c, u = moe_w2.requant(torch.from_numpy(t.e2m1).cuda(), torch.from_numpy(t.e4m3).cuda(),
                              torch.from_numpy(t.scale_2).cuda(), status=st, options=balance)
        rc, ru, rst = oracle.requant(t.e2m1, t.e4m3, t.scale_2, parallel=True, options=balance)
        assert int(st.item()) == rst == 0
        assert np.array_equal(u.cpu().numpy(), ru) and np.array_equal(c.cpu().numpy(), rc)
