"""GPU parity of the decode path (T <= 64) of moe_w2_forward against the oracle.

Bar: relative L2 <= 1e-3 and max abs <= 1e-2 * max|oracle| on the layer output
(bf16), over every token of every case (the full-size T = 32 step through the
OpenMP build of the oracle); repeated runs must be bitwise identical.  Both
decode kernels also run activations with a wide dynamic range inside each
32-element block (one element 2^8..2^12 times the rest, blocks mixing zeros with
large values) and layers whose h has one large element per 32.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.helpers import assert_close_layer, from_dev_bf16, planes_to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _run(lay: inputs.LayerInputs, planes_dev=None, ids=None, weights=None):
    planes_dev = planes_dev or planes_to_dev(lay.planes)
    ids = lay.ids if ids is None else ids
    weights = lay.weights if weights is None else weights
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe_w2.forward(to_dev_bf16(lay.x), torch.from_numpy(ids).cuda(), torch.from_numpy(weights).cuda(),
                       planes_dev, status=st)
    return from_dev_bf16(y), int(st.item())


@pytest.fixture
def stream_kernel():
    # the stream-K kernel for steps of at most 16 pairs (H, I multiples of 512)
    with moe_w2.decode_stream():
        yield

def test_tiny_config_all_tokens():
    lay = inputs.layer_inputs(inputs.CONFIGS["tiny"])
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == 0
    assert_close_layer(y, ref, "tiny")


# Steps of more than 16 pairs with H and I multiples of 512 run the block-scaled
# tcgen05 kernel, at most 16 pairs the stream-K kernel, and H or I not a
# multiple of 512 the mma.sync kernel (all three kinds are listed).
@pytest.mark.parametrize("H,I,E,k,T,seed", [(256, 256, 4, 1, 1, 1), (512, 256, 8, 2, 3, 2), (768, 512, 16, 4, 17, 3),
                                            (1024, 768, 8, 8, 64, 4), (512, 512, 2, 2, 64, 5),
                                            (256, 1024, 64, 16, 40, 6), (1024, 512, 16, 4, 17, 7),
                                            (512, 1024, 64, 16, 40, 8), (1536, 1024, 8, 8, 64, 9),
                                            (512, 512, 4, 1, 17, 10)])
def test_small_shapes_all_tokens(H, I, E, k, T, seed):
    # (512,512,2,2,64): each expert gets ~64 pairs -> several tiles per expert
    lay = inputs.small_layer_inputs(H, I, E, k, T, seed)
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == 0
    assert_close_layer(y, ref, f"H{H} I{I} E{E} k{k} T{T}")


def test_duplicates_invalid_ids_and_zero_weights():
    lay = inputs.small_layer_inputs(512, 256, 8, 4, 6, 11)
    ids = lay.ids.copy()
    w = lay.weights.copy()
    ids[0] = [3, 3, 3, 1]          # the same expert three times
    ids[1, 2] = -1                  # invalid -> contributes 0
    ids[2, 0] = 8
    w[3, :] = 0.0                   # a token with all-zero weights
    y, st = _run(lay, ids=ids, weights=w)
    ref, rst = oracle.forward_tokens(lay.x, ids, w, lay.planes)
    assert st == rst == moe_w2.DEV_BAD_EXPERT_ID
    assert_close_layer(y, ref, "duplicates/invalid")
    assert np.all(y[3] == 0)


@pytest.mark.parametrize("H,I,T,seed,kernel", [(512, 256, 4, 12, "decode_mma_kernel"),
                                                (512, 512, 16, 13, "decode_layer_kernel"),
                                                (512, 512, 4, 14, "decode_stream_kernel")])
def test_bad_scale_bytes_zero_their_blocks(H, I, T, seed, kernel):
    lay = inputs.small_layer_inputs(H, I, 4, 2, T, seed)
    planes = {k: v.copy() for k, v in lay.planes.items()}
    planes["w13_scales"][1, 5, 3] = 0
    planes["w2_scales"][2, 7, 1] = 255
    planes["w2_scales"][0, 100, 0] = 253
    planes["w13_scales"][3, 2 * I - 1, H // 32 - 1] = 0   # last block of the last up row
    with moe_w2.decode_stream(kernel == "decode_stream_kernel"):
        assert moe_w2.decode_kernel(T, 2, H, I) == kernel
        y, st = _run(lay, planes_dev=planes_to_dev(planes))
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, planes)
    assert rst == moe_w2.DEV_BAD_SCALE
    assert st & moe_w2.DEV_BAD_SCALE
    assert_close_layer(y, ref, "bad scales")


# Steps of at most 16 pairs with H and I multiples of 512, where the stream-K
# kernel is selected (one CTA per SM): small layers leave most CTAs without
# chunks, and the larger ones cut row blocks between CTAs at many places.
@pytest.mark.parametrize("H,I,E,k,T,seed", [(512, 512, 8, 2, 1, 70), (512, 512, 4, 1, 1, 71),
                                            (1024, 512, 16, 4, 4, 72), (512, 1024, 64, 16, 1, 73),
                                            (1536, 1024, 8, 8, 2, 74), (2048, 1536, 32, 8, 2, 75),
                                            (6144, 2048, 16, 4, 4, 76), (4096, 2048, 32, 8, 1, 77)])
@pytest.mark.usefixtures("stream_kernel")
def test_stream_kernel_shapes_all_tokens(H, I, E, k, T, seed):
    assert moe_w2.decode_kernel(T, k, H, I) == "decode_stream_kernel"
    lay = inputs.small_layer_inputs(H, I, E, k, T, seed)
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == 0
    assert_close_layer(y, ref, f"stream kernel H{H} I{I} E{E} k{k} T{T}")


@pytest.mark.usefixtures("stream_kernel")
def test_stream_kernel_several_tiles_per_expert_and_invalid_ids():
    # expert 2 takes 7 of the 16 pairs (two tiles of at most four), expert 5 four;
    # ids -1 and 9 (E = 8) are left out and flagged
    lay = inputs.small_layer_inputs(1024, 512, 8, 4, 4, 78)
    ids = np.array([[2, 2, 2, 5], [2, 2, 5, 5], [5, -1, 1, 2], [2, 9, 0, 3]], dtype=np.int32)
    assert moe_w2.decode_kernel(4, 4, 1024, 512) == "decode_stream_kernel"
    y, st = _run(lay, ids=ids)
    ref, rst = oracle.forward_tokens(lay.x, ids, lay.weights, lay.planes)
    assert st == rst == moe_w2.DEV_BAD_EXPERT_ID
    assert_close_layer(y, ref, "stream kernel, several tiles per expert, invalid ids")


@pytest.mark.usefixtures("stream_kernel")
def test_stream_kernel_no_valid_pair_gives_zeros():
    lay = inputs.small_layer_inputs(512, 512, 8, 2, 2, 79)
    assert moe_w2.decode_kernel(2, 2, 512, 512) == "decode_stream_kernel"
    ids = np.full((2, 2), -1, dtype=np.int32)
    y, st = _run(lay, ids=ids)
    assert st == moe_w2.DEV_BAD_EXPERT_ID
    assert np.all(y == 0)


@pytest.fixture(scope="module")
def decode_t32():
    lay = inputs.layer_inputs(inputs.CONFIGS["decode_t32"])
    return lay, planes_to_dev(lay.planes)


@pytest.mark.parametrize("kernel", ["decode_mma_kernel", "decode_stream_kernel"])
def test_decode_t1_full_size(kernel):
    lay = inputs.layer_inputs(inputs.CONFIGS["decode_t1"])
    with moe_w2.decode_stream(kernel == "decode_stream_kernel"):
        assert moe_w2.decode_kernel(1, 8, 6144, 2048) == kernel
        y, st = _run(lay)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == 0
    assert_close_layer(y, ref, f"decode_t1 full size, {kernel}")


def test_decode_t32_full_size_all_tokens(decode_t32):
    lay, pd = decode_t32
    y, st = _run(lay, planes_dev=pd)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes, parallel=True)
    assert st == rst == 0
    assert_close_layer(y, ref, "decode_t32 full size, all 32 tokens")


# Wide in-block dynamic range.  T = 4 top-2 (8 pairs) runs the stream-K kernel
# or, deselected, the mma.sync kernel (bf16 activations); T = 16 top-2 (32
# pairs) the block-scaled one: it and the stream-K kernel take activations as
# e2m1 digit rows with one scale per 32 elements.
WIDE_CASES = [(4, "decode_mma_kernel"), (4, "decode_stream_kernel"), (16, "decode_layer_kernel")]


@pytest.mark.parametrize("T,kernel", WIDE_CASES)
@pytest.mark.parametrize("mode", ["outlier", "zeros", "both"])
def test_wide_range_activations(T, kernel, mode):
    lay = inputs.small_layer_inputs(512, 512, 8, 2, T, 40 + T)
    x = inputs.wide_range_activations(np.random.default_rng(T), T, 512, mode)
    lay = inputs.LayerInputs(lay.cfg, x, lay.ids, lay.weights, lay.planes)
    with moe_w2.decode_stream(kernel == "decode_stream_kernel"):
        assert moe_w2.decode_kernel(T, 2, 512, 512) == kernel
        y, st = _run(lay)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == 0
    assert_close_layer(y, ref, f"{kernel} wide-range x ({mode}) T={T}")


@pytest.mark.parametrize("T,kernel", WIDE_CASES)
def test_wide_range_h(T, kernel):
    lay = inputs.small_layer_inputs(512, 512, 8, 2, T, 50 + T)
    planes = inputs.boost_gate_up_rows(np.random.default_rng(T), lay.planes, boost=4)
    with moe_w2.decode_stream(kernel == "decode_stream_kernel"):
        assert moe_w2.decode_kernel(T, 2, 512, 512) == kernel
        y, st = _run(lay, planes_dev=planes_to_dev(planes))
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, planes)
    assert st == rst == 0
    assert_close_layer(y, ref, f"{kernel} wide-range h T={T}")


@pytest.mark.parametrize("name", ["decode_t1", "decode_t32"])
def test_full_size_wide_range(name, decode_t32):
    # the full-size layers with outlier activations and h outliers at once
    lay = decode_t32[0] if name == "decode_t32" else inputs.layer_inputs(inputs.CONFIGS[name])
    T = lay.x.shape[0]
    x = inputs.wide_range_activations(np.random.default_rng(7), T, lay.x.shape[1], "outlier")
    planes = inputs.boost_gate_up_rows(np.random.default_rng(8), lay.planes, boost=4)
    lay = inputs.LayerInputs(lay.cfg, x, lay.ids, lay.weights, planes)
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, planes, parallel=True)
    assert st == rst == 0
    assert_close_layer(y, ref, f"{name} full size, wide-range x and h, all tokens")


def test_decode_deterministic_repeats(decode_t32):
    lay, pd = decode_t32
    ys = [_run(lay, planes_dev=pd)[0] for _ in range(6)]
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
