"""GPU parity of the prefill path (T > 64, tcgen05 kernels) of moe_w2_forward.

Bar: relative L2 <= 1e-3 and max abs <= 1e-2 * max|oracle| of the layer output,
over every token for small shapes (several 256-pair tiles with a ragged tail,
many 16-pair tiles, duplicate and invalid ids, bad scale bytes) and, at
T = 8192, over more than 256 tokens chosen so that every expert's first and last
pair (its first and its last, ragged, tile) is checked, through the OpenMP build
of the oracle; repeated runs must be bitwise identical.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.helpers import assert_close_layer, from_dev_bf16, planes_to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _run(lay, planes_dev=None, ids=None, weights=None):
    planes_dev = planes_dev or planes_to_dev(lay.planes)
    ids = lay.ids if ids is None else ids
    weights = lay.weights if weights is None else weights
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe_w2.forward(to_dev_bf16(lay.x), torch.from_numpy(ids).cuda(), torch.from_numpy(weights).cuda(),
                       planes_dev, status=st)
    return from_dev_bf16(y), int(st.item())


@pytest.mark.parametrize("H,I,E,k,T,seed", [
    (512, 256, 8, 2, 96, 1),      # one tile per expert
    (256, 256, 2, 2, 300, 2),     # 300 pairs per expert: two tiles (150 + 150)
    (768, 512, 16, 4, 200, 3),
    (512, 768, 64, 8, 65, 4),     # smallest prefill T, ~8 pairs per expert (16-wide tiles)
    (1024, 256, 4, 8, 400, 5),    # 800 pairs per expert: four tiles
])
def test_small_shapes_all_tokens(H, I, E, k, T, seed):
    lay = inputs.small_layer_inputs(H, I, E, k, T, seed)
    y, st = _run(lay)
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes)
    assert st == rst == 0
    assert_close_layer(y, ref, f"H{H} I{I} E{E} k{k} T{T}")


def test_duplicates_invalid_ids_zero_weights():
    lay = inputs.small_layer_inputs(512, 256, 8, 4, 100, 11)
    ids, w = lay.ids.copy(), lay.weights.copy()
    ids[0] = [5, 5, 5, 5]
    ids[1, 1] = -7
    ids[50, 3] = 8
    w[2] = 0.0
    y, st = _run(lay, ids=ids, weights=w)
    ref, rst = oracle.forward_tokens(lay.x, ids, w, lay.planes)
    assert st == rst == moe_w2.DEV_BAD_EXPERT_ID
    assert_close_layer(y, ref, "prefill duplicates/invalid")
    assert np.all(y[2] == 0)


def test_all_pairs_invalid_gives_zero():
    lay = inputs.small_layer_inputs(256, 256, 4, 2, 70, 12)
    ids = np.full_like(lay.ids, 99)
    y, st = _run(lay, ids=ids)
    assert st == moe_w2.DEV_BAD_EXPERT_ID and np.all(y == 0)


def test_bad_scale_bytes():
    lay = inputs.small_layer_inputs(512, 256, 4, 2, 80, 13)
    planes = {k: v.copy() for k, v in lay.planes.items()}
    planes["w13_scales"][0, 3, 1] = 0
    planes["w2_scales"][3, 9, 2] = 254
    y, st = _run(lay, planes_dev=planes_to_dev(planes))
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, planes)
    assert rst == moe_w2.DEV_BAD_SCALE and st & moe_w2.DEV_BAD_SCALE
    assert_close_layer(y, ref, "prefill bad scales")


@pytest.fixture(scope="module")
def prefill_full():
    lay = inputs.layer_inputs(inputs.CONFIGS["prefill_t8192"])
    return lay, planes_to_dev(lay.planes)


def coverage_tokens(ids: np.ndarray, E: int, extra: int, seed: int) -> np.ndarray:
    """Tokens holding the first and the last pair (in expert-grouped order) of
    every expert, plus `extra` more drawn at random, sorted and unique."""
    T, k = ids.shape
    flat = ids.reshape(-1)
    chosen = set()
    for e in range(E):
        pairs = np.nonzero(flat == e)[0]          # increasing pair index = grouped order
        if pairs.size:
            chosen.update((int(pairs[0]) // k, int(pairs[-1]) // k))
    rng = np.random.default_rng(seed)
    chosen.update(int(t) for t in rng.choice(T, size=extra, replace=False))
    return np.array(sorted(chosen), dtype=np.int64)


def test_prefill_t8192_full_size_covering_every_expert(prefill_full):
    lay, pd = prefill_full
    y, st = _run(lay, planes_dev=pd)
    E = lay.cfg.num_experts
    tokens = coverage_tokens(lay.ids, E, extra=160, seed=3)
    hit = np.unique(lay.ids[tokens])
    assert len(tokens) >= 256 and np.array_equal(hit, np.arange(E))
    ref, rst = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes, tokens=tokens, parallel=True)
    assert st == rst == 0
    assert_close_layer(y[tokens], ref, f"prefill_t8192 full size, {len(tokens)} tokens covering all experts")


def test_prefill_deterministic_repeats(prefill_full):
    lay, pd = prefill_full
    ys = [_run(lay, planes_dev=pd)[0] for _ in range(6)]
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
