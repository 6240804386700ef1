"""GPU parity of moe_w2_forward_cached, the forward behind an expert cache.

The planes hold resident experts in slots and a residency table maps routed
expert ids to slots (negative: not resident).  Checked on the four paths
(mma.sync, block-scaled and stream-K decode, prefill) and on the decode_t1 layer:
  * every expert resident, slots in a random order with free slots full of
    other weights: y bitwise equal to moe_w2_forward over the planes in expert
    order (the replay after a miss reproduces the resident forward), no misses;
  * some experts missing: y within the layer bar of the oracle's cached forward,
    the miss counter equal to the pairs whose expert is missing, no status bit;
  * every expert missing: y = 0, every pair counted;
  * ids past the table and slots past the planes: status bit 1, and the rest of
    y still within the bar.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs, moe_w2
from tests.helpers import assert_close_layer, from_dev_bf16, planes_to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

BAD_EXPERT_ID = 1

# (H, I, E, k, T, stream): mma.sync decode, block-scaled decode, prefill, and
# the stream-K decode kernel (selected by moe_w2_set_decode_stream)
SHAPES = [(256, 256, 8, 4, 2, False), (512, 512, 8, 4, 8, False), (256, 512, 8, 2, 80, False),
          (512, 512, 8, 4, 2, True)]


@pytest.fixture(autouse=True)
def _decode_kernel_choice(request):
    params = getattr(getattr(request.node, "callspec", None), "params", {})
    with moe_w2.decode_stream(bool(params.get("stream", False))):
        yield


def _slot_planes(planes, slot_of, S, rng):
    out = {}
    for name, v in planes.items():
        junk = rng.integers(0, 256, size=(S,) + v.shape[1:], dtype=np.uint8)
        if "scales" in name:
            junk = rng.integers(117, 122, size=junk.shape, dtype=np.uint8)
        for e, s in enumerate(slot_of):
            if 0 <= s < S:
                junk[s] = v[e]
        out[name] = junk
    return out


def _cached(lay, sp_dev, slot_of, ids=None):
    ids = lay.ids if ids is None else ids
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    miss = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe_w2.forward_cached(to_dev_bf16(lay.x), torch.from_numpy(ids).cuda(), torch.from_numpy(lay.weights).cuda(),
                              sp_dev, torch.from_numpy(slot_of).cuda(), misses=miss, status=st)
    return from_dev_bf16(y), int(st.item()), int(miss.item())


def _plain(lay, planes_dev):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = moe_w2.forward(to_dev_bf16(lay.x), torch.from_numpy(lay.ids).cuda(), torch.from_numpy(lay.weights).cuda(),
                       planes_dev, status=st)
    return from_dev_bf16(y), int(st.item())


@pytest.mark.parametrize("H,I,E,k,T,stream", SHAPES)
def test_all_resident_is_bitwise_the_plain_forward(H, I, E, k, T, stream):
    rng = np.random.default_rng(H + T)
    lay = inputs.small_layer_inputs(H, I, E, k, T, 70 + T)
    S = E + 5
    slot_of = rng.permutation(S)[:E].astype(np.int32)
    y_c, st_c, m = _cached(lay, planes_to_dev(_slot_planes(lay.planes, slot_of, S, rng)), slot_of)
    y_p, st_p = _plain(lay, planes_to_dev(lay.planes))
    assert st_c == st_p == 0 and m == 0
    assert np.array_equal(y_c, y_p), f"{moe_w2.forward_path(T, k, S, H, I)}: cached y differs from the plain forward"


@pytest.mark.parametrize("H,I,E,k,T,stream", SHAPES)
def test_missing_experts_contribute_zero_and_are_counted(H, I, E, k, T, stream):
    rng = np.random.default_rng(H + T + 1)
    lay = inputs.small_layer_inputs(H, I, E, k, T, 80 + T)
    S = E
    slot_of = rng.permutation(S).astype(np.int32)
    used = np.unique(lay.ids)
    missing = rng.choice(used, size=max(1, len(used) // 3), replace=False)
    slot_of[missing] = -1
    sp = _slot_planes(lay.planes, slot_of, S, rng)
    y, st, m = _cached(lay, planes_to_dev(sp), slot_of)
    ref, rst, rm = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, sp, slot_of)
    assert st == rst == 0
    assert m == rm == int(np.isin(lay.ids, missing).sum())
    assert_close_layer(y, ref, f"cached, {len(missing)} experts missing, T={T} H={H} I={I}")


@pytest.mark.parametrize("H,I,E,k,T,stream", SHAPES)
def test_every_expert_missing_gives_zero(H, I, E, k, T, stream):
    lay = inputs.small_layer_inputs(H, I, E, k, T, 90 + T)
    slot_of = np.full(E, -1, np.int32)
    y, st, m = _cached(lay, planes_to_dev(lay.planes), slot_of)
    assert st == 0 and m == T * k and (y == 0).all()


@pytest.mark.parametrize("H,I,E,k,T,stream", SHAPES)
def test_ids_past_the_table_and_slots_past_the_planes(H, I, E, k, T, stream):
    rng = np.random.default_rng(H + T + 2)
    lay = inputs.small_layer_inputs(H, I, E, k, T, 100 + T)
    S = E
    slot_of = rng.permutation(S).astype(np.int32)
    far = int(lay.ids[0, 0])
    slot_of[far] = S + 3                       # a slot past the planes
    ids = lay.ids.copy()
    ids[-1, -1] = E + 1                        # an id past the table
    sp = _slot_planes(lay.planes, slot_of, S, rng)
    y, st, m = _cached(lay, planes_to_dev(sp), slot_of, ids=ids)
    ref, rst, rm = oracle.forward_tokens_cached(lay.x, ids, lay.weights, sp, slot_of)
    assert st == rst == BAD_EXPERT_ID and m == rm == 0
    assert_close_layer(y, ref, f"cached, invalid ids and slots, T={T}")


def test_decode_t1_layer_from_a_cache():
    """The decode_t1 layer (H=6144, I=2048, 256 routed experts, top-8) from a cache
    of 24 slots: resident replay bitwise equal to the plain forward; then two of
    the token's experts evicted."""
    cfg = inputs.CONFIGS["decode_t1"]
    lay = inputs.layer_inputs(cfg)
    rng = np.random.default_rng(7)
    routed = lay.ids.reshape(-1)
    others = rng.choice(np.setdiff1d(np.arange(cfg.num_experts), routed), size=16, replace=False)
    resident = np.concatenate([routed, others])
    S = len(resident)
    slots = rng.permutation(S).astype(np.int32)
    slot_of = np.full(cfg.num_experts, -1, np.int32)
    slot_of[resident] = slots
    sp = {n: np.ascontiguousarray(v[resident[np.argsort(slots)]]) for n, v in lay.planes.items()}
    y_c, st_c, m = _cached(lay, planes_to_dev(sp), slot_of)
    y_p, st_p = _plain(lay, planes_to_dev(lay.planes))
    assert st_c == st_p == 0 and m == 0
    assert np.array_equal(y_c, y_p)
    slot_of[routed[[2, 5]]] = -1
    y, st, m = _cached(lay, planes_to_dev(sp), slot_of)
    ref, rst, rm = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, sp, slot_of, parallel=True)
    assert st == rst == 0 and m == rm == 2
    assert_close_layer(y, ref, "decode_t1 from a 24-slot cache, 2 of 8 experts missing")
