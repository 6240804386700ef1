"""Pins for the oracle's forward behind an expert cache (CPU only).

What fixes the result (page "vLLM-Moet wiki", BASE-cache paragraph; page "The
v0.24.0 port", section "Our hooks", BASE-cache bullet): the planes hold the
resident experts in slots, a table maps each routed expert to its slot, and a
pair whose expert is missing contributes zero and is counted, so that a replay
with every expert resident reproduces the resident forward bit for bit.  Pins,
each stated differently from the oracle's own code:
  * where an expert sits does not matter: planes re-ordered by a random slot
    permutation (with unused slots holding other weights) give the plain
    forward's y and h bitwise;
  * a missing expert's pair gives what the plain forward gives with that pair's
    router weight 0 (y bitwise), and its h row is zero;
  * the miss count is the number of pairs whose table entry is negative,
    counted here with numpy;
  * ids outside the table and slots past the planes are invalid ids (status
    bit 1), again equal to weight 0.
"""
import numpy as np

import oracle
from bit_moe_expert_w2_gb300 import inputs

BAD_EXPERT_ID = 1


def _slot_planes(planes, slot_of, S, rng):
    """Planes of S slots: expert e's four sections at slot slot_of[e]; free slots random."""
    out = {}
    for name, v in planes.items():
        junk = rng.integers(0, 256, size=(S,) + v.shape[1:], dtype=np.uint8)
        if "scales" in name:
            junk = rng.integers(117, 122, size=junk.shape, dtype=np.uint8)
        for e, s in enumerate(slot_of):
            if s >= 0:
                junk[s] = v[e]
        out[name] = junk
    return out


def test_slot_position_does_not_matter():
    rng = np.random.default_rng(3)
    lay = inputs.small_layer_inputs(256, 256, 6, 3, 5, 31)
    S = 9
    slot_of = rng.permutation(S)[:6].astype(np.int32)
    sp = _slot_planes(lay.planes, slot_of, S, rng)
    y0, h0, st0 = oracle.forward_tokens(lay.x, lay.ids, lay.weights, lay.planes, want_h=True)
    y1, h1, st1, m = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, sp, slot_of, want_h=True)
    assert st0 == st1 == 0 and m == 0
    assert np.array_equal(y0, y1) and np.array_equal(h0, h1)


def test_missing_expert_is_weight_zero_and_counted():
    rng = np.random.default_rng(4)
    lay = inputs.small_layer_inputs(256, 256, 8, 3, 6, 32)
    S = 8
    slot_of = rng.permutation(S).astype(np.int32)
    missing = np.array([1, 4, 6])
    slot_of[missing] = [-1, -7, -(2 ** 31)]
    sp = _slot_planes(lay.planes, slot_of, S, rng)
    y1, h1, st1, m = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, sp, slot_of, want_h=True)
    miss_pair = np.isin(lay.ids, missing)
    assert miss_pair.any() and not miss_pair.all()
    w0 = lay.weights.copy()
    w0[miss_pair] = 0.0
    y0, h0, st0 = oracle.forward_tokens(lay.x, lay.ids, w0, lay.planes, want_h=True)
    assert st0 == st1 == 0
    assert m == int(miss_pair.sum())
    assert np.array_equal(y0, y1)
    assert (h1[miss_pair] == 0).all() and np.array_equal(h1[~miss_pair], h0[~miss_pair])


def test_every_expert_missing_gives_zero():
    lay = inputs.small_layer_inputs(256, 256, 4, 2, 3, 33)
    slot_of = np.full(4, -1, np.int32)
    y, st, m = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, lay.planes, slot_of)
    assert st == 0 and m == lay.ids.size and (y == 0).all()


def test_out_of_table_ids_and_slots_are_invalid():
    rng = np.random.default_rng(5)
    lay = inputs.small_layer_inputs(256, 256, 4, 2, 4, 34)
    ids = lay.ids.copy()
    ids[0, 0] = 4            # past the table
    ids[1, 1] = -3           # negative id
    slot_of = np.array([2, 9, 0, 1], np.int32)   # expert 1 -> slot 9, past S = 4
    S = 4
    sp = _slot_planes(lay.planes, np.where(slot_of < S, slot_of, -1).astype(np.int32), S, rng)
    y1, st1, m = oracle.forward_tokens_cached(lay.x, ids, lay.weights, sp, slot_of)
    bad = (ids < 0) | (ids >= 4) | np.isin(ids, [1])
    assert st1 == BAD_EXPERT_ID and m == 0
    w0 = lay.weights.copy()
    w0[bad] = 0.0
    ids0 = np.where(bad, 0, ids).astype(np.int32)
    y0, st0 = oracle.forward_tokens(lay.x, ids0, w0, lay.planes)
    assert np.array_equal(y0, y1)


def test_parallel_build_agrees():
    rng = np.random.default_rng(6)
    lay = inputs.small_layer_inputs(256, 256, 8, 4, 9, 35)
    slot_of = rng.permutation(8).astype(np.int32)
    slot_of[[0, 5]] = -1
    a = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, lay.planes, slot_of)
    b = oracle.forward_tokens_cached(lay.x, lay.ids, lay.weights, lay.planes, slot_of, parallel=True)
    assert np.array_equal(a[0], b[0]) and a[1:] == b[1:]
