"""Pins of the pair-structured layout oracle (oracle/elastic.py) to the already-pinned
plain paths (decode, BASE and E4M3 demotion), not to its own formulas:

* identity locations (value page at its own slot) reproduce the plain decode;
* packing pairs of pages into one slot (two located transitions) and reading them
  through the value block table gives exactly the decode of the same pages demoted in
  place, and the freed slots are never read (garbage written there changes nothing);
* TARGET-BASE-TARGET boundaries give the decode of the equivalent mode table;
* has_base = 0 reads every page as TARGET, ignoring boundaries and the mode table;
* promotion into a fresh slot restores the TARGET bytes exactly;
* the elastic gather equals the plain gather (identity locations; packed pairs against
  the same pages demoted in place; boundaries against the mode table; has_base = 0).
"""

import numpy as np

from oracle import base, decode, demote, elastic, gather

H, G, D, S = 2, 2, 64, 16
N = S * H * D


def _pool(P, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((P, S, H, D)).astype(np.float16)
    x = rng.standard_normal((P, S, H, D)).astype(np.float16)
    v = x.reshape(P, -1).view(np.uint8).copy()          # slot p holds page p (TARGET)
    return k, x, v


def test_identity_locations_reproduce_plain_decode():
    k, x, v = _pool(10, 1)
    rng = np.random.default_rng(2)
    lens = np.array([40, 100], np.int32)
    bt = np.array([[3, 1, 7, 0, 0, 0, 0], [2, 4, 5, 6, 8, 9, 0]], np.int32)
    modes = np.zeros(10, np.uint8)
    v2, modes, sc, _ = elastic.transition(elastic.OP_TO_E4M3, v, [1, 5], None, None, modes,
                                          np.ones((10, H), np.float32), None, H, D)
    v2, modes, _, _ = elastic.transition(elastic.OP_TO_BASE, v2, [4, 7], None, None, modes, sc, None, H, D)
    q = rng.standard_normal((2, H * G, D)).astype(np.float16)
    ref, ref_l = decode.paged_decode(q, k, v2, sc, 1, modes, 0, bt, lens)
    out, l = elastic.paged_decode_elastic(q, k, v2, sc, 1, modes, 0, bt, 2 * bt, None, 1, lens)
    assert np.array_equal(out, ref) and np.array_equal(l, ref_l)
    # in-place transitions equal the plain demotion oracles
    rv, rm, rs = demote.demote_pages(v, [1, 5], np.zeros(10, np.uint8), np.ones((10, H), np.float32), H, D)
    assert np.array_equal(v2[[1, 5]], rv[[1, 5]]) and np.array_equal(sc[[1, 5]], rs[[1, 5]])
    rb, _, _, _ = base.demote_to_base(v, [4, 7], np.zeros(10, np.uint8), H, D)
    assert np.array_equal(v2[[4, 7]], rb[[4, 7]])


def test_packed_pairs_read_like_in_place_demotion():
    P = 12
    k, x, v = _pool(P, 3)
    rng = np.random.default_rng(4)
    lens = np.array([16 * 6, 16 * 5 + 3], np.int32)
    bt = np.array([[0, 1, 2, 3, 4, 5], [6, 7, 8, 9, 10, 0]], np.int32)
    pairs = [(1, 2), (3, 4), (7, 8)]                   # logical pages packed into the first's slot
    modes = np.zeros(P, np.uint8)
    low = np.zeros((3, N), np.uint8)
    # step 1: A pages in place (half 0 of their own slot)
    a = [p for p, _ in pairs]
    vp, modes, _, low_a = elastic.transition(elastic.OP_TO_BASE, v, a, None, None, modes, None, low, H, D)
    # step 2: B pages from their slots into half 1 of the partner's slot
    b = [q for _, q in pairs]
    vp, modes, _, low_b = elastic.transition(elastic.OP_TO_BASE, vp, b, [2 * q for q in b],
                                             [2 * p + 1 for p in a], modes, None, low, H, D)
    vtab = 2 * bt.copy()
    for p, q in pairs:
        vtab[bt == q] = 2 * p + 1
    for _, q in pairs:                                 # freed slots: anything may be written there
        vp[q] = 0x7E
    qv = rng.standard_normal((2, H * G, D)).astype(np.float16)
    out, l = elastic.paged_decode_elastic(qv, k, vp, None, 0, modes, 0, bt, vtab, None, 1, lens)
    # reference: the same pages demoted to BASE in place, plain decode
    rb, rm, rlow, _ = base.demote_to_base(v, a + b, np.zeros(P, np.uint8), H, D)
    ref, ref_l = decode.paged_decode(qv, k, rb, None, 0, rm, 0, bt, lens)
    assert np.array_equal(out, ref) and np.array_equal(l, ref_l)
    assert np.array_equal(low_a, rlow[a]) and np.array_equal(low_b, rlow[b])
    # promote B of the first pair into a fresh slot (11): exact TARGET bytes
    vq, mq, _, _ = elastic.transition(elastic.OP_PROMOTE, vp, [2], [2 * 1 + 1], [2 * 11], modes, None,
                                      low_b[:1], H, D)
    assert mq[2] == 0 and np.array_equal(vq[11], v[2])


def test_boundaries_equal_the_mode_table():
    P = 14
    k, x, v = _pool(P, 5)
    rng = np.random.default_rng(6)
    lens = np.array([16 * 6, 16 * 7 - 5], np.int32)
    bt = np.array([[0, 1, 2, 3, 4, 5, 0], [6, 7, 8, 9, 10, 11, 12]], np.int32)
    bnd = np.array([[2, 5], [1, 7]], np.int32)         # T T B B B T / T B B B B B B
    base_pages = [bt[0, j] for j in range(2, 5)] + [bt[1, j] for j in range(1, 7)]
    vb, modes, _, _ = base.demote_to_base(v, base_pages, np.zeros(P, np.uint8), H, D)
    q = rng.standard_normal((2, H * G, D)).astype(np.float16)
    out, l = elastic.paged_decode_elastic(q, k, vb, None, 0, None, 0, bt, 2 * bt, bnd, 1, lens)
    ref, ref_l = decode.paged_decode(q, k, vb, None, 0, modes, 0, bt, lens)
    assert np.array_equal(out, ref) and np.array_equal(l, ref_l)


def test_has_base_zero_reads_target_everywhere():
    P = 8
    k, x, v = _pool(P, 7)
    rng = np.random.default_rng(8)
    lens = np.array([100], np.int32)
    bt = np.array([[0, 2, 4, 6, 1, 3, 5]], np.int32)
    q = rng.standard_normal((1, H * G, D)).astype(np.float16)
    junk_modes = np.full(P, 2, np.uint8)
    out, l = elastic.paged_decode_elastic(q, k, v, None, 0, junk_modes, 2, bt, 2 * bt,
                                          np.array([[0, 7]], np.int32), 0, lens)
    ref, ref_l = decode.paged_decode(q, k, v, None, 0, None, 0, bt, lens)
    assert np.array_equal(out, ref) and np.array_equal(l, ref_l)


def _gather_pair_case():
    """Pairs of E4M3 and BASE pages packed into shared slots (two located transitions),
    with the in-place demotion of the same pages as the reference pool."""
    P = 12
    k, x, v = _pool(P, 9)
    bt = np.array([[0, 1, 2, 3, 4, 5], [6, 7, 8, 9, 10, 11]], np.int32)
    modes = np.zeros(P, np.uint8)
    sc = np.ones((P, H), np.float32)
    # E4M3 pair (1, 2) and BASE pair (7, 8): A in place, then B into half 1 of A's slot
    vp, modes, sc, _ = elastic.transition(elastic.OP_TO_E4M3, v, [1], None, None, modes, sc, None, H, D)
    vp, modes, sc, _ = elastic.transition(elastic.OP_TO_E4M3, vp, [2], [4], [3], modes, sc, None, H, D)
    vp, modes, sc, _ = elastic.transition(elastic.OP_TO_BASE, vp, [7], None, None, modes, sc, None, H, D)
    vp, modes, sc, _ = elastic.transition(elastic.OP_TO_BASE, vp, [8], [16], [15], modes, sc, None, H, D)
    vtab = 2 * bt.copy()
    vtab[0, 2] = 3
    vtab[1, 2] = 15
    vp[2] = 0x7E                                        # freed slots: never read
    vp[8] = 0x7E
    rv, rm, rs = demote.demote_pages(v, [1, 2], np.zeros(P, np.uint8), np.ones((P, H), np.float32), H, D)
    rb, rmb, _, _ = base.demote_to_base(rv, [7, 8], rm, H, D)
    return k, vp, modes, sc, bt, vtab, rb, rmb, rs


def test_elastic_gather_identity_locations_is_the_plain_gather():
    k, x, v = _pool(10, 11)
    modes = np.zeros(10, np.uint8)
    v2, modes, sc, _ = elastic.transition(elastic.OP_TO_E4M3, v, [1, 5], None, None, modes,
                                          np.ones((10, H), np.float32), None, H, D)
    v2, modes, _, _ = elastic.transition(elastic.OP_TO_BASE, v2, [4, 7], None, None, modes, sc, None, H, D)
    bt = np.array([[3, 1, 7, 0], [2, 4, 5, 6]], np.int32)
    pr = np.array([[0, 0, 3], [1, 1, 3]])
    ek, ev, ei = elastic.gather_prefill_elastic(k, v2, sc, 1, modes, 0, bt, 2 * bt, None, 1, pr)
    rk, rv, ri = gather.gather_prefill(k, v2, sc, 1, modes, 0, bt, pr)
    assert np.array_equal(ek.view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(ev.view(np.uint16), rv.view(np.uint16)) and np.array_equal(ei, ri)


def test_elastic_gather_of_packed_pairs_is_the_gather_of_in_place_demotion():
    k, vp, modes, sc, bt, vtab, rb, rmb, rs = _gather_pair_case()
    pr = np.array([[0, 0, 6], [1, 0, 6]])
    ek, ev, _ = elastic.gather_prefill_elastic(k, vp, sc, 1, modes, 0, bt, vtab, None, 1, pr)
    rk, rv, _ = gather.gather_prefill(k, rb, rs, 1, rmb, 0, bt, pr)
    assert np.array_equal(ek.view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(ev.view(np.uint16), rv.view(np.uint16))


def test_elastic_gather_boundaries_and_has_base():
    P = 14
    k, x, v = _pool(P, 12)
    bt = np.array([[0, 1, 2, 3, 4, 5, 0], [6, 7, 8, 9, 10, 11, 12]], np.int32)
    bnd = np.array([[2, 5], [1, 7]], np.int32)
    base_pages = [bt[0, j] for j in range(2, 5)] + [bt[1, j] for j in range(1, 7)]
    vb, modes, _, _ = base.demote_to_base(v, base_pages, np.zeros(P, np.uint8), H, D)
    pr = np.array([[0, 0, 6], [1, 0, 7]])
    ek, ev, _ = elastic.gather_prefill_elastic(k, vb, None, 0, None, 0, bt, 2 * bt, bnd, 1, pr)
    rk, rv, _ = gather.gather_prefill(k, vb, None, 0, modes, 0, bt, pr)
    assert np.array_equal(ev.view(np.uint16), rv.view(np.uint16))
    # has_base = 0: the original TARGET pool, modes and boundaries ignored
    ek, ev, _ = elastic.gather_prefill_elastic(k, v, None, 0, np.full(P, 2, np.uint8), 2, bt, 2 * bt, bnd, 0, pr)
    rk, rv, _ = gather.gather_prefill(k, v, None, 0, None, 0, bt, pr)
    assert np.array_equal(ev.view(np.uint16), rv.view(np.uint16))
