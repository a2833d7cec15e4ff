"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: hand-worked
golden values, closed forms, invariants, brute force on tiny inputs, or a
library routine (numpy / scipy) in a special case that reduces to it.  The
sources are the OasisKV pages: "Pith review of OasisKV" (pith.science),
section "What carries the argument" (shared attention kernel, min/max
summaries, head-wise top-K of all logical blocks, capped LRS eviction) and
"Assumptions & free parameters" (B = 16, K = 128, fetch ratio, summaries at
1/16 of KV); the agihunt summary's fetch-cap ablation.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from tests._bf16 import to_bits, to_float

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def make_store(keys, vals, B):
    """host_kv [1][1][NB][2][B][d] from per-token key/value rows (padded)."""
    keys = np.asarray(keys, dtype=np.float32)
    vals = np.asarray(vals, dtype=np.float32)
    n, d = keys.shape
    nb = -(-n // B)
    kv = np.zeros((1, 1, nb, 2, B, d), dtype=np.float32)
    for t in range(n):
        kv[0, 0, t // B, 0, t % B] = keys[t]
        kv[0, 0, t // B, 1, t % B] = vals[t]
    return to_bits(kv)


# ----------------------------------------------------------------- summaries
def test_summary_min_max_and_tail_mask():
    rng = np.random.default_rng(0)
    R, H, NB, B, d = 2, 3, 5, 16, 128
    kv = rng.standard_normal((R, H, NB, 2, B, d)).astype(np.float32)
    lens = np.array([5 * 16, 3 * 16 + 7], dtype=np.int32)
    # plant extreme values past request 1's context: they must not show up
    kv[1, :, 3, 0, 7:] = 1e4
    kv[1, :, 4, 0, :] = -1e4
    bits = to_bits(kv)
    s = oracle.summary_build(bits, lens)
    kf = to_float(bits)
    for r in range(R):
        nb = -(-lens[r] // B)
        for b in range(nb):
            valid = min(B, lens[r] - b * B)
            blk = kf[r, :, b, 0, :valid]                     # [H][valid][d]
            np.testing.assert_array_equal(to_float(s[r, :, b, 0]), blk.min(axis=1))
            np.testing.assert_array_equal(to_float(s[r, :, b, 1]), blk.max(axis=1))
    # blocks past the context are left untouched (zeros here)
    assert not s[1, :, 4].any()


def test_summary_is_one_sixteenth_of_kv():
    # min + max rows (2*d values) per block vs 2*B*d values of keys+values
    B, d = 16, 128
    assert (2 * d) / (2 * B * d) == 1.0 / 16


# ------------------------------------------------------------------- scores
def test_score_hand_worked():
    cases = json.load(open(os.path.join(GOLD, "quest_bound_hand.json")))["cases"]
    for c in cases:
        kv = make_store(c["keys"], np.zeros_like(c["keys"]), B=2)
        lens = np.array([2], dtype=np.int32)
        summ = oracle.summary_build(kv, lens)
        np.testing.assert_array_equal(to_float(summ[0, 0, 0, 0]), c["min"])
        np.testing.assert_array_equal(to_float(summ[0, 0, 0, 1]), c["max"])
        qd = to_bits(np.asarray(c["q"], dtype=np.float32).reshape(1, 1, 2))
        s = oracle.score_rh(summ, lens, qd, 0, 0, B=2)
        assert s[0] == np.float32(c["score"])
        qk = to_float(qd)[0, 0] @ to_float(kv)[0, 0, 0, 0].T
        assert qk.max() == c["max_qk"]
        assert s[0] >= qk.max()


def test_score_upper_bounds_every_key_and_sums_group():
    rng = np.random.default_rng(1)
    R, Hkv, G, NB, B, d = 1, 2, 4, 12, 16, 128
    kv = to_bits(rng.standard_normal((R, Hkv, NB, 2, B, d)))
    lens = np.array([NB * B - 5], dtype=np.int32)
    summ = oracle.summary_build(kv, lens)
    qd = to_bits(rng.standard_normal((R, Hkv * G, d)) * 2.0)
    kf, qf = to_float(kv).astype(np.float64), to_float(qd).astype(np.float64)
    for h in range(Hkv):
        s = oracle.score_rh(summ, lens, qd, 0, h, B)
        single = []
        for g in range(G):
            only = qd.copy()
            for g2 in range(G):
                if g2 != g:
                    only[0, h * G + g2] = 0
            single.append(oracle.score_rh(summ, lens, only, 0, h, B))
            for b in range(NB):
                valid = min(B, lens[0] - b * B)
                qk = kf[0, h, b, 0, :valid] @ qf[0, h * G + g]
                # the bound holds in exact arithmetic; allow the one fp32 rounding
                assert single[-1][b] >= qk.max() - 1e-6 * abs(qk.max())
        # the group score is the sum of the per-head bounds
        np.testing.assert_allclose(s, np.sum(single, axis=0), rtol=1e-6)


def test_score_two_drafts_hand_worked():
    gold = json.load(open(os.path.join(GOLD, "quest_bound_hand.json")))
    for c in gold["draft_cases"]:
        kv = make_store(c["keys"], np.zeros_like(c["keys"]), B=2)
        lens = np.array([2], dtype=np.int32)
        summ = oracle.summary_build(kv, lens)
        qd = to_bits(np.asarray(c["drafts"], dtype=np.float32).reshape(len(c["drafts"]), 1, 1, 2))
        s = oracle.score_rh(summ, lens, qd, 0, 0, B=2)
        assert s[0] == np.float32(c["score"])
        kf = to_float(kv)[0, 0, 0, 0].astype(np.float64)
        best = sum((to_float(qd)[e, 0, 0] @ kf.T).max() for e in range(qd.shape[0]))
        assert best == c["sum_max_qk"]
        assert s[0] >= best


def test_score_drafts_bound_each_draft_and_add_up():
    # Several drafts on a multi-request layer (so a wrong draft or request
    # stride shows): the score bounds the sum over drafts of each draft's
    # best key in every block, equals the sum of the single-draft scores, and
    # two identical drafts give exactly twice the single-draft score.
    rng = np.random.default_rng(4)
    R, Hkv, G, NB, B, d, D = 3, 2, 2, 10, 16, 128, 3
    kv = to_bits(rng.standard_normal((R, Hkv, NB, 2, B, d)))
    lens = np.array([NB * B, NB * B - 21, 37], dtype=np.int32)
    summ = oracle.summary_build(kv, lens)
    qd = to_bits(rng.standard_normal((D, R, Hkv * G, d)) * 1.5)
    kf, qf = to_float(kv).astype(np.float64), to_float(qd).astype(np.float64)
    for r in range(R):
        nb = -(-lens[r] // B)
        for h in range(Hkv):
            s = oracle.score_rh(summ, lens, qd, r, h, B)
            single = [oracle.score_rh(summ, lens, np.ascontiguousarray(qd[e]), r, h, B)
                      for e in range(D)]
            np.testing.assert_allclose(s[:nb], np.sum(single, axis=0)[:nb], rtol=1e-6)
            assert np.isneginf(s[nb:]).all()
            for b in range(nb):
                valid = min(B, lens[r] - b * B)
                best = sum((kf[r, h, b, 0, :valid] @ qf[e, r, h * G:(h + 1) * G].T).max(axis=0).sum()
                           for e in range(D))
                assert s[b] >= best - 1e-6 * abs(best)
            twice = oracle.score_rh(summ, lens, np.stack([qd[1], qd[1]]), r, h, B)
            np.testing.assert_array_equal(twice, 2 * single[1])


def test_score_single_token_block_is_exact_dot():
    # one valid token: min = max = k, so the bound collapses to q.k
    rng = np.random.default_rng(2)
    d, B = 128, 16
    kv = to_bits(rng.standard_normal((1, 1, 3, 2, B, d)))
    lens = np.array([2 * B + 1], dtype=np.int32)
    summ = oracle.summary_build(kv, lens)
    qd = to_bits(rng.standard_normal((1, 1, d)))
    s = oracle.score_rh(summ, lens, qd, 0, 0, B)
    exact = np.dot(to_float(qd)[0, 0].astype(np.float64),
                   to_float(kv)[0, 0, 2, 0, 0].astype(np.float64))
    assert s[2] == np.float32(exact)
    assert np.isneginf(s[3:]).all() if s.size > 3 else True


def test_score_past_context_is_minus_inf():
    rng = np.random.default_rng(3)
    kv = to_bits(rng.standard_normal((1, 1, 6, 2, 16, 128)))
    lens = np.array([40], dtype=np.int32)          # 3 blocks
    summ = oracle.summary_build(kv, lens)
    s = oracle.score_rh(summ, lens, to_bits(np.ones((1, 1, 128))), 0, 0, 16)
    assert np.isfinite(s[:3]).all() and np.isneginf(s[3:]).all()


# -------------------------------------------------------------------- top-K
def brute_topk(s, K):
    """Rank of b = number of blocks that beat it (higher score, or equal score
    and lower id); top-K = blocks of rank < K, listed by rank."""
    n = len(s)
    rank = [sum(1 for c in range(n) if s[c] > s[b] or (s[c] == s[b] and c < b))
            for b in range(n)]
    out = [-1] * K
    for b in range(n):
        if rank[b] < K:
            out[rank[b]] = b
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    for n in range(0, 9):
        s = rng.choice([-1.5, 0.0, 0.25, 2.0], size=n).astype(np.float32)
        for K in (1, 3, 8, 10):
            assert list(oracle.topk_rh(s, n, K)) == brute_topk(list(s), K)


def test_topk_exhaustive_subset_is_best():
    # The chosen set maximises the score sum among all K-subsets (distinct scores).
    rng = np.random.default_rng(7)
    s = rng.permutation(9).astype(np.float32)
    got = set(oracle.topk_rh(s, 9, 4))
    best = max(itertools.combinations(range(9), 4), key=lambda c: s[list(c)].sum())
    assert got == set(best)


def test_topk_large_matches_partition():
    rng = np.random.default_rng(8)
    s = rng.standard_normal(1024).astype(np.float32)
    t = oracle.topk_rh(s, 1024, 128)
    np.testing.assert_array_equal(t, np.argsort(-s, kind="stable")[:128])


# ---------------------------------------------------------------- attention
def dense_reference(kf, vf, x, scale):
    """Library special case: scipy softmax over all tokens, numpy weighted sum."""
    w = scipy.special.softmax((kf @ x) * scale)
    return w @ vf


def rand_layer(rng, R, Hkv, G, NB, B=16, d=128):
    kv = to_bits(rng.standard_normal((R, Hkv, NB, 2, B, d)))
    q = to_bits(rng.standard_normal((R, Hkv * G, d)))
    qd = to_bits(rng.standard_normal((R, Hkv * G, d)))
    return kv, q, qd


def test_attention_full_residency_equals_dense_softmax():
    rng = np.random.default_rng(10)
    R, Hkv, G, NB, B, d = 2, 2, 4, 8, 16, 128
    kv, q, qd = rand_layer(rng, R, Hkv, G, NB)
    lens = np.array([NB * B, NB * B - 9], dtype=np.int32)
    res = np.stack([np.stack([rng.permutation(NB) for _ in range(Hkv)])
                    for _ in range(R)]).astype(np.int32)
    kf, qf, qdf = to_float(kv).astype(np.float64), to_float(q), to_float(qd)
    for r in range(R):
        for h in range(Hkv):
            o = oracle.attention_rh(kv, lens, res, q, qd, r, h)
            keys = kf[r, h, :, 0].reshape(-1, d)[:lens[r]]
            vals = kf[r, h, :, 1].reshape(-1, d)[:lens[r]]
            for g in range(G):
                j = h * G + g
                np.testing.assert_allclose(
                    o[0, g], dense_reference(keys, vals, qf[r, j], 1 / math.sqrt(d)),
                    rtol=1e-5, atol=1e-6)
                np.testing.assert_allclose(
                    o[1, g], dense_reference(keys, vals, qdf[r, j], 1 / math.sqrt(d)),
                    rtol=1e-5, atol=1e-6)


def test_attention_two_token_closed_form_checks_scale():
    d, B = 128, 16
    rng = np.random.default_rng(11)
    keys = rng.standard_normal((2, d))
    vals = rng.standard_normal((2, d))
    kv = make_store(keys, vals, B)
    kf = to_float(kv)[0, 0, 0]
    x = to_bits(rng.standard_normal((1, 1, d)))
    xf = to_float(x)[0, 0].astype(np.float64)
    res = np.array([[[0]]], dtype=np.int32)
    o = oracle.attention_rh(kv, np.array([2], np.int32), res, x, x, 0, 0)
    delta = (xf @ kf[0, 1] - xf @ kf[0, 0]) / math.sqrt(d)
    want = (kf[1, 0] + math.exp(delta) * kf[1, 1]) / (1 + math.exp(delta))
    np.testing.assert_allclose(o[0, 0], want, rtol=1e-6, atol=1e-7)


def test_attention_constant_values_and_identical_keys():
    rng = np.random.default_rng(12)
    d, B, NB = 128, 16, 4
    c = rng.standard_normal(d)
    keys = rng.standard_normal((NB * B, d))
    kv = make_store(keys, np.tile(c, (NB * B, 1)), B)
    res = np.arange(NB, dtype=np.int32).reshape(1, 1, NB)
    x = to_bits(rng.standard_normal((1, 1, d)))
    o = oracle.attention_rh(kv, np.array([NB * B], np.int32), res, x, x, 0, 0)
    np.testing.assert_allclose(o[0, 0], to_float(to_bits(c)), rtol=1e-6, atol=1e-7)
    # identical keys: uniform weights, output = mean of the values
    vals = rng.standard_normal((NB * B, d))
    kv2 = make_store(np.tile(keys[0], (NB * B, 1)), vals, B)
    o2 = oracle.attention_rh(kv2, np.array([NB * B], np.int32), res, x, x, 0, 0)
    np.testing.assert_allclose(o2[0, 0], to_float(to_bits(vals)).mean(axis=0),
                               rtol=1e-5, atol=1e-6)


def test_attention_masks_tail_and_empty_slots_and_routes_heads():
    rng = np.random.default_rng(13)
    R, Hkv, G, NB, B, d = 1, 2, 4, 6, 16, 128
    kvf = rng.standard_normal((R, Hkv, NB, 2, B, d)).astype(np.float32)
    kvf[0, :, 4, :, 5:] = 1e4                      # past the context (ctx = 4*16+5)
    kvf[0, 1, :, 1] = 7.0                          # KV head 1 values constant 7
    kv = to_bits(kvf)
    lens = np.array([4 * B + 5], dtype=np.int32)
    q = to_bits(rng.standard_normal((R, Hkv * G, d)))
    qd = to_bits(rng.standard_normal((R, Hkv * G, d)))
    res = np.array([[[4, -1, 1, -1], [0, 4, -1, 2]]], dtype=np.int32)
    kf = to_float(kv).astype(np.float64)
    o = oracle.attention_rh(kv, lens, res, q, qd, 0, 0)
    keys = np.concatenate([kf[0, 0, 4, 0, :5], kf[0, 0, 1, 0]])
    vals = np.concatenate([kf[0, 0, 4, 1, :5], kf[0, 0, 1, 1]])
    for g in range(G):
        np.testing.assert_allclose(
            o[1, g], dense_reference(keys, vals, to_float(qd)[0, g], 1 / math.sqrt(d)),
            rtol=1e-5, atol=1e-6)
    o1 = oracle.attention_rh(kv, lens, res, q, qd, 0, 1)
    np.testing.assert_allclose(o1, 7.0, rtol=1e-6)     # heads 4..7 read KV head 1
    # nothing resident -> zeros
    empty = np.full((1, Hkv, 4), -1, dtype=np.int32)
    assert not oracle.attention_rh(kv, lens, empty, q, qd, 0, 0).any()
    # slot order does not matter
    perm = res[:, :, ::-1].copy()
    np.testing.assert_allclose(oracle.attention_rh(kv, lens, perm, q, qd, 0, 0), o,
                               rtol=1e-6, atol=1e-7)


def test_attention_each_draft_reads_the_one_resident_set():
    # D drafts: row 0 is the normal query's output, row 1 + e equals the
    # one-draft output for draft e (pinned above against dense softmax),
    # on a multi-request layer so a wrong draft or request stride shows.
    rng = np.random.default_rng(14)
    R, Hkv, G, NB, B, d, D = 3, 2, 4, 6, 16, 128, 3
    kv, q, _ = rand_layer(rng, R, Hkv, G, NB)
    qd = to_bits(rng.standard_normal((D, R, Hkv * G, d)))
    lens = np.array([NB * B, 3 * B + 2, NB * B - 1], dtype=np.int32)
    res = np.stack([np.stack([rng.permutation(NB)[:4] for _ in range(Hkv)])
                    for _ in range(R)]).astype(np.int32)
    res[1, 1, 2] = -1
    for r in range(R):
        for h in range(Hkv):
            o = oracle.attention_rh(kv, lens, res, q, qd, r, h)
            assert o.shape == (1 + D, G, d)
            for e in range(D):
                one = oracle.attention_rh(kv, lens, res, q, np.ascontiguousarray(qd[e]), r, h)
                np.testing.assert_array_equal(o[0], one[0])
                np.testing.assert_array_equal(o[1 + e], one[1])


def test_step_with_two_identical_drafts_ranks_as_one():
    # Doubling every score (exact in binary floating point) changes no rank:
    # two copies of one draft give the one-draft top-K and eviction.
    from sparse_kv_block_gb300 import workload
    shape = workload.SHAPES["tiny"]
    lens = workload.ctx_lens(shape)
    kv = workload.bf16_bits(workload.host_kv(shape, 0, 0, lens, device="cpu"))
    summ = oracle.summary_build(kv, lens)
    res0 = workload.initial_resident(shape, 0, 0, lens)
    pairs = [(r, h) for r in range(shape.R) for h in range(shape.Hkv)]
    one = oracle.LayerOracle(kv, summ, lens, res0, shape.K, shape.C, pairs)
    two = oracle.LayerOracle(kv, summ, lens, res0, shape.K, shape.C, pairs)
    q, qd = workload.queries(shape, 0, 0, 3, device="cpu")
    for t in range(3):
        qb, qdb = workload.bf16_bits(q[t]), workload.bf16_bits(qd[t])
        a = one.step(qb, qdb, t)
        b = two.step(qb, np.stack([qdb, qdb]), t)
        for p in pairs:
            np.testing.assert_array_equal(b[p]["scores"], 2 * a[p]["scores"])
            np.testing.assert_array_equal(b[p]["topk"], a[p]["topk"])
            np.testing.assert_array_equal(b[p]["admit_ids"], a[p]["admit_ids"])
            np.testing.assert_array_equal(b[p]["attn"][:2], a[p]["attn"])
            np.testing.assert_array_equal(b[p]["attn"][2], a[p]["attn"][1])
    np.testing.assert_array_equal(one.res, two.res)
    np.testing.assert_array_equal(one.stamp, two.stamp)


# ----------------------------------------------------------------- eviction
def test_eviction_hand_worked():
    cases = json.load(open(os.path.join(GOLD, "lrs_eviction_hand.json")))["cases"]
    for c in cases:
        res = np.array(c["res0"], dtype=np.int32)
        stamp = np.array(c["stamp0"], dtype=np.int32)
        for st in c["steps"]:
            a, s, e, n = oracle.admit_evict_rh(res, stamp, np.array(st["topk"], np.int32),
                                               c["C"], st["t"])
            assert n == st["n"], (c["name"], st["t"])
            assert list(a[:n]) == st["admit_ids"] and list(s[:n]) == st["admit_slots"]
            assert list(e[:n]) == st["evict_ids"]
            assert list(res) == st["res"] and list(stamp) == st["stamp"], (c["name"], st["t"])


@pytest.mark.parametrize("seed", range(4))
def test_eviction_invariants_random_walk(seed):
    rng = np.random.default_rng(100 + seed)
    NB, K = 40, 12
    for C in (0, 1, 3, K):
        res = rng.permutation(NB)[:K].astype(np.int32)
        stamp = np.full(K, -1, dtype=np.int32)
        for t in range(30):
            topk = rng.permutation(NB)[:K].astype(np.int32)
            before_res, before_stamp = res.copy(), stamp.copy()
            a, s, e, n = oracle.admit_evict_rh(res, stamp, topk, C, t)
            T = set(topk.tolist())
            missing = [b for b in topk if b not in set(before_res.tolist())]
            assert n == min(len(missing), C)
            assert len(set(res.tolist())) == K                      # distinct, count fixed
            assert list(a[:n]) == missing[:n]                       # best-ranked first
            assert all(x not in T for x in e[:n])                   # never evict a selected block
            kept = [i for i in range(K) if i not in set(s[:n].tolist())]
            for i in kept:                                          # untouched slots keep ids
                assert res[i] == before_res[i]
                assert stamp[i] == (t if before_res[i] in T else before_stamp[i])
            # every evictee was no more recently selected than any unselected survivor
            surv = [before_stamp[i] for i in kept if before_res[i] not in T]
            for slot in s[:n]:
                assert all(before_stamp[slot] <= x for x in surv)
            if C == K:
                assert set(res.tolist()) == T                       # fetch-all: resident = top-K


def test_eviction_cap_zero_only_restamps():
    res = np.array([3, 1, 2], dtype=np.int32)
    stamp = np.array([-1, -1, -1], dtype=np.int32)
    a, s, e, n = oracle.admit_evict_rh(res, stamp, np.array([1, 9, 8], np.int32), 0, 5)
    assert n == 0 and list(res) == [3, 1, 2] and list(stamp) == [-1, 5, -1]


# ------------------------------------------------------------------- append
def test_append_token_matches_numpy_minmax():
    rng = np.random.default_rng(20)
    R, H, NB, B, d = 2, 2, 3, 16, 128
    kv = to_bits(np.zeros((R, H, NB, 2, B, d)))
    summ = np.zeros((R, H, NB, 2, d), dtype=np.uint16)
    lens = np.array([0, 0], dtype=np.int32)
    for step in range(2 * B + 3):
        k = to_bits(rng.standard_normal((H, d)))
        v = to_bits(rng.standard_normal((H, d)))
        for r in range(R):
            oracle.append_token(kv, summ, lens, k, v, r)
        lens += 1
    kf = to_float(kv)
    for b in range(3):
        valid = min(B, lens[0] - b * B)
        np.testing.assert_array_equal(to_float(summ[:, :, b, 0]), kf[:, :, b, 0, :valid].min(axis=2))
        np.testing.assert_array_equal(to_float(summ[:, :, b, 1]), kf[:, :, b, 0, :valid].max(axis=2))


# ------------------------------------------------------------ remote tier
def test_remote_fetch_hand_worked():
    g = json.load(open(os.path.join(GOLD, "remote_fetch_hand.json")))
    local_map = np.full(g["NBmax"], -1, dtype=np.int32)
    count = np.zeros(1, dtype=np.int32)
    for c in g["calls"]:
        mi, ms, full = oracle.remote_fetch_rh(c["ids"], local_map, count, g["capacity"])
        assert mi.tolist() == c["miss_ids"], c["why"]
        assert ms.tolist() == c["miss_slots"], c["why"]
        assert int(count[0]) == c["count"] and full == c["full"], c["why"]
    want = np.full(g["NBmax"], -1, dtype=np.int32)
    for k, v in g["final_map"].items():
        want[int(k)] = v
    np.testing.assert_array_equal(local_map, want)


@pytest.mark.parametrize("seed,capacity", [(0, 64), (1, 12), (2, 3)])
def test_remote_fetch_matches_set_model(seed, capacity):
    """Brute-force model with Python sets and a list of first appearances:
    the held set is the first `capacity` distinct ids ever listed, slot =
    position in that order, and each call fetches exactly the newly held
    ids in list order."""
    rng = np.random.default_rng(seed)
    NB = 64
    local_map = np.full(NB, -1, dtype=np.int32)
    count = np.zeros(1, dtype=np.int32)
    order = []
    for _ in range(40):
        n = int(rng.integers(0, 9))
        ids = rng.choice(NB, size=n, replace=False).astype(np.int32)
        ids[rng.random(n) < 0.15] = -1
        before = list(order)
        new = []
        overflow = False
        for x in ids.tolist():
            if x < 0 or x in order:
                continue
            if len(order) < capacity:
                order.append(x)
                new.append(x)
            else:
                overflow = True
        mi, ms, full = oracle.remote_fetch_rh(ids, local_map, count, capacity)
        assert mi.tolist() == new
        assert ms.tolist() == list(range(len(before), len(order)))
        assert full == overflow
        assert int(count[0]) == len(order)
        held = {int(b) for b in np.nonzero(local_map >= 0)[0]}
        assert held == set(order)
        assert sorted(local_map[local_map >= 0].tolist()) == list(range(len(order)))
        for slot, b in enumerate(order):
            assert local_map[b] == slot


def test_remote_fetch_oracle_layer_tracks_admissions():
    """LayerOracle with a remote tier: the initial fetch is the resident set
    in slot order, and every later fetch is the step's admitted blocks that
    were never held before (capacity = NBmax, so nothing overflows)."""
    from sparse_kv_block_gb300 import workload
    shape = workload.SHAPES["tiny"]
    lens = workload.ctx_lens(shape)
    kv = workload.bf16_bits(workload.host_kv(shape, 0, 0, lens, device="cpu"))
    summ = oracle.summary_build(kv, lens)
    res0 = workload.initial_resident(shape, 0, 0, lens)
    pairs = [(r, h) for r in range(shape.R) for h in range(shape.Hkv)]
    orc = oracle.LayerOracle(kv, summ, lens, res0, shape.K, shape.C, pairs,
                             remote_capacity=shape.NBmax)
    seen = {p: [int(x) for x in res0[p] if x >= 0] for p in pairs}
    for p in pairs:
        assert orc.resident_misses[p]["miss_ids"].tolist() == seen[p]
        assert orc.initial_misses[p]["n_miss"] == 0          # 1024-token contexts: no tail
    q, qd = workload.queries(shape, 0, 0, 4, device="cpu")
    for t in range(4):
        out = orc.step(workload.bf16_bits(q[t]), workload.bf16_bits(qd[t]), t)
        for p in pairs:
            adm = out[p]["admit_ids"][:out[p]["n_admit"]].tolist()
            new = [x for x in adm if x not in seen[p]]
            assert out[p]["miss_ids"].tolist() == new
            assert out[p]["miss_slots"].tolist() == list(range(len(seen[p]), len(seen[p]) + len(new)))
            seen[p] += new
            assert int(orc.local_count[p]) == len(seen[p])


def test_remote_oracle_tail_fetch_and_appends():
    """Remote tier with ragged contexts: the load fetches the resident set and
    then each context's partial tail block; appends inside a held block take
    no slot, an append that opens a block takes the next one."""
    from sparse_kv_block_gb300 import workload
    shape = workload.SHAPES["tiny"]
    lens = np.array([1000, 32], dtype=np.int32)          # 1000 = 62*16 + 8; 32 = 2*16
    kv = workload.bf16_bits(workload.host_kv(shape, 0, 0, lens, device="cpu"))
    summ = oracle.summary_build(kv, lens)
    res0 = workload.initial_resident(shape, 0, 0, lens)
    pairs = [(0, 0), (1, 0)]
    orc = oracle.LayerOracle(kv, summ, lens.copy(), res0, shape.K, shape.C, pairs,
                             remote_capacity=shape.NBmax)
    # request 0: tail block 62 fetched unless resident already
    tail0 = orc.initial_misses[(0, 0)]
    assert tail0["miss_ids"].tolist() == ([] if 62 in res0[0, 0] else [62])
    assert orc.local_map[0, 0, 62] >= 0
    # request 1: context ends on a block boundary, nothing extra
    assert orc.initial_misses[(1, 0)]["n_miss"] == 0
    c0 = orc.local_count.copy()
    assert orc.append_local(0) is False                  # position 1000: inside block 62
    assert (orc.local_count == c0).all()
    assert orc.append_local(1) is False                  # position 32: opens block 2
    assert orc.local_count[1, 0] == c0[1, 0] + (0 if 2 in res0[1, 0] else 1)
    assert orc.local_map[1, 0, 2] >= 0
