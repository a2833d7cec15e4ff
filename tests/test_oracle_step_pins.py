"""Pins of the oracle's step compositions: the look-ahead step (orc_step_rh,
behind LayerOracle.step) and the miss-stall step (orc_demand_rh +
orc_stall_step_rh, behind LayerOracle.stall_step).

Sources: "Pith review of OasisKV" (pith.science), the abstract (prefetched
blocks are placed in HBM one decode step before they are used, so a step's
attention reads the resident set as it stands when the step starts) and the
section "What would settle it" (a block the look-ahead missed is either
dropped from attention or fetched on demand, which stalls the step).

The hand-worked layer below is built so that every attention output has a
closed form: all tokens of a block share one key and one value, so the
summary min = max = key, every score is an exact dot product and the softmax
weights are equal within a block.  Computing the attention after the step's
admission, or ranking the demand fetch with the draft instead of the normal
query, changes the outputs there.
"""
import math

import numpy as np
import pytest

import oracle
from tests._bf16 import to_bits, to_float

B, D_HEAD = 16, 128
SCALE = 1.0 / math.sqrt(D_HEAD)


def hand_layer():
    """One request, one query head on one KV head, 4 full blocks.
    Block b: key = c_b * e0 + f_b * e1 with c = [0, 1, 3, 2], f = [0, 0, 0, 2];
    value = b in every dim.  q = e1 (normal query), qd = e0 (draft)."""
    c = [0.0, 1.0, 3.0, 2.0]
    f = [0.0, 0.0, 0.0, 2.0]
    kv = np.zeros((1, 1, 4, 2, B, D_HEAD), dtype=np.float32)
    for b in range(4):
        kv[0, 0, b, 0, :, 0] = c[b]
        kv[0, 0, b, 0, :, 1] = f[b]
        kv[0, 0, b, 1] = float(b)
    q = np.zeros((1, 1, D_HEAD), dtype=np.float32)
    q[0, 0, 1] = 1.0
    qd = np.zeros((1, 1, D_HEAD), dtype=np.float32)
    qd[0, 0, 0] = 1.0
    kvb = to_bits(kv)
    lens = np.array([4 * B], dtype=np.int32)
    return kvb, oracle.summary_build(kvb, lens), lens, to_bits(q), to_bits(qd)


def two_block_softmax(v_a, v_b, logit_a, logit_b):
    """softmax over two blocks of B tokens each with constant logits/values."""
    wa, wb = math.exp(logit_a), math.exp(logit_b)
    return (v_a * wa + v_b * wb) / (wa + wb)


def test_step_attends_before_its_admission_hand_worked():
    kv, summ, lens, q, qd = hand_layer()
    res0 = np.array([[[0, 1]]], dtype=np.int32)
    orc = oracle.LayerOracle(kv, summ, lens, res0, K=2, C=1, pairs=[(0, 0)])
    # step 0: resident {0, 1}.  q . k = 0 on both blocks -> uniform -> 0.5.
    # qd . k0 = 0, qd . k1 = 1 -> weights 1 : e^s.
    v = orc.step(q, qd, 0)[(0, 0)]
    np.testing.assert_allclose(v["attn"][0, 0], 0.5, rtol=1e-7)
    np.testing.assert_allclose(v["attn"][1, 0], two_block_softmax(0, 1, 0, SCALE), rtol=1e-6)
    # scores of qd = c = [0, 1, 3, 2] -> top-2 = [2, 3]; neither is resident,
    # C = 1: block 2 (best-ranked) replaces the LRS slot 0 (both stamps -1,
    # lower id first) and block 0 is evicted.
    np.testing.assert_array_equal(v["scores"][:4], [0, 1, 3, 2])
    assert list(v["topk"]) == [2, 3]
    assert (v["n_admit"], list(v["admit_ids"]), list(v["admit_slots"]),
            list(v["evict_ids"])) == (1, [2], [0], [0])
    assert orc.res[0, 0].tolist() == [2, 1] and orc.stamp[0, 0].tolist() == [0, -1]
    # Had the step attended after admitting, q would see {2, 1}: 1.5, not 0.5.
    # step 1: resident {2, 1}: q uniform -> 1.5; qd logits 3s (block 2), s (block 1).
    v = orc.step(q, qd, 1)[(0, 0)]
    np.testing.assert_allclose(v["attn"][0, 0], 1.5, rtol=1e-7)
    np.testing.assert_allclose(v["attn"][1, 0], two_block_softmax(2, 1, 3 * SCALE, SCALE),
                               rtol=1e-6)
    # block 2 re-selected (stamp 1), block 3 replaces slot 1 (block 1 evicted)
    assert (v["n_admit"], list(v["admit_ids"]), list(v["admit_slots"]),
            list(v["evict_ids"])) == (1, [3], [1], [1])
    assert orc.res[0, 0].tolist() == [2, 3] and orc.stamp[0, 0].tolist() == [1, 1]


def test_stall_step_fetches_the_query_topk_before_attending_hand_worked():
    kv, summ, lens, q, qd = hand_layer()
    res0 = np.array([[[0, 1]]], dtype=np.int32)
    orc = oracle.LayerOracle(kv, summ, lens, res0, K=2, C=1, pairs=[(0, 0)])
    v = orc.stall_step(q, qd, 0)[(0, 0)]
    # Demand: scores of q = f = [0, 0, 0, 2] -> top-2 = [3, 0] (ties by id).
    # Block 0 is resident (stamped 0); block 3 replaces slot 1 (block 1),
    # uncapped (K = 2 would allow both).
    np.testing.assert_array_equal(v["dm_scores"][:4], [0, 0, 0, 2])
    assert list(v["dm_topk"]) == [3, 0]
    assert v["dm_n_admit"] == 1
    assert list(v["dm_admit_ids"]) == [3, -1] and list(v["dm_admit_slots"]) == [1, -1]
    assert list(v["dm_evict_ids"]) == [1, -1]
    # Attention over {0, 3}: q . k3 = 2, qd . k3 = 2, both 0 on block 0.
    want = two_block_softmax(0, 3, 0, 2 * SCALE)
    np.testing.assert_allclose(v["attn"][0, 0], want, rtol=1e-6)
    np.testing.assert_allclose(v["attn"][1, 0], want, rtol=1e-6)
    # Look-ahead on the post-demand table: top-2 of qd = [2, 3]; block 3 is
    # resident (stamp 0), block 2 replaces slot 0 (block 0, stamp 0).
    assert list(v["topk"]) == [2, 3]
    assert (v["n_admit"], list(v["admit_ids"]), list(v["admit_slots"]),
            list(v["evict_ids"])) == (1, [2], [0], [0])
    assert orc.res[0, 0].tolist() == [2, 3] and orc.stamp[0, 0].tolist() == [0, 0]


def test_demand_fetch_is_not_capped_hand_worked():
    # Nothing of the query's top-K is resident: every block is fetched at
    # once although the look-ahead cap is 1.
    kv, summ, lens, q, qd = hand_layer()
    res = np.array([[[1, 2]]], dtype=np.int32)
    stamp = np.array([[[4, 3]]], dtype=np.int32)
    d = oracle.demand_rh(summ, lens, res, stamp, q, 0, 0, K=2, step=5, B=B)
    assert list(d["topk"]) == [3, 0] and d["n_admit"] == 2
    # LRS order: slot 1 (stamp 3) before slot 0 (stamp 4).
    assert list(d["admit_ids"]) == [3, 0] and list(d["admit_slots"]) == [1, 0]
    assert list(d["evict_ids"]) == [2, 1]
    assert res[0, 0].tolist() == [0, 3] and stamp[0, 0].tolist() == [5, 5]


def rand_layer(rng, R, Hkv, G, NB, lens):
    kv = to_bits(rng.standard_normal((R, Hkv, NB, 2, B, D_HEAD)))
    q = to_bits(rng.standard_normal((R, Hkv * G, D_HEAD)))
    qd = to_bits(rng.standard_normal((R, Hkv * G, D_HEAD)))
    return kv, oracle.summary_build(kv, lens), q, qd


@pytest.mark.parametrize("seed", range(3))
def test_step_is_attention_then_score_topk_then_admission(seed):
    # LayerOracle.step against the stage functions run by hand in the
    # reading's order: (a) attention on the table before the admission,
    # (b) top-K of the summary scores, (c) capped eviction fed that list.
    rng = np.random.default_rng(200 + seed)
    R, Hkv, G, NB, K, C = 2, 2, 4, 12, 5, 2
    lens = np.array([NB * B, NB * B - 21], dtype=np.int32)
    kv, summ, _, _ = rand_layer(rng, R, Hkv, G, NB, lens)
    res0 = np.stack([np.stack([rng.permutation(NB)[:K] for _ in range(Hkv)])
                     for _ in range(R)]).astype(np.int32)
    pairs = [(r, h) for r in range(R) for h in range(Hkv)]
    orc = oracle.LayerOracle(kv, summ, lens, res0, K, C, pairs)
    res, stamp = res0.copy(), np.full_like(res0, -1)
    for t in range(4):
        q = to_bits(rng.standard_normal((R, Hkv * G, D_HEAD)))
        qd = to_bits(rng.standard_normal((R, Hkv * G, D_HEAD)))
        got = orc.step(q, qd, t)
        for (r, h) in pairs:
            v = got[(r, h)]
            np.testing.assert_array_equal(v["attn"], oracle.attention_rh(kv, lens, res, q, qd, r, h))
            s = oracle.score_rh(summ, lens, qd, r, h, B)
            np.testing.assert_array_equal(v["scores"], s)
            tk = oracle.topk_rh(s, -(-int(lens[r]) // B), K)
            np.testing.assert_array_equal(v["topk"], tk)
            a, sl, e, n = oracle.admit_evict_rh(res[r, h], stamp[r, h], tk, C, t)
            assert v["n_admit"] == n
            np.testing.assert_array_equal(v["admit_ids"], a)
            np.testing.assert_array_equal(v["admit_slots"], sl)
            np.testing.assert_array_equal(v["evict_ids"], e)
        np.testing.assert_array_equal(orc.res, res)
        np.testing.assert_array_equal(orc.stamp, stamp)


def dense_softmax(keys, vals, x, scale):
    logits = keys @ x * scale
    w = np.exp(logits - logits.max())
    return (w[:, None] * vals).sum(axis=0) / w.sum()


@pytest.mark.parametrize("seed", range(3))
def test_stall_step_attends_over_exactly_the_query_topk(seed):
    # With at least K blocks in the context the demand fetch leaves exactly
    # the normal query's top-K resident, whatever was resident before, so
    # the stall step's attention is dense softmax attention over the tokens
    # of those K blocks (textbook numpy over the blocks ranked here by brute
    # force on the summaries).
    rng = np.random.default_rng(300 + seed)
    R, Hkv, G, NB, K, C = 2, 2, 4, 10, 4, 1
    lens = np.array([NB * B, NB * B - 5], dtype=np.int32)
    kv, summ, _, _ = rand_layer(rng, R, Hkv, G, NB, lens)
    res0 = np.stack([np.stack([rng.permutation(NB)[:K] for _ in range(Hkv)])
                     for _ in range(R)]).astype(np.int32)
    pairs = [(r, h) for r in range(R) for h in range(Hkv)]
    orc = oracle.LayerOracle(kv, summ, lens, res0, K, C, pairs)
    kf, sf = to_float(kv).astype(np.float64), to_float(summ).astype(np.float64)
    for t in range(3):
        q = to_bits(rng.standard_normal((R, Hkv * G, D_HEAD)))
        qd = to_bits(rng.standard_normal((R, Hkv * G, D_HEAD)))
        qf, qdf = to_float(q).astype(np.float64), to_float(qd).astype(np.float64)
        before = orc.res.copy()
        got = orc.stall_step(q, qd, t)
        for (r, h) in pairs:
            v = got[(r, h)]
            nb = -(-int(lens[r]) // B)
            x = qf[r, h * G:(h + 1) * G]                              # [G][d]
            bound = np.maximum(x[:, None, :] * sf[r, h, :nb, 0][None],
                               x[:, None, :] * sf[r, h, :nb, 1][None]).sum(axis=(0, 2))
            order = sorted(range(nb), key=lambda b: (-np.float32(bound[b]), b))
            assert list(v["dm_topk"]) == order[:K]
            T = set(order[:K])
            missing = [b for b in order[:K] if b not in set(before[r, h].tolist())]
            assert v["dm_n_admit"] == len(missing)
            assert list(v["dm_admit_ids"][:len(missing)]) == missing
            assert all(e not in T for e in v["dm_evict_ids"][:len(missing)])
            blocks = sorted(T)
            keys = np.concatenate([kf[r, h, b, 0, :min(B, lens[r] - b * B)] for b in blocks])
            vals = np.concatenate([kf[r, h, b, 1, :min(B, lens[r] - b * B)] for b in blocks])
            for g in range(G):
                np.testing.assert_allclose(v["attn"][0, g], dense_softmax(keys, vals, x[g], SCALE),
                                           rtol=1e-5, atol=1e-6)
                np.testing.assert_allclose(v["attn"][1, g],
                                           dense_softmax(keys, vals, qdf[r, h * G + g], SCALE),
                                           rtol=1e-5, atol=1e-6)
            # the look-ahead admission that follows keeps the count and ids distinct
            assert len(set(orc.res[r, h].tolist())) == K


def test_stall_step_with_the_draft_equal_to_the_query_admits_nothing_ahead():
    # The look-ahead top-K equals the demand top-K, which is resident by then.
    rng = np.random.default_rng(400)
    R, Hkv, G, NB, K, C = 1, 2, 2, 9, 4, 2
    lens = np.array([NB * B - 3], dtype=np.int32)
    kv, summ, q, _ = rand_layer(rng, R, Hkv, G, NB, lens)
    res0 = np.array([[[0, 1, 2, 3], [4, 5, 6, 7]]], dtype=np.int32)
    orc = oracle.LayerOracle(kv, summ, lens, res0, K, C, [(0, 0), (0, 1)])
    for t in range(3):
        got = orc.stall_step(q, q, t)
        for v in got.values():
            assert v["n_admit"] == 0
            np.testing.assert_array_equal(v["topk"], v["dm_topk"])
            np.testing.assert_array_equal(v["attn"][0], v["attn"][1])


def test_stall_step_equals_demand_then_step():
    # The stall step is exactly the demand fetch followed by the pinned
    # look-ahead step on the updated table.
    rng = np.random.default_rng(500)
    R, Hkv, G, NB, K, C = 2, 1, 4, 11, 4, 1
    lens = np.array([NB * B, 6 * B + 1], dtype=np.int32)
    kv, summ, q, qd = rand_layer(rng, R, Hkv, G, NB, lens)
    res0 = np.array([[[0, 1, 2, 3]], [[3, 2, 1, 0]]], dtype=np.int32)
    pairs = [(0, 0), (1, 0)]
    a = oracle.LayerOracle(kv, summ, lens, res0, K, C, pairs)
    b = oracle.LayerOracle(kv, summ, lens, res0, K, C, pairs)
    for t in range(3):
        got = a.stall_step(q, qd, t)
        dm = {p: oracle.demand_rh(summ, lens, b.res, b.stamp, q, p[0], p[1], K, t, B)
              for p in pairs}
        ref = b.step(q, qd, t)
        for p in pairs:
            for k in ("scores", "topk", "admit_ids", "admit_slots", "evict_ids", "n_admit"):
                np.testing.assert_array_equal(got[p]["dm_" + k], dm[p][k])
                np.testing.assert_array_equal(got[p][k], ref[p][k])
            np.testing.assert_array_equal(got[p]["attn"], ref[p]["attn"])
    np.testing.assert_array_equal(a.res, b.res)
    np.testing.assert_array_equal(a.stamp, b.stamp)
