"""Host-side checks of the seeded input generators (no method arithmetic in
them): the hot-block drift keeps the number of hot blocks, moves each to a
block that was not hot, is reproducible from the seed, and rewrites keys by
exactly the planted offset; several draft queries extend the one-draft
recipe."""
import dataclasses

import numpy as np
import torch

from sparse_kv_block_gb300 import workload


def _shape():
    return dataclasses.replace(workload.SHAPES["qwen3_8b_36l"], R=3, ctx=4000)


def test_move_hot_blocks_keeps_count_and_targets_free_blocks():
    sh = _shape()
    lens = workload.ctx_lens(sh)
    hot = workload.hot_blocks(sh, 0, 0, lens)
    before = [[set(x.tolist()) for x in row] for row in hot]
    moves = []
    for step in range(50):
        mv = workload.move_hot_blocks(sh, 0, 0, step, hot, lens)
        for (r, h, old, new) in mv:
            assert old in before[r][h] and new not in before[r][h]
            before[r][h].discard(old)
            before[r][h].add(new)
        moves += mv
    nb = -(-4000 // 16)
    for r in range(sh.R):
        for h in range(sh.Hkv):
            ids = hot[r][h].tolist()
            assert len(ids) == len(set(ids)) == round(sh.hot_frac * nb)
            assert set(ids) == before[r][h]
            assert all(0 <= b < nb for b in ids)
    # with probability 0.02 per hot block and step, ~0.02 * 50 * 13 * 24 moves
    assert 200 < len(moves) < 450
    hot2 = workload.hot_blocks(sh, 0, 0, lens)
    for step in range(50):
        workload.move_hot_blocks(sh, 0, 0, step, hot2, lens)
    assert all(np.array_equal(a, b) for ra, rb in zip(hot, hot2) for a, b in zip(ra, rb))


def test_apply_hot_moves_shifts_keys_of_valid_tokens_only():
    sh = _shape()
    lens = np.array([4000, 4000, 250], dtype=np.int32)     # request 2 ends mid-block 15
    store = torch.zeros((sh.R, sh.Hkv, sh.NBmax, 2, 16, 128), dtype=torch.bfloat16)
    moves = [(0, 1, 3, 7), (2, 0, 0, 15)]
    workload.apply_hot_moves(sh, 0, 0, store, moves, lens)
    u = workload.head_directions(sh, 0, 0)
    shift = (sh.hot_shift * u).to(torch.bfloat16)
    assert torch.equal(store[0, 1, 7, 0], shift[1].expand(16, 128))
    assert torch.equal(store[0, 1, 3, 0], (-shift[1]).expand(16, 128))
    assert torch.equal(store[0, 1, 7, 1], torch.zeros(16, 128, dtype=torch.bfloat16))  # values untouched
    valid = 250 - 15 * 16                                     # 10 tokens of block 15
    assert torch.equal(store[2, 0, 15, 0, :valid], shift[0].expand(valid, 128))
    assert torch.equal(store[2, 0, 15, 0, valid:], torch.zeros(16 - valid, 128, dtype=torch.bfloat16))


def test_draft_queries_extend_the_one_draft_recipe():
    # Draft 0 is the one-draft recipe's draft (the same draws); draft e
    # follows the query noise of step t + 1 + e (correlation about 0.95 with
    # it, about 0 with the noise of other steps); the queries are unchanged.
    sh = dataclasses.replace(workload.SHAPES["qwen3_8b_16k"], R=4)
    q1, qd1 = workload.queries(sh, 7, 0, 6)
    q, qd = workload.draft_queries(sh, 7, 0, 6, 3)
    assert tuple(qd.shape) == (6, 3, sh.R, sh.Hq, sh.d)
    assert torch.equal(q, q1) and torch.equal(qd[:, 0], qd1)
    u = workload.head_directions(sh, 7, 0)
    mean = (sh.q_mean * u).repeat_interleave(sh.G, dim=0)
    zq = q.float() - mean                       # query noise of steps 0..5
    for e in range(3):
        for t in range(6 - 1 - e):
            zd = (qd[t, e].float() - mean).flatten()
            c_next = torch.corrcoef(torch.stack([zd, zq[t + 1 + e].flatten()]))[0, 1]
            c_same = torch.corrcoef(torch.stack([zd, zq[t].flatten()]))[0, 1]
            assert c_next > 0.9 and abs(c_same) < 0.1, (e, t, float(c_next), float(c_same))
    # plain recipe: every draft is the step's query plus small fresh noise
    tiny = workload.SHAPES["tiny"]
    qt, qdt = workload.draft_queries(tiny, 3, 0, 2, 2)
    for e in range(2):
        d = (qdt[:, e].float() - qt.float())
        assert 0.05 < float(d.std()) < 0.2
    assert not torch.equal(qdt[:, 0], qdt[:, 1])
