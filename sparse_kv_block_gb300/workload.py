"""Seeded synthetic workloads for the look-ahead sparse decode step.

This module draws random inputs only: it holds none of the method's
arithmetic (no summaries, scores, top-K, eviction or attention).  Both the
CUDA path and the CPU oracle consume the very bytes it produces.

Values are drawn in fp32 with torch's Philox/MT generators seeded per tensor
and rounded to bf16 (round to nearest even).  Draws on a CUDA device and on
the CPU give different (equally valid) streams; a test or benchmark draws once
and hands the same buffers to both sides.

Workloads (shapes follow the pages' Qwen3-8B / Llama-3.1-8B setting: B = 16,
K = 128 blocks = a 2,048-token budget, fetch cap 0.05; the pages' datasets
and model weights are not available, so these draws stand in for them):

* ``tiny``            2 requests x 1024 tokens, 8 q / 2 KV heads, d = 128,
                      K = 16, cap 0.25; K/V/q ~ N(0,1), qd = q + N(0, 0.1^2).
* ``qwen3_8b_16k``    128 requests x 16384 tokens (1024 blocks), 32 q / 8 KV
                      heads, K = 128, cap 0.05.  Per KV head a unit direction
                      u_h; 5 % of the blocks of every (request, KV head) are
                      "hot": their keys are N(0,1) + 3 u_h.  Queries
                      q_t = 8 u_h + z_t, z_t ~ N(0, I); the draft query
                      qd_t = 8 u_h + 0.95 z_{t+1} + sqrt(1 - 0.95^2) e_t, so
                      its noise is 0.95-correlated with the next step's query.
* ``qwen3_8b_36l``    the same per-layer shapes at 90 requests, 36 layers;
                      every step each hot block moves to a random block with
                      probability 0.02.
* ``llama31_8b_32k``  32 layers, 64 requests from 32768 tokens (2048 blocks)
                      growing by one token per step.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    R: int
    Hq: int
    Hkv: int
    d: int
    B: int
    ctx: int                 # initial tokens per request
    K: int
    fetch_ratio: float
    layers: int = 1
    grow_steps: int = 0      # tokens appended per request over the run
    hot_frac: float = 0.0    # share of hot blocks per (request, KV head)
    hot_shift: float = 0.0   # hot keys get + hot_shift * u_h
    q_mean: float = 0.0      # queries get + q_mean * u_h
    draft_corr: Optional[float] = None  # None: qd = q + N(0, draft_sigma^2)
    draft_sigma: float = 0.1
    hot_move_prob: float = 0.0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def NBmax(self) -> int:
        return -(-(self.ctx + self.grow_steps) // self.B)

    @property
    def C(self) -> int:
        return int(math.floor(self.fetch_ratio * self.K + 1e-9))


SHAPES = {
    "tiny": Shape("tiny", R=2, Hq=8, Hkv=2, d=128, B=16, ctx=1024, K=16,
                  fetch_ratio=0.25),
    "qwen3_8b_16k": Shape("qwen3_8b_16k", R=128, Hq=32, Hkv=8, d=128, B=16,
                          ctx=16384, K=128, fetch_ratio=0.05, hot_frac=0.05,
                          hot_shift=3.0, q_mean=8.0, draft_corr=0.95),
    "qwen3_8b_36l": Shape("qwen3_8b_36l", R=90, Hq=32, Hkv=8, d=128, B=16,
                          ctx=16384, K=128, fetch_ratio=0.05, layers=36,
                          hot_frac=0.05, hot_shift=3.0, q_mean=8.0,
                          draft_corr=0.95, hot_move_prob=0.02),
    "llama31_8b_32k": Shape("llama31_8b_32k", R=64, Hq=32, Hkv=8, d=128, B=16,
                            ctx=32768, K=128, fetch_ratio=0.05, layers=32,
                            grow_steps=256, hot_frac=0.05, hot_shift=3.0,
                            q_mean=8.0, draft_corr=0.95),
}


def _gen(device, *key: int) -> torch.Generator:
    """A generator on `device` seeded from an integer key tuple."""
    seed = 0x9E3779B97F4A7C15
    for k in key:
        seed = (seed * 6364136223846793005 + (int(k) & 0xFFFFFFFF) + 1442695040888963407) % (1 << 63)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def ctx_lens(shape: Shape, ragged: Optional[list] = None) -> np.ndarray:
    """Per-request context lengths: the shape's context, or an explicit list."""
    if ragged is not None:
        return np.asarray(ragged, dtype=np.int32)
    return np.full(shape.R, shape.ctx, dtype=np.int32)


def head_directions(shape: Shape, seed: int, layer: int) -> torch.Tensor:
    """Unit vectors u_h, [Hkv][d] fp32 (CPU)."""
    u = torch.randn(shape.Hkv, shape.d, generator=_gen("cpu", seed, layer, 1))
    return u / u.norm(dim=1, keepdim=True)


def hot_blocks(shape: Shape, seed: int, layer: int, lens: np.ndarray) -> list:
    """Per (r, h): the sorted ids of the hot blocks (hot_frac of its blocks)."""
    rng = np.random.default_rng([seed, layer, 2])
    out = []
    for r in range(shape.R):
        nb = -(-int(lens[r]) // shape.B) if lens[r] > 0 else 0
        nh = int(round(shape.hot_frac * nb))
        row = []
        for _ in range(shape.Hkv):
            row.append(np.sort(rng.permutation(nb)[:nh]).astype(np.int64))
        out.append(row)
    return out


def host_kv(shape: Shape, seed: int, layer: int, lens: np.ndarray,
            device="cpu", out: Optional[torch.Tensor] = None,
            hot: Optional[list] = None) -> torch.Tensor:
    """The full KV store [R][Hkv][NBmax][2][B][d] bf16.

    Keys and values ~ N(0,1); hot blocks' keys + hot_shift * u_h; tokens at or
    past a request's context are zero.  Drawn request by request on `device`
    and written into `out` (e.g. a pinned host tensor) when given.
    """
    R, H, NB, B, d = shape.R, shape.Hkv, shape.NBmax, shape.B, shape.d
    if out is None:
        out = torch.empty((R, H, NB, 2, B, d), dtype=torch.bfloat16,
                          pin_memory=False)
    assert tuple(out.shape) == (R, H, NB, 2, B, d) and out.dtype == torch.bfloat16
    g = _gen(device, seed, layer, 3)
    u = head_directions(shape, seed, layer).to(device)
    if shape.hot_frac > 0 and hot is None:
        hot = hot_blocks(shape, seed, layer, lens)
    tok = torch.arange(NB * B, device=device).view(NB, B)
    for r in range(R):
        x = torch.randn((H, NB, 2, B, d), generator=g, device=device)
        if hot is not None:
            for h in range(H):
                ids = torch.as_tensor(hot[r][h], device=device)
                if ids.numel():
                    x[h, ids, 0] += shape.hot_shift * u[h]
        dead = (tok >= int(lens[r])).view(1, NB, 1, B, 1)
        x.masked_fill_(dead, 0.0)
        out[r].copy_(x.to(torch.bfloat16), non_blocking=False)
    return out


def queries(shape: Shape, seed: int, layer: int, steps: int,
            device="cpu", direction_layer: Optional[int] = None) -> tuple:
    """(q, qd) for `steps` consecutive steps: [steps][R][Hq][d] bf16 each.
    The query mean points along the head directions of `direction_layer`
    (default `layer`): the layer whose host store the queries read."""
    q, qd = draft_queries(shape, seed, layer, steps, 1, device, direction_layer)
    return q, qd[:, 0]


def draft_queries(shape: Shape, seed: int, layer: int, steps: int, num_drafts: int,
                  device="cpu", direction_layer: Optional[int] = None) -> tuple:
    """(q, qd) with D = num_drafts draft queries per step: q [steps][R][Hq][d],
    qd [steps][D][R][Hq][d] bf16.  Draft 0 is the draft of `queries` (the same
    draws).  Draft e > 0 looks e steps further: in the correlated recipe it
    follows the query noise of step t + 1 + e; in the plain recipe it is the
    step's query plus fresh noise."""
    R, Hq, d, G = shape.R, shape.Hq, shape.d, shape.G
    D = int(num_drafts)
    if D < 1:
        raise ValueError("num_drafts must be >= 1")
    g = _gen(device, seed, layer, 4)
    z = torch.randn((steps + 1, R, Hq, d), generator=g, device=device)
    e = torch.randn((steps, R, Hq, d), generator=g, device=device)
    if D > 1:  # drawn after the one-draft stream, which stays unchanged
        z = torch.cat([z, torch.randn((D - 1, R, Hq, d), generator=g, device=device)])
        e_more = torch.randn((D - 1, steps, R, Hq, d), generator=g, device=device)
        e = torch.stack([e] + list(e_more))
    else:
        e = e.unsqueeze(0)
    if shape.draft_corr is None:
        q = z[:steps]
        qd = torch.stack([q + shape.draft_sigma * e[k] for k in range(D)], dim=1)
    else:
        u = head_directions(shape, seed, layer if direction_layer is None
                            else direction_layer).to(device)
        mean = (shape.q_mean * u).repeat_interleave(G, dim=0)  # [Hq][d]
        rho = shape.draft_corr
        q = mean + z[:steps]
        c = math.sqrt(1.0 - rho * rho)
        qd = torch.stack([mean + rho * z[1 + k:1 + k + steps] + c * e[k] for k in range(D)],
                         dim=1)
    return q.to(torch.bfloat16), qd.to(torch.bfloat16)


def move_hot_blocks(shape: Shape, seed: int, layer: int, step: int, hot: list,
                    lens: np.ndarray) -> list:
    """Drift of the planted structure between two steps: every hot block of
    every (r, h) moves, with probability hot_move_prob, to a block drawn
    uniformly from the request's blocks that are not hot.  Updates `hot` in
    place and returns the moves as (r, h, old, new) tuples."""
    rng = np.random.default_rng([seed, layer, 7, step])
    moves = []
    for r in range(shape.R):
        nb = -(-int(lens[r]) // shape.B) if lens[r] > 0 else 0
        for h in range(shape.Hkv):
            ids = hot[r][h]
            if len(ids) == 0 or len(ids) >= nb:
                continue
            go = np.nonzero(rng.random(len(ids)) < shape.hot_move_prob)[0]
            for k in go:
                taken = set(int(x) for x in ids)
                new = int(rng.integers(0, nb))
                while new in taken:
                    new = int(rng.integers(0, nb))
                moves.append((r, h, int(ids[k]), new))
                ids[k] = new
    return moves


def apply_hot_moves(shape: Shape, seed: int, layer: int, store: torch.Tensor,
                    moves: list, lens: np.ndarray) -> None:
    """Rewrite the keys of moved hot blocks in a host store: the old block
    loses the hot_shift * u_h offset, the new block gains it (valid tokens
    only; tokens past the context stay zero).  `store` may be a CPU tensor or
    a CUDA view of a pinned store (the rewrite then runs on the GPU)."""
    if not moves:
        return
    dev = store.device
    u = head_directions(shape, seed, layer).to(dev)
    m = torch.as_tensor(moves, dtype=torch.int64, device=dev)
    r, h, old, new = m[:, 0], m[:, 1], m[:, 2], m[:, 3]
    tok = torch.arange(shape.B, device=dev)
    L = torch.as_tensor(lens, dtype=torch.int64, device=dev)
    for blk, sign in ((old, -1.0), (new, 1.0)):
        valid = (blk[:, None] * shape.B + tok[None, :]) < L[r][:, None]      # [n][B]
        x = store[r, h, blk, 0].float()                                       # [n][B][d]
        x += sign * shape.hot_shift * u[h][:, None, :] * valid[:, :, None]
        store[r, h, blk, 0] = x.to(torch.bfloat16)


def initial_resident(shape: Shape, seed: int, layer: int,
                     lens: np.ndarray) -> np.ndarray:
    """A random resident set per (r, h): [R][Hkv][K] int32, distinct ids in a
    random slot order, -1 for the slots a short context cannot fill."""
    rng = np.random.default_rng([seed, layer, 5])
    res = np.full((shape.R, shape.Hkv, shape.K), -1, dtype=np.int32)
    for r in range(shape.R):
        nb = -(-int(lens[r]) // shape.B) if lens[r] > 0 else 0
        for h in range(shape.Hkv):
            ids = rng.permutation(nb)[:shape.K]
            res[r, h, :len(ids)] = ids
            res[r, h] = res[r, h, rng.permutation(shape.K)]
    return res


def new_tokens(shape: Shape, seed: int, layer: int, step: int,
               device="cpu") -> tuple:
    """Keys and values of one appended token per request: [R][Hkv][d] bf16."""
    g = _gen(device, seed, layer, 6, step)
    kv = torch.randn((2, shape.R, shape.Hkv, shape.d), generator=g, device=device)
    kv = kv.to(torch.bfloat16)
    return kv[0].contiguous(), kv[1].contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A CPU bf16 tensor's bit patterns as a uint16 numpy view (no copy)."""
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.view(torch.int16).numpy().view(np.uint16)
