"""Seeded synthetic inputs for the QSA block scorer and top-k select.

This module only builds input arrays. It holds none of the method's arithmetic
(no dot products, no ReLU, no head sums, no ranking), so the CPU oracle and the
CUDA path can both draw their inputs from it without sharing any computation.

Shapes follow the scorer's statement of the problem (Strata PR #228, part 1,
"qsa_block_scores_wmma"): q is [nq, H, D] fp16 with D contiguous, kb is one key
vector per KV block, [nb, D] fp16, and nb = ceil(n_kv / block).

Every array is drawn in float64 from ``numpy.random.default_rng(seed)`` and
rounded once to fp16 (round to nearest even, numpy ``astype``).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, selection size and value recipe."""

    name: str
    nq: int
    H: int
    D: int
    n_kv: int
    block: int
    k: int
    dist: str  # "normal1", "normal_d", "normal_d_x8", "normal_d_onehot"
    seed: int

    @property
    def nb(self) -> int:
        return -(-self.n_kv // self.block)

    @property
    def n_full(self) -> int:
        return self.n_kv // self.block

    @property
    def has_tail(self) -> bool:
        return self.n_kv % self.block != 0


# The five workloads: a tiny CPU-checkable case, short, mid and long (128K)
# contexts at nq=256, and a large prefill batch with one-hot key rows.
WORKLOADS = [
    Workload("tiny_nq16_h4_d64_kv4000", 16, 4, 64, 4000, 64, 8, "normal1", 1001),
    Workload("short_nq256_h8_d128_kv1024", 256, 8, 128, 1024, 64, 8, "normal_d", 1002),
    Workload("mid_nq256_h8_d128_kv32805", 256, 8, 128, 32768 + 37, 64, 32, "normal_d", 1003),
    Workload("long128k_nq256_h8_d128_kv131072", 256, 8, 128, 131072, 64, 64, "normal_d_x8", 1004),
    Workload("prefill_nq4096_h16_d128_kv131073", 4096, 16, 128, 131072 + 1, 64, 64, "normal_d_onehot", 1005),
]

# Decode-shaped batches (few queries against a long context), same recipe.
DECODE_WORKLOADS = [
    Workload("decode_nq1_h8_d128_kv131072", 1, 8, 128, 131072, 64, 64, "normal_d", 1101),
    Workload("decode_nq4_h8_d128_kv131072", 4, 8, 128, 131072, 64, 64, "normal_d", 1102),
    Workload("decode_nq16_h8_d128_kv131072", 16, 8, 128, 131072, 64, 64, "normal_d", 1103),
]

BY_NAME = {w.name: w for w in WORKLOADS + DECODE_WORKLOADS}


def _f16(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float16))


def _seed(w: Workload, variant: int, salt: int = 0) -> int:
    return w.seed + salt + 104729 * variant


def make_inputs(w: Workload, variant: int = 0):
    """Return (q f16 [nq,H,D], kb f16 [nb,D]) for workload ``w``.

    ``variant`` > 0 draws another input set of the same recipe (distinct
    buffers for benchmarks that rotate through more data than L2 holds).

    normal1:          q, kb ~ N(0, 1)
    normal_d:         q, kb ~ N(0, 1/sqrt(D)) (standard deviation 1/sqrt(D))
    normal_d_x8:      as normal_d, both multiplied by 8 before rounding
    normal_d_onehot:  as normal_d; then ceil(1% of nb) kb rows are replaced by
                      one-hot rows (value 4.0 at a drawn coordinate), and the
                      second chosen row is forced onto the first one's
                      coordinate so that exact score ties exist.
    """
    rng = np.random.default_rng(_seed(w, variant))
    nb = w.nb
    if w.dist == "normal1":
        sd = 1.0
    else:
        sd = 1.0 / math.sqrt(w.D)
    q = rng.normal(0.0, sd, size=(w.nq, w.H, w.D))
    kb = rng.normal(0.0, sd, size=(nb, w.D))
    if w.dist == "normal_d_x8":
        q = q * 8.0
        kb = kb * 8.0
    if w.dist == "normal_d_onehot":
        n_hot = math.ceil(0.01 * nb)
        rows = rng.choice(nb, size=n_hot, replace=False)
        coords = rng.integers(0, w.D, size=n_hot)
        if n_hot >= 2:
            coords[1] = coords[0]
        for r, c in zip(rows, coords):
            kb[r, :] = 0.0
            kb[r, c] = 4.0
    return _f16(q), _f16(kb)


def make_f32_inputs(w: Workload, variant: int = 0):
    """Workload inputs as the f32 arrays that feed the fp32->fp16 stage.

    The f32 values are the drawn float64 values rounded to float32 (not to
    fp16), so the conversion stage has real rounding work to do.
    """
    rng = np.random.default_rng(_seed(w, variant, 7919))
    sd = 1.0 if w.dist == "normal1" else 1.0 / math.sqrt(w.D)
    scale = 8.0 if w.dist == "normal_d_x8" else 1.0
    q = rng.normal(0.0, sd, size=(w.nq, w.H, w.D)) * scale
    kb = rng.normal(0.0, sd, size=(w.nb, w.D)) * scale
    return (np.ascontiguousarray(q.astype(np.float32)),
            np.ascontiguousarray(kb.astype(np.float32)))


def random_case(nq: int, H: int, D: int, nb: int, seed: int, scale: float = 1.0):
    """Plain N(0, scale) fp16 q [nq,H,D] and kb [nb,D]."""
    rng = np.random.default_rng(seed)
    q = rng.normal(0.0, scale, size=(nq, H, D))
    kb = rng.normal(0.0, scale, size=(nb, D))
    return _f16(q), _f16(kb)


def random_case_f32(nq: int, H: int, D: int, nb: int, seed: int, scale: float = 1.0):
    """N(0, scale) q [nq,H,D] as f32 (the input of the fp32->fp16 stage) and
    kb [nb,D] as fp16."""
    rng = np.random.default_rng(seed)
    q = rng.normal(0.0, scale, size=(nq, H, D))
    kb = rng.normal(0.0, scale, size=(nb, D))
    return np.ascontiguousarray(q.astype(np.float32)), _f16(kb)


def coordinate_coded_case(nq: int, H: int, D: int, nb: int):
    """Coordinate-coded fixture: kb[b] = e_(b mod D) (one-hot, value 1) and
    q[qi,h,i] = ((7*qi + 3*h + i) mod 61) - 30, small integers exact in fp16.

    Each score then depends on one coordinate of each head only, so a
    transposed operand, a duplicated lane or a misplaced store changes the
    value; the expected result is exact at zero tolerance.
    """
    qi = np.arange(nq)[:, None, None]
    h = np.arange(H)[None, :, None]
    i = np.arange(D)[None, None, :]
    q = ((7 * qi + 3 * h + i) % 61) - 30
    kb = np.zeros((nb, D))
    kb[np.arange(nb), np.arange(nb) % D] = 1.0
    return _f16(q), _f16(kb)


def one_hot_case(nq: int, H: int, D: int, nb: int, seed: int):
    """One-hot q rows and one-hot kb rows (value 1 at a drawn coordinate)."""
    rng = np.random.default_rng(seed)
    q = np.zeros((nq, H, D))
    cq = rng.integers(0, D, size=(nq, H))
    for a in range(nq):
        for b in range(H):
            q[a, b, cq[a, b]] = 1.0
    kb = np.zeros((nb, D))
    ck = rng.integers(0, D, size=nb)
    kb[np.arange(nb), ck] = 1.0
    return _f16(q), _f16(kb)


def random_scores(nq: int, nb: int, seed: int, kind: str = "normal"):
    """f32 score matrices for the select stage on its own.

    normal:   N(0,1) f32
    ties:     small integers, so that many exact ties exist
    signed0:  a mix of +0.0, -0.0 and a few positive values
    const:    every entry equal
    """
    rng = np.random.default_rng(seed)
    if kind == "normal":
        s = rng.normal(0.0, 1.0, size=(nq, nb))
    elif kind == "ties":
        s = rng.integers(-3, 4, size=(nq, nb)).astype(np.float64)
    elif kind == "signed0":
        s = np.where(rng.random((nq, nb)) < 0.5, 0.0, -0.0)
        hot = rng.random((nq, nb)) < 0.05
        s = np.where(hot, rng.random((nq, nb)) + 0.5, s)
    elif kind == "const":
        s = np.full((nq, nb), 1.25)
    else:
        raise ValueError(kind)
    return np.ascontiguousarray(s.astype(np.float32))


# ------------------------------------------------ flash-attention split reduce
# Second workload: the reduce that closes a split (multi-block) flash-attention
# decode (1bit-MONSTER llama.cpp pull request 30, "What" and "Changes": the
# reduce_completed.multipass output pass). Per group g (one sequence and KV
# head) and query row r (the query heads sharing that KV head), every KV block
# b has left a block maximum of its scores, partial_max[g,r,b], the block's
# sum of exp(score - that maximum), partial_sum[g,r,b], and the block's
# unnormalised output over the value head, partial_out[g,r,b,c] (fp16).

@dataclasses.dataclass(frozen=True)
class SplitWorkload:
    """G groups x R rows, B active blocks, C = value_head_size channels."""

    name: str
    G: int
    R: int
    B: int
    C: int
    seed: int


SPLIT_WORKLOADS = [
    # the multipass path's first depth past 2048 tokens (33 blocks of 64)
    SplitWorkload("split_g2_r8_c128_b33", 2, 8, 33, 128, 2001),
    # depth 4800 (76 blocks), the largest the page measured
    SplitWorkload("split_g4_r8_c128_b76", 4, 8, 76, 128, 2002),
    # 128K tokens (2048 blocks) at the production GQA shape
    SplitWorkload("split_g4_r8_c128_b2048", 4, 8, 2048, 128, 2003),
    # the review's worst staging case: 16 rows, 262,144 tokens (4096 blocks)
    SplitWorkload("split_g2_r16_c128_b4096", 2, 16, 4096, 128, 2004),
]
SPLIT_BY_NAME = {w.name: w for w in SPLIT_WORKLOADS}


def make_split_partials(w: SplitWorkload, variant: int = 0):
    """Return (partial_max f32 [G,R,B], partial_sum f32 [G,R,B],
    partial_out f16 [G,R,B,C]) drawn from a fixed recipe:

      partial_max ~ N(0, 2), plus +6 on one drawn block per row (a dominant
                    block, as an attention sink gives), so the per-block
                    scales span many orders of magnitude;
      partial_sum ~ U[1, 64] (a block of 64 tokens whose largest term is 1);
      partial_out = partial_sum * N(0, 0.3) per channel, rounded to fp16.
    """
    rng = np.random.default_rng(w.seed + 104729 * variant)
    pm = rng.normal(0.0, 2.0, size=(w.G, w.R, w.B))
    hot = rng.integers(0, w.B, size=(w.G, w.R))
    np.put_along_axis(pm, hot[..., None], np.take_along_axis(pm, hot[..., None], 2) + 6.0, 2)
    ps = rng.uniform(1.0, 64.0, size=(w.G, w.R, w.B))
    po = ps[..., None] * rng.normal(0.0, 0.3, size=(w.G, w.R, w.B, w.C))
    return (np.ascontiguousarray(pm.astype(np.float32)),
            np.ascontiguousarray(ps.astype(np.float32)), _f16(po))


def split_random_case(G: int, R: int, B: int, C: int, seed: int, pm_sd: float = 2.0):
    """Small plain cases of the same recipe (no dominant block)."""
    rng = np.random.default_rng(seed)
    pm = rng.normal(0.0, pm_sd, size=(G, R, B))
    ps = rng.uniform(1.0, 64.0, size=(G, R, B))
    po = ps[..., None] * rng.normal(0.0, 0.3, size=(G, R, B, C))
    return (np.ascontiguousarray(pm.astype(np.float32)),
            np.ascontiguousarray(ps.astype(np.float32)), _f16(po))


def attention_scores_values(R: int, n_tokens: int, C: int, seed: int):
    """Raw decode-attention operands for end-to-end checks of the reduce:
    scores [R, n_tokens] ~ N(0, 3) (already scaled q.k) and values
    [n_tokens, C] ~ N(0, 1), both float64."""
    rng = np.random.default_rng(seed)
    return rng.normal(0.0, 3.0, size=(R, n_tokens)), rng.normal(0.0, 1.0, size=(n_tokens, C))
