"""CPU oracle for the QSA block scorer and top-k block selection.

TEST INFRASTRUCTURE. Only the test suite, the smoke check in
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this module. The product (the CUDA library and
its Python binding) never imports, calls or links it, and it imports nothing
from the product.

Everything here is the plain definition, written out in float64 numpy (or in
float32 where the pages fix a float32 procedure), with no blocking, fusion or
reordering beyond what the definition states. Sources, by page and section:

  [P228-1]  Strata pull request 228, part 1 "qsa_block_scores_wmma: the prompt
            scorer arm on tensor cores": the score definition, the error bound
            B, the bitwise tail-block requirement, the parity suite (ragged
            tiles, x8 headroom, n_kv = 0, one-hot / coordinate-coded fixtures,
            write-set canaries, selection-ID agreement, +2.5*B negative
            control, worst bound utilisation).
  [P856-W]  Strata pull request 856 ("hip: RDNA3 (gfx1100) WMMA kernel for
            the QSA block-score select/scorer"), section "What": the shared
            tail-block kernel and the +1e9 dead-tail rule.
  [P856-A]  the same page, section "Arithmetic contract and parity": the bound
            again, and selection agreement with a near-tie-gap guard.

Readings where the pages are silent (each also listed in the design notes):
  R1  nb = ceil(n_kv / block); blocks 0..n_full-1 are full, block nb-1 is the
      tail when n_kv % block != 0. kb holds one key row per block, the tail's
      included.
  R2  "+1e9" adds 1e9 (an fp32 add of 1e9f) to the tail score; it does not
      replace it.
  R3  The tail is computed in one pinned fp32 order: per head, a sequential
      sum over i of the (exact) fp32 products; then a sequential sum over h of
      max(acc_h, 0); then + 1e9f. Every operation is IEEE binary32
      round-to-nearest-even.
  R4  Top-k order: descending score; equal scores -> smaller block index
      first; -0.0 equals +0.0; when nb < k the ids are padded with -1.
  R5  S(qi,b) sums |q*kb| over every head, the clipped ones included.
  R6  fp32 -> fp16 is IEEE round-to-nearest-even; overflow gives +-inf.

Functions whose result has a closed definition are pinned by the CPU tests
against brute force (exact rationals), closed forms and special cases; none
is marked "parity unpinned".
"""
from __future__ import annotations

import numpy as np

TAIL_BONUS_F32 = np.float32(1.0e9)   # [P856-W] the dead-tail constant (1e9 is exact in fp32)
BOUND_REL_S = 2.0 ** -9.5            # [P228-1] B = 2^-9.5 * S + 8 * 2^-24 * |score_ref|
BOUND_REL_SCORE = 8.0 * 2.0 ** -24


# ---------------------------------------------------------------- partition
def block_partition(n_kv: int, block: int):
    """Reading R1: (nb, n_full, has_tail) for a context of n_kv tokens."""
    if block < 1 or n_kv < 0:
        raise ValueError("block must be >= 1 and n_kv >= 0")
    nb = -(-n_kv // block)
    n_full = n_kv // block
    return nb, n_full, (n_kv % block) != 0


# ------------------------------------------------------------------- scores
def _relu(x):
    return np.maximum(x, 0.0)


def _preactivations_f64(q, kb):
    """pre[qi, h, b] = sum_i q[qi, h, i] * kb[b, i] in float64 ([P228-1])."""
    nq, H, D = q.shape
    q2 = q.astype(np.float64).reshape(nq * H, D)
    pre = q2 @ kb.astype(np.float64).T
    return pre.reshape(nq, H, kb.shape[0])


def scores_f64(q, kb, n_kv: int, block: int):
    """score(qi, b) = sum_h relu(sum_i kb[b, i] * q[qi, h, i]), float64.

    [P228-1] gives the definition. Returned for every block 0..nb-1; the tail
    block's entry here is its plain score, without the dead-tail bonus (see
    ``tail_scores_f32`` for the value the path must produce there).
    """
    nb, _, _ = block_partition(n_kv, block)
    _check_shapes(q, kb, nb)
    if nb == 0 or q.shape[0] == 0:
        return np.zeros((q.shape[0], nb), dtype=np.float64)
    pre = _preactivations_f64(q, kb[:nb])
    return _relu(pre).sum(axis=1)


def abs_product_sum_f64(q, kb, n_kv: int, block: int):
    """S(qi, b) = sum_h sum_i |q[qi, h, i] * kb[b, i]| (reading R5), float64."""
    nb, _, _ = block_partition(n_kv, block)
    _check_shapes(q, kb, nb)
    if nb == 0 or q.shape[0] == 0:
        return np.zeros((q.shape[0], nb), dtype=np.float64)
    pre_abs = _preactivations_f64(np.abs(q), np.abs(kb[:nb]))
    return pre_abs.sum(axis=1)


def error_bound(S, s_ref):
    """B(qi, b) = 2^-9.5 * S + 8 * 2^-24 * |score_ref| ([P228-1], [P856-A])."""
    return BOUND_REL_S * np.asarray(S, np.float64) + BOUND_REL_SCORE * np.abs(np.asarray(s_ref, np.float64))


def tail_scores_f32(q, kb, n_kv: int, block: int):
    """Tail-block scores for every query, fp32, bitwise (readings R2, R3).

    [P228-1] requires the tail bitwise equal to the shared tail kernel's; [P856-W]
    adds 1e9 to it. Returns None when n_kv is a multiple of block (no tail).
    """
    nb, _, has_tail = block_partition(n_kv, block)
    if not has_tail:
        return None
    _check_shapes(q, kb, nb)
    nq, H, D = q.shape
    krow = kb[nb - 1].astype(np.float32)
    q32 = q.astype(np.float32)
    acc = np.zeros((nq, H), dtype=np.float32)
    for i in range(D):
        prod = q32[:, :, i] * krow[i]          # exact: fp16 * fp16 fits in fp32
        acc = acc + prod                       # fp32 add, round to nearest even
    t = np.zeros(nq, dtype=np.float32)
    for h in range(H):
        t = t + np.maximum(acc[:, h], np.float32(0.0))
    return t + TAIL_BONUS_F32


def reference_scores(q, kb, n_kv: int, block: int):
    """What the path must produce, for checking.

    Returns (s_ref, S, B, tail):
      s_ref f64 [nq, nb]: the float64 definition for full blocks, and in the
                          tail column the fp32 tail value (which is exact).
      S, B  f64 [nq, nb]: absolute product sum and error bound; B is 0 in the
                          tail column, which must match bitwise.
      tail  f32 [nq] or None.
    """
    s_ref = scores_f64(q, kb, n_kv, block)
    S = abs_product_sum_f64(q, kb, n_kv, block)
    B = error_bound(S, s_ref)
    tail = tail_scores_f32(q, kb, n_kv, block)
    if tail is not None:
        s_ref[:, -1] = tail.astype(np.float64)
        S[:, -1] = 0.0
        B[:, -1] = 0.0
    return s_ref, S, B, tail


# ------------------------------------------------------------------- select
def select_topk(scores, k: int):
    """ids[qi] = the k block indices with the largest scores (reading R4).

    [P228-1] and [P856-A] select the top-k blocks per query. Order: score
    descending, then block index ascending; -0.0 == +0.0; ids padded with -1
    when nb < k. Computed by a stable lexicographic sort of (-score, index).
    """
    if k < 1:
        raise ValueError("k must be >= 1")
    s = np.asarray(scores, dtype=np.float64)
    nq, nb = s.shape
    out = np.full((nq, k), -1, dtype=np.int32)
    if nq == 0 or nb == 0:
        return out
    idx = np.broadcast_to(np.arange(nb), s.shape)
    order = np.lexsort((idx, -s), axis=-1)
    kk = min(k, nb)
    out[:, :kk] = order[:, :kk]
    return out


# --------------------------------------------------------------- conversion
def f32_to_f16(x):
    """fp32 -> fp16, IEEE round to nearest even, overflow to +-inf (R6)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float32).astype(np.float16)


# ----------------------------------------------------------------- checkers
def bound_report(s_gpu, s_ref, B):
    """Check |s_gpu - s_ref| <= B for every entry ([P228-1]).

    Returns dict(ok, worst_util, n_bad, worst_index). Entries with B == 0 must
    be exact. worst_util = max |err| / B over entries with B > 0.
    """
    s = np.asarray(s_gpu, dtype=np.float64)
    err = np.abs(s - s_ref)
    bad = ~(err <= B)
    pos = B > 0
    util = np.zeros_like(err)
    util[pos] = err[pos] / B[pos]
    worst = float(util.max()) if util.size else 0.0
    worst_idx = tuple(int(v) for v in np.unravel_index(np.argmax(util), util.shape)) if util.size else None
    return {"ok": not bool(bad.any()), "worst_util": worst, "n_bad": int(bad.sum()),
            "worst_index": worst_idx}


def selection_report(ids_gpu, s_ref, B, k: int):
    """Selection-ID agreement with a near-tie-gap guard ([P228-1], [P856-A]).

    Per query, with the oracle's order on s_ref, s_k and s_k1 its k-th and
    (k+1)-th scores and g = 2 * max(B_k, B_k1):
      * ids are distinct, in range, padded with -1 exactly when nb < k;
      * if s_k - s_k1 >= g, the id set equals the oracle's; otherwise every
        block with s_ref > s_k + g is selected and every selected block has
        s_ref >= s_k - g (the row is counted as guarded);
      * consecutive ids are ordered within noise:
        s_ref[a] >= s_ref[b] - (B[a] + B[b]);
      * if every gap between consecutive oracle entries among the first
        min(k+1, nb) is >= twice the larger of their bounds, the ids equal the
        oracle's exactly, order included (counted as exact rows).
    """
    ids = np.asarray(ids_gpu)
    nq, nb = s_ref.shape
    ref = select_topk(s_ref, k)
    kk = min(k, nb)
    fails = []
    guarded = 0
    exact_rows = 0
    for r in range(nq):
        row = ids[r]
        if np.any(row[kk:] != -1):
            fails.append((r, "padding"))
            continue
        sel = row[:kk]
        if kk and (sel.min() < 0 or sel.max() >= nb or len(set(sel.tolist())) != kk):
            fails.append((r, "range/duplicate"))
            continue
        if kk == 0:
            exact_rows += 1
            continue
        sr, br = s_ref[r], B[r]
        if np.any(sr[sel[:-1]] < sr[sel[1:]] - (br[sel[:-1]] + br[sel[1:]])):
            fails.append((r, "order"))
            continue
        o = ref[r, :kk]
        if kk < nb:
            ok_idx = int(o[kk - 1])
            nxt = int(np.lexsort((np.arange(nb), -sr))[kk])
            g = 2.0 * max(br[ok_idx], br[nxt])
            if sr[ok_idx] - sr[nxt] >= g:
                if set(sel.tolist()) != set(o.tolist()):
                    fails.append((r, "set"))
                    continue
            else:
                guarded += 1
                sk = sr[ok_idx]
                must = np.nonzero(sr > sk + g)[0]
                if not set(must.tolist()) <= set(sel.tolist()) or np.any(sr[sel] < sk - g):
                    fails.append((r, "guarded-set"))
                    continue
        m = min(k + 1, nb)
        full_order = np.lexsort((np.arange(nb), -sr))[:m]
        gaps = sr[full_order[:-1]] - sr[full_order[1:]]
        need = 2.0 * np.maximum(br[full_order[:-1]], br[full_order[1:]])
        if np.all(gaps >= need) or m == 1:
            if not np.array_equal(sel, o):
                fails.append((r, "exact"))
                continue
            exact_rows += 1
    return {"ok": not fails, "fails": fails[:10], "n_fail": len(fails),
            "guarded_rows": guarded, "exact_rows": exact_rows}


def _check_shapes(q, kb, nb):
    if q.ndim != 3 or kb.ndim != 2 or q.shape[2] != kb.shape[1]:
        raise ValueError("q must be [nq,H,D] and kb [nb,D] with matching D")
    if kb.shape[0] < nb:
        raise ValueError("kb must hold one row per block")
