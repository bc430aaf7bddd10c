"""CPU pins for the oracle: it is checked against things other than itself.

Each pin is a function that takes the function under test and raises
AssertionError on a mismatch. The oracle must pass every pin, and the
planted-mistake tests at the end show that plausible mistakes (a dropped
ReLU, a wrong sign, a transposed operand, a floor instead of a ceil, a lost
dead-tail bonus, a reversed tie-break, a reordered tail sum) each fail one.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import qsa_inputs as qi
from oracle import qsa_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        txt = "".join(line for line in f if not line.lstrip().startswith("#"))
    return json.loads(txt)


def _fl(v):
    return float(v) if not isinstance(v, str) else float(v)


# ----------------------------------------------------------------- exact math
def exact_scores(q, kb, n_kv, block):
    """Brute force over exact rationals (fp16 values are dyadic)."""
    nb = -(-n_kv // block)
    nq, H, D = q.shape
    out = [[None] * nb for _ in range(nq)]
    S = [[None] * nb for _ in range(nq)]
    for a in range(nq):
        for b in range(nb):
            tot = Fraction(0)
            tot_abs = Fraction(0)
            for h in range(H):
                pre = Fraction(0)
                for i in range(D):
                    p = Fraction(float(q[a, h, i])) * Fraction(float(kb[b, i]))
                    pre += p
                    tot_abs += abs(p)
                tot += max(pre, Fraction(0))
            out[a][b] = tot
            S[a][b] = tot_abs
    return out, S


def fl32(x):
    """Round a Python float (binary64) to binary32, round to nearest even."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def tail_struct_model(q, kb, n_kv, block):
    """Second, independent fp32 tail model: scalar binary64 ops rounded to
    binary32 after every step (innocuous double rounding for + and *)."""
    nb = -(-n_kv // block)
    nq, H, D = q.shape
    res = []
    for a in range(nq):
        t = 0.0
        for h in range(H):
            acc = 0.0
            for i in range(D):
                acc = fl32(acc + fl32(float(q[a, h, i]) * float(kb[nb - 1, i])))
            t = fl32(t + (acc if acc > 0.0 else 0.0))
        res.append(fl32(t + 1.0e9))
    return np.array(res, dtype=np.float32)


def rne_f16_exact(x):
    """IEEE binary16 round-to-nearest-even of a finite binary64 value, from
    the format's definition (1 sign, 5 exponent, 10 fraction bits, bias 15)."""
    if math.isnan(x):
        return float("nan")
    if math.isinf(x):
        return x
    fx = Fraction(x)
    sign = -1 if fx < 0 or (fx == 0 and math.copysign(1.0, x) < 0) else 1
    ax = abs(fx)
    if ax == 0:
        return math.copysign(0.0, sign)
    e = 0
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    while Fraction(2) ** e > ax:
        e -= 1
    e = max(e, -14)                       # subnormals share the quantum 2^-24
    quantum = Fraction(2) ** (e - 10)
    n = ax / quantum
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * quantum
    if val > 65504:
        return math.copysign(float("inf"), sign)
    return math.copysign(float(val), sign)


# ----------------------------------------------------------------------- pins
def pin_bruteforce(scores_fn, S_fn=orc.abs_product_sum_f64):
    for seed, (nq, H, D, n_kv, block) in enumerate(
            [(1, 1, 1, 1, 1), (2, 3, 5, 9, 2), (3, 2, 16, 10, 2), (3, 3, 16, 17, 4), (2, 1, 7, 5, 1)]):
        q, kb = qi.random_case(nq, H, D, -(-n_kv // block), seed=100 + seed, scale=2.0)
        ex, exS = exact_scores(q, kb, n_kv, block)
        got = scores_fn(q, kb, n_kv, block)
        gotS = S_fn(q, kb, n_kv, block)
        assert got.shape == (nq, -(-n_kv // block))
        for a in range(nq):
            for b in range(got.shape[1]):
                tol = float(exS[a][b]) * 2.0 ** -44
                assert abs(got[a, b] - float(ex[a][b])) <= tol, (a, b, got[a, b], float(ex[a][b]))
                assert abs(gotS[a, b] - float(exS[a][b])) <= tol


def pin_coordinate_coded(scores_fn):
    nq, H, D, n_kv, block = 5, 3, 16, 77, 4
    nb = -(-n_kv // block)
    q, kb = qi.coordinate_coded_case(nq, H, D, nb)
    got = scores_fn(q, kb, n_kv, block)
    assert got.shape == (nq, nb)
    qf = q.astype(np.float64)
    for a in range(nq):
        for b in range(nb):
            want = sum(max(qf[a, h, b % D], 0.0) for h in range(H))
            assert got[a, b] == want, (a, b, got[a, b], want)


def pin_one_hot(scores_fn):
    nq, H, D, nb = 4, 5, 16, 9
    q, kb = qi.one_hot_case(nq, H, D, nb, seed=7)
    cq = q.astype(np.float64).argmax(axis=2)
    ck = kb.astype(np.float64).argmax(axis=1)
    got = scores_fn(q, kb, nb * 3, 3)
    for a in range(nq):
        for b in range(nb):
            assert got[a, b] == sum(1 for h in range(H) if cq[a, h] == ck[b])


def pin_relu_identity(scores_fn):
    """relu(x) - relu(-x) = x: scores(q) - scores(-q) = sum_h q_h . kb, and
    equal heads give H times the one-head score."""
    q, kb = qi.random_case(6, 4, 32, 11, seed=5)
    n_kv, block = 11 * 8, 8
    d = scores_fn(q, kb, n_kv, block) - scores_fn(-q, kb, n_kv, block)
    qsum = q.astype(np.float64).sum(axis=1)
    kbf = kb.astype(np.float64)
    for a in range(6):
        for b in range(11):
            lin = math.fsum(float(qsum[a, i]) * float(kbf[b, i]) for i in range(32))
            assert abs(d[a, b] - lin) <= 1e-12 * (1 + abs(lin))
    q1 = np.repeat(q[:, :1, :], 4, axis=1)
    s1 = scores_fn(q[:, :1, :], kb, n_kv, block)
    s4 = scores_fn(q1, kb, n_kv, block)
    assert np.allclose(s4, 4 * s1, rtol=1e-14, atol=0)


def pin_partition(part_fn):
    for n_kv in list(range(0, 70)) + [4000, 1024, 32805, 131072, 131073]:
        for block in (1, 2, 3, 7, 64):
            blocks = {t // block for t in range(n_kv)} if n_kv < 5000 else None
            nb, n_full, tail = part_fn(n_kv, block)
            if blocks is not None:
                assert nb == len(blocks)
                full = sum(1 for b in blocks if (b + 1) * block <= n_kv)
                assert n_full == full
                assert tail == (full != nb)
            else:
                assert nb * block >= n_kv > (nb - 1) * block
                assert n_full * block <= n_kv < (n_full + 1) * block


def pin_hand_example(scores_fn, tail_fn, select_fn, S_fn=orc.abs_product_sum_f64,
                     bound_fn=orc.error_bound):
    g = _load_golden("hand_example.txt")
    q = np.array(g["q"], dtype=np.float16)
    kb = np.array(g["kb"], dtype=np.float16)
    s = scores_fn(q, kb, g["n_kv"], g["block"])
    assert np.array_equal(s[:, :2], np.array(g["full_scores"]))
    # S and the bound B, worked by hand in the fixture from the printed formula
    S = S_fn(q, kb, g["n_kv"], g["block"])
    assert np.array_equal(S[:, :2], np.array(g["S_full"]))
    B = bound_fn(S[:, :2], s[:, :2])
    assert np.allclose(B, np.array(g["B_full"]), rtol=1e-13, atol=0.0)
    tail = tail_fn(q, kb, g["n_kv"], g["block"])
    assert tail.dtype == np.float32
    assert np.array_equal(tail, np.array(g["tail"], dtype=np.float32))
    full = np.concatenate([np.array(g["full_scores"]), tail[:, None].astype(np.float64)], axis=1)
    assert np.array_equal(select_fn(full, 2), np.array(g["top2"]))
    assert np.array_equal(select_fn(full, 4), np.array(g["top4"]))


def pin_tail(tail_fn):
    cases = [(3, 2, 16, 37, 8, 1.0), (4, 8, 128, 131073, 64, 8.0 / math.sqrt(128)),
             (2, 4, 64, 4000, 64, 1.0), (5, 3, 32, 9, 4, 30.0)]
    for seed, (nq, H, D, n_kv, block, sc) in enumerate(cases):
        nb = -(-n_kv // block)
        q, kb = qi.random_case(nq, H, D, nb, seed=200 + seed, scale=sc)
        got = tail_fn(q, kb, n_kv, block)
        want = tail_struct_model(q, kb, n_kv, block)
        assert got.view(np.uint32).tolist() == want.view(np.uint32).tolist()
        s64 = orc.scores_f64(q, kb, n_kv, block)[:, -1]
        near = (s64 + 1e9).astype(np.float32)
        ulp = np.float32(64.0)
        assert np.all(np.abs(got.astype(np.float64) - near.astype(np.float64)) <= ulp)
    q, kb = qi.random_case(2, 2, 16, 4, seed=3)
    assert tail_fn(q, kb, 4 * 8, 8) is None


def pin_select(select_fn):
    g = _load_golden("select_ties.txt")
    s = np.array([[_fl(v) for v in row] for row in g["scores"]], dtype=np.float32)
    assert np.array_equal(select_fn(s, 3), np.array(g["top3"]))
    assert np.array_equal(select_fn(s[:1], 7)[0], np.array(g["top7_row0"]))
    for seed, kind in enumerate(["normal", "ties", "signed0", "const"]):
        for nb, k in [(1, 1), (5, 3), (40, 8), (100, 100), (33, 64), (257, 31)]:
            sc = qi.random_scores(4, nb, seed=300 + seed, kind=kind)
            got = select_fn(sc, k)
            for r in range(4):
                vals = [float(v) for v in sc[r]]
                want = sorted(range(nb), key=lambda b: (-vals[b], b))[:k]
                want = want + [-1] * (k - len(want))
                assert got[r].tolist() == want, (kind, nb, k, r)
    assert select_fn(np.zeros((3, 0), np.float32), 4).tolist() == [[-1] * 4] * 3


# ---------------------------------------------------------------- the oracle
def test_oracle_bruteforce():
    pin_bruteforce(orc.scores_f64)


def test_oracle_coordinate_coded():
    pin_coordinate_coded(orc.scores_f64)


def test_oracle_one_hot():
    pin_one_hot(orc.scores_f64)


def test_oracle_relu_identity():
    pin_relu_identity(orc.scores_f64)


def test_oracle_partition():
    pin_partition(orc.block_partition)


def test_oracle_hand_example():
    pin_hand_example(orc.scores_f64, orc.tail_scores_f32, orc.select_topk)


def test_oracle_tail_bitwise_second_model():
    pin_tail(orc.tail_scores_f32)


def test_oracle_select():
    pin_select(orc.select_topk)


def test_oracle_empty_context():
    q, kb = qi.random_case(3, 2, 16, 0, seed=1)
    assert orc.scores_f64(q, kb, 0, 64).shape == (3, 0)
    assert orc.tail_scores_f32(q, kb, 0, 64) is None
    s_ref, S, B, tail = orc.reference_scores(q, kb, 0, 64)
    assert s_ref.shape == S.shape == B.shape == (3, 0) and tail is None
    assert orc.select_topk(s_ref, 5).tolist() == [[-1] * 5] * 3


def test_oracle_ragged_shapes_and_tail_column():
    for nq in (1, 17, 129):
        for nb_target, tail in [(1, False), (1, True), (63, True), (129, False), (129, True)]:
            block = 4
            n_kv = nb_target * block - (2 if tail else 0)
            q, kb = qi.random_case(nq, 2, 16, nb_target, seed=nq + nb_target)
            s_ref, S, B, t = orc.reference_scores(q, kb, n_kv, block)
            assert s_ref.shape == (nq, nb_target)
            assert (t is not None) == tail
            if tail:
                assert np.array_equal(s_ref[:, -1], t.astype(np.float64))
                assert np.all(B[:, -1] == 0)
            assert np.all(B[:, :nb_target - (1 if tail else 0)] > 0)


def test_oracle_conversion_rne():
    specials = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, -65520.0, 65536.0, 1e6,
                2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14,
                2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -11 + 2.0 ** -20,
                2049.0, 2051.0, 4097.0, 0.1, -0.3, 1.0 / 3.0, float("inf"), float("-inf")]
    rng = np.random.default_rng(9)
    rand = (rng.normal(size=2000) * np.exp2(rng.integers(-30, 17, size=2000))).tolist()
    vals = np.array(specials + rand, dtype=np.float32)
    got = orc.f32_to_f16(vals)
    for v, g16 in zip(vals.tolist(), got.tolist()):
        want = rne_f16_exact(float(np.float32(v)))
        assert (g16 == want and math.copysign(1, g16) == math.copysign(1, want)), (v, g16, want)
    nan = orc.f32_to_f16(np.array([float("nan")], np.float32))
    assert np.isnan(nan[0])
    # every fp16 value round-trips unchanged
    allh = np.arange(0, 1 << 16, dtype=np.uint16).view(np.float16)
    fin = allh[np.isfinite(allh)]
    assert np.array_equal(orc.f32_to_f16(fin.astype(np.float32)).view(np.uint16), fin.view(np.uint16))


def test_bound_checker_negative_control():
    w = qi.WORKLOADS[0]
    q, kb = qi.make_inputs(w)
    s_ref, S, B, tail = orc.reference_scores(q, kb, w.n_kv, w.block)
    full = B > 0
    assert full.sum() > 0
    ok = orc.bound_report(s_ref + 0.5 * B, s_ref, B)
    assert ok["ok"] and 0.49 < ok["worst_util"] <= 0.5 + 1e-9
    bad = orc.bound_report(s_ref + 2.5 * B, s_ref, B)
    assert not bad["ok"] and bad["n_bad"] == int(full.sum())
    # the tail column has B == 0: one ulp off must fail
    if tail is not None:
        s = s_ref.copy()
        s[0, -1] = float(np.nextafter(np.float32(s[0, -1]), np.float32(np.inf)))
        assert not orc.bound_report(s, s_ref, B)["ok"]


def test_bound_checker_at_the_hand_worked_bound():
    """The checker passes an error just below the hand-worked B and fails one
    just above it (golden hand example, full entries)."""
    g = _load_golden("hand_example.txt")
    s_ref = np.array(g["full_scores"], dtype=np.float64)
    B_hand = np.array(g["B_full"], dtype=np.float64)
    S = np.array(g["S_full"], dtype=np.float64)
    B = orc.error_bound(S, s_ref)
    for sign in (1.0, -1.0):
        assert orc.bound_report(s_ref + sign * B_hand * (1 - 1e-9), s_ref, B)["ok"]
        bad = orc.bound_report(s_ref + sign * B_hand * (1 + 1e-9), s_ref, B)
        assert not bad["ok"] and bad["n_bad"] == B.size


@pytest.mark.parametrize("name,value", [("BOUND_REL_S", 2.0 ** -9), ("BOUND_REL_S", 2.0 ** -7),
                                        ("BOUND_REL_SCORE", 0.0), ("BOUND_REL_SCORE", 2.0 ** -24)])
def test_planted_bound_mistakes_are_caught(monkeypatch, name, value):
    """A wrong exponent on the S term or a dropped / shrunk |score| term in B
    fails the hand-worked bound pin."""
    monkeypatch.setattr(orc, name, value)
    with pytest.raises(AssertionError):
        pin_hand_example(orc.scores_f64, orc.tail_scores_f32, orc.select_topk)


def test_selection_checker_controls():
    w = qi.WORKLOADS[0]
    q, kb = qi.make_inputs(w)
    s_ref, S, B, _ = orc.reference_scores(q, kb, w.n_kv, w.block)
    ids = orc.select_topk(s_ref, w.k)
    rep = orc.selection_report(ids, s_ref, B, w.k)
    assert rep["ok"], rep
    swapped = ids.copy()
    # replace the last selected id by the lowest-scoring block of the row
    swapped[0, -1] = int(np.argmin(s_ref[0]))
    assert not orc.selection_report(swapped, s_ref, B, w.k)["ok"]
    rev = ids[:, ::-1].copy()
    assert not orc.selection_report(rev, s_ref, B, w.k)["ok"]
    dup = ids.copy()
    dup[1, 1] = dup[1, 0]
    assert not orc.selection_report(dup, s_ref, B, w.k)["ok"]


def test_workload_recipe():
    shapes = [(16, 4, 64, 63, 8), (256, 8, 128, 16, 8), (256, 8, 128, 513, 32),
              (256, 8, 128, 2048, 64), (4096, 16, 128, 2049, 64)]
    for w, (nq, H, D, nb, k) in zip(qi.WORKLOADS, shapes):
        assert (w.nq, w.H, w.D, w.nb, w.k, w.block) == (nq, H, D, nb, k, 64)
    w5 = qi.WORKLOADS[4]
    _, kb = qi.make_inputs(w5)
    kf = kb.astype(np.float64)
    hot = np.nonzero((np.count_nonzero(kf, axis=1) == 1) & (kf.max(axis=1) == 4.0))[0]
    assert len(hot) == 21
    coords = kf[hot].argmax(axis=1)
    assert len(set(coords.tolist())) < len(coords)          # a shared coordinate -> exact ties


# ------------------------------------------------------- planted mistakes
def test_planted_dropped_relu_is_caught(monkeypatch):
    monkeypatch.setattr(orc, "_relu", lambda x: x)
    with pytest.raises(AssertionError):
        pin_coordinate_coded(orc.scores_f64)
    with pytest.raises(AssertionError):
        pin_relu_identity(orc.scores_f64)


def test_planted_sign_and_transpose_are_caught(monkeypatch):
    orig = orc._preactivations_f64
    monkeypatch.setattr(orc, "_preactivations_f64", lambda q, kb: -orig(q, kb))
    with pytest.raises(AssertionError):
        pin_bruteforce(orc.scores_f64, S_fn=lambda *a: orc.abs_product_sum_f64(*a))
    monkeypatch.setattr(orc, "_preactivations_f64", lambda q, kb: orig(q, kb[:, ::-1]))
    with pytest.raises(AssertionError):
        pin_coordinate_coded(orc.scores_f64)


def test_planted_partition_floor_is_caught():
    with pytest.raises(AssertionError):
        pin_partition(lambda n_kv, block: (n_kv // block, n_kv // block, n_kv % block != 0))


def test_planted_tail_mistakes_are_caught(monkeypatch):
    monkeypatch.setattr(orc, "TAIL_BONUS_F32", np.float32(0.0))
    with pytest.raises(AssertionError):
        pin_hand_example(orc.scores_f64, orc.tail_scores_f32, orc.select_topk)
    monkeypatch.undo()

    def tail_pairwise(q, kb, n_kv, block):   # same math, another summation order
        nb = -(-n_kv // block)
        pre = (q.astype(np.float32) * kb[nb - 1].astype(np.float32)).sum(axis=2, dtype=np.float32)
        return np.maximum(pre, np.float32(0)).sum(axis=1, dtype=np.float32) + np.float32(1e9)
    with pytest.raises(AssertionError):
        pin_tail(tail_pairwise)


def test_planted_select_mistakes_are_caught():
    def reversed_tie(s, k):
        s = np.asarray(s, np.float64)
        nb = s.shape[1]
        out = np.full((s.shape[0], k), -1, np.int32)
        o = np.lexsort((-np.broadcast_to(np.arange(nb), s.shape), -s), axis=-1)[:, :k]
        out[:, :o.shape[1]] = o
        return out

    def ascending(s, k):
        s = np.asarray(s, np.float64)
        out = np.full((s.shape[0], k), -1, np.int32)
        o = np.lexsort((np.broadcast_to(np.arange(s.shape[1]), s.shape), s), axis=-1)[:, :k]
        out[:, :o.shape[1]] = o
        return out

    def signed_zero_distinct(s, k):   # orders -0.0 below +0.0 (compares bit patterns)
        s = np.asarray(s, np.float32)
        key = np.where(s.view(np.int32) < 0, ~s.view(np.int32) & 0x7FFFFFFF, s.view(np.int32) | 0)
        key = key.astype(np.int64) + np.where(s.view(np.int32) < 0, 0, 1 << 31)
        out = np.full((s.shape[0], k), -1, np.int32)
        o = np.lexsort((np.broadcast_to(np.arange(s.shape[1]), s.shape), -key), axis=-1)[:, :k]
        out[:, :o.shape[1]] = o
        return out

    for bad in (reversed_tie, ascending, signed_zero_distinct):
        with pytest.raises(AssertionError):
            pin_select(bad)
