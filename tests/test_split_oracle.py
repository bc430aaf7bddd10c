"""CPU pins for the split-reduce oracle (oracle/split_reduce_oracle.py).

Each check ties the oracle to something other than itself: math.exp, a
direct softmax over the tokens, closed forms, a hand-worked example, and
planted mistakes that the checks must catch.
"""
import math
import struct
import os

import numpy as np
import pytest

import qsa_inputs as qi
from oracle import split_reduce_oracle as sro

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "split_reduce_hand.txt")


def ulp_error(approx32, exact64):
    """|approx - exact| in units of the last place of the float32 result."""
    a = np.asarray(approx32, np.float32)
    spacing = np.spacing(np.abs(a)).astype(np.float64)
    return np.abs(a.astype(np.float64) - exact64) / spacing


# ------------------------------------------------------------- exponential
def test_exp_f32_within_3_ulp_of_math_exp():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        np.linspace(-86.0, 0.0, 400001, dtype=np.float64),
        -rng.exponential(3.0, size=200000),
        -np.arange(0, 125) * math.log(2.0),            # reduction boundaries
        -(np.arange(0, 125) + 0.5) * math.log(2.0),
    ])
    x = x[x >= -86.0].astype(np.float32)
    got = sro.exp_f32(x)
    exact = np.exp(x.astype(np.float64))
    assert ulp_error(got, exact).max() <= 3.0


def test_exp_f32_special_values():
    assert sro.exp_f32(np.float32(0.0)) == np.float32(1.0)
    assert sro.exp_f32(np.float32(-86.5)) == 0.0
    assert sro.exp_f32(np.float32(-1e30)) == 0.0
    # e^-1 to within an ulp of the correctly rounded value
    assert ulp_error(sro.exp_f32(np.float32(-1.0)), math.exp(-1.0)) <= 1.0


def test_planted_exp_mistakes_are_caught(monkeypatch):
    x = np.linspace(-80.0, 0.0, 50001).astype(np.float32)
    exact = np.exp(x.astype(np.float64))
    monkeypatch.setattr(sro, "LN2_LO_F32", np.float32(0.0))          # dropped low part
    assert ulp_error(sro.exp_f32(x), exact).max() > 3.0
    monkeypatch.undo()
    coeffs = list(sro.TAYLOR_F32)
    coeffs[-2] = np.float32(-1.0)                                     # wrong sign of t
    monkeypatch.setattr(sro, "TAYLOR_F32", coeffs)
    assert ulp_error(sro.exp_f32(x), exact).max() > 3.0


# ------------------------------------------------------ the float64 reduce
def block_partials(scores, values, block):
    """Split-attention partials of a decode: for each block of tokens its
    score maximum, its sum of exp(score - maximum) and its unnormalised
    output (float64; the upstream kernel's job, written out here)."""
    R, n = scores.shape
    B = -(-n // block)
    pm = np.zeros((1, R, B))
    ps = np.zeros((1, R, B))
    po = np.zeros((1, R, B, values.shape[1]))
    for b in range(B):
        s = scores[:, b * block:(b + 1) * block]
        m = s.max(axis=1)
        w = np.exp(s - m[:, None])
        pm[0, :, b] = m
        ps[0, :, b] = w.sum(axis=1)
        po[0, :, b] = w @ values[b * block:(b + 1) * block]
    return pm, ps, po


@pytest.mark.parametrize("n_tokens", [1, 64, 300, 2113])
def test_f64_reduce_equals_softmax_attention(n_tokens):
    """The reduce of the blocks' partials is softmax(scores) @ values over
    every token: the quantity a split flash-attention decode computes."""
    scores, values = qi.attention_scores_values(3, n_tokens, 8, seed=n_tokens)
    pm, ps, po = block_partials(scores, values, 64)
    got = sro.split_reduce_f64(pm, ps, po)[0]
    p = np.exp(scores - scores.max(axis=1, keepdims=True))
    want = (p / p.sum(axis=1, keepdims=True)) @ values
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_hand_example():
    """Values worked by hand from the definition (golden file)."""
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    vals = {r[0]: [float(v) for v in r[1:]] for r in rows}
    pm = np.array(vals["partial_max"]).reshape(1, 1, -1)
    ps = np.array(vals["partial_sum"]).reshape(1, 1, -1)
    B = pm.shape[2]
    po = np.array(vals["partial_out"]).reshape(1, 1, B, -1)
    want = np.array(vals["out"])
    assert np.allclose(sro.split_reduce_f64(pm, ps, po)[0, 0], want, rtol=1e-15, atol=0)


# ------------------------------------------------------- the fp32 procedure
CASES = [(1, 1, 1, 4), (2, 3, 5, 8), (1, 8, 63, 16), (1, 8, 64, 16), (2, 8, 65, 16),
         (1, 4, 130, 128), (1, 16, 300, 32), (2, 8, 33, 128), (1, 2, 129, 8), (1, 3, 1000, 12)]


@pytest.mark.parametrize("G,R,B,C", CASES)
def test_f32_procedure_within_bound(G, R, B, C):
    pm, ps, po = qi.split_random_case(G, R, B, C, seed=B * 7 + C)
    out32 = sro.split_reduce_f32(pm, ps, po)
    rep = sro.bound_report(out32, sro.split_reduce_f64(pm, ps, po), sro.error_bound(pm, ps, po))
    assert rep["ok"], rep
    assert rep["worst_util"] < 0.5, rep


def test_f32_procedure_within_bound_on_workload():
    w = qi.SPLIT_BY_NAME["split_g2_r8_c128_b33"]
    pm, ps, po = qi.make_split_partials(w)
    out32 = sro.split_reduce_f32(pm, ps, po)
    rep = sro.bound_report(out32, sro.split_reduce_f64(pm, ps, po), sro.error_bound(pm, ps, po))
    assert rep["ok"], rep


def test_f32_single_block_is_one_division():
    """B = 1: the scale is exactly 1, so out = fl(partial_out / partial_sum)."""
    pm, ps, po = qi.split_random_case(2, 4, 1, 8, seed=3)
    out32 = sro.split_reduce_f32(pm, ps, po)
    want = po[:, :, 0, :].astype(np.float32) / ps[:, :, 0, None]
    assert np.array_equal(out32.view(np.uint32), want.astype(np.float32).view(np.uint32))


def test_f32_exact_sums_give_the_correctly_rounded_quotient():
    """Equal maxima (every scale 1) and small integer partials: every sum is
    exact in fp32, so out is the correctly rounded quotient of the integer
    sums, for any chunking."""
    rng = np.random.default_rng(11)
    G, R, B, C = 2, 3, 200, 8
    pm = np.full((G, R, B), 1.5, np.float32)
    ps = rng.integers(1, 9, size=(G, R, B)).astype(np.float32)
    po = rng.integers(-20, 21, size=(G, R, B, C)).astype(np.float16)
    out32 = sro.split_reduce_f32(pm, ps, po)
    num = po.astype(np.int64).sum(axis=2)
    den = ps.astype(np.int64).sum(axis=2)
    want = (num.astype(np.float64) / den[..., None]).astype(np.float32)   # exact / exact, one rounding
    assert np.array_equal(out32, want)


def test_planted_reduce_mistakes_are_caught(monkeypatch):
    w = qi.SPLIT_BY_NAME["split_g2_r8_c128_b33"]
    pm, ps, po = qi.make_split_partials(w)
    ref = sro.split_reduce_f64(pm, ps, po)
    bound = sro.error_bound(pm, ps, po)
    # the scale dropped (every block weighted 1)
    monkeypatch.setattr(sro, "exp_f32", lambda x: np.ones_like(np.asarray(x, np.float32)))
    assert not sro.bound_report(sro.split_reduce_f32(pm, ps, po), ref, bound)["ok"]
    monkeypatch.undo()
    # the scale's argument negated (exp(maximum - partial_max), clipped to stay finite)
    orig = sro.exp_f32
    monkeypatch.setattr(sro, "exp_f32", lambda x: orig(np.maximum(-np.asarray(x, np.float32) - 80.0, -86.0)))
    assert not sro.bound_report(sro.split_reduce_f32(pm, ps, po), ref, bound)["ok"]


def test_chunk_count():
    assert [sro.n_chunks(b) for b in (1, 128, 129, 2048, 4096)] == [1, 1, 2, 16, 32]


def test_run_order_is_what_changes_the_bits():
    """The pinned order is observable: on the same inputs a different run
    length gives other fp32 bits (so the kernel must follow this one), while
    both stay within the bound."""
    pm, ps, po = qi.split_random_case(1, 4, 300, 64, seed=21)
    a = sro.split_reduce_f32(pm, ps, po)
    ref, bound = sro.split_reduce_f64(pm, ps, po), sro.error_bound(pm, ps, po)
    old = sro.RUN
    try:
        sro.RUN = 128
        b = sro.split_reduce_f32(pm, ps, po)
    finally:
        sro.RUN = old
    assert not np.array_equal(a, b)
    assert sro.bound_report(a, ref, bound)["ok"] and sro.bound_report(b, ref, bound)["ok"]


# ------------------------------------ a second, scalar model of the procedure
# Written from the statement of the fixed order (chunks of 128 blocks, each
# in runs of 32; inside a run one rounded product then one rounded add per
# block, from 0; runs added in order into the chunk partial, chunk partials
# added in chunk order; one rounded division) and of the exponential (Cody
# and Waite's reduction with ln 2 split, the degree-7 Taylor polynomial in
# Horner form, exact scaling by 2^n, flush below -86), in plain Python
# floats, each operation's binary64 result rounded to binary32 with struct.
# For +, -, * and / on binary32 operands the binary64 result rounded once
# more to binary32 equals the correctly rounded binary32 result (53 >= 2*24
# + 2), so this is IEEE binary32 arithmetic, computed another way.
def _f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


_LN2_HI = 0.693145751953125                     # 16 significant bits: n * LN2_HI is exact
_LN2_LO = _f32(math.log(2.0) - _LN2_HI)
_LOG2E = _f32(1.0 / math.log(2.0))


def _exp_scalar(x):
    if x < -86.0:
        return 0.0
    n = float(round(_f32(x * _LOG2E)))           # Python's round() is half-to-even
    t = _f32(_f32(x - _f32(n * _LN2_HI)) - _f32(n * _LN2_LO))
    p = _f32(1.0 / math.factorial(7))
    for k in range(6, -1, -1):
        p = _f32(_f32(p * t) + _f32(1.0 / math.factorial(k)))
    return _f32(p * math.ldexp(1.0, int(n)))


def split_reduce_scalar(pm, ps, po, chunk=128, run=32):
    G, R, B = pm.shape
    C = po.shape[3]
    out = np.zeros((G, R, C), np.float32)
    for g in range(G):
        for r in range(R):
            m = max(float(v) for v in pm[g, r])
            scale = [_exp_scalar(_f32(float(pm[g, r, b]) - m)) for b in range(B)]
            tot_s, tot_o = 0.0, [0.0] * C
            for c0 in range(0, B, chunk):
                part_s, part_o = 0.0, [0.0] * C
                for r0 in range(c0, min(B, c0 + chunk), run):
                    run_s, run_o = 0.0, [0.0] * C
                    for b in range(r0, min(B, r0 + run)):
                        run_s = _f32(run_s + _f32(scale[b] * float(ps[g, r, b])))
                        for c in range(C):
                            run_o[c] = _f32(run_o[c] + _f32(scale[b] * float(po[g, r, b, c])))
                    part_s = _f32(part_s + run_s)
                    part_o = [_f32(a + v) for a, v in zip(part_o, run_o)]
                tot_s = _f32(tot_s + part_s)
                tot_o = [_f32(a + v) for a, v in zip(tot_o, part_o)]
            out[g, r] = [_f32(v / tot_s) for v in tot_o]
    return out


def test_exp_scalar_model_equals_exp_f32():
    """The two exponentials agree bit for bit (reduction boundaries, the flush
    threshold and random arguments included)."""
    rng = np.random.default_rng(8)
    x = np.concatenate([-rng.exponential(4.0, size=3000), np.linspace(-86.0, 0.0, 2001),
                        -np.arange(0, 125) * math.log(2.0), [-85.999, -86.0, -86.001, -0.0]])
    x = x.astype(np.float32)
    got = np.array([_exp_scalar(float(v)) for v in x], np.float32)
    assert np.array_equal(got.view(np.uint32), sro.exp_f32(x).view(np.uint32))


@pytest.mark.parametrize("G,R,B,C", [(1, 1, 1, 4), (1, 2, 31, 4), (1, 3, 33, 8), (2, 2, 100, 4),
                                     (1, 2, 129, 8), (1, 1, 257, 4), (1, 2, 300, 12)])
def test_f32_procedure_equals_scalar_model(G, R, B, C):
    """split_reduce_f32 equals the scalar model bit for bit, on block counts
    that are and are not multiples of the run (32) and chunk (128) sizes."""
    pm, ps, po = qi.split_random_case(G, R, B, C, seed=1000 + B)
    got = sro.split_reduce_f32(pm, ps, po)
    want = split_reduce_scalar(pm, ps, po)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_scalar_model_catches_a_changed_order():
    """The scalar model sees a different run length (its bits differ), so the
    equality above pins the order, not just the value."""
    pm, ps, po = qi.split_random_case(1, 2, 300, 12, seed=1300)
    assert not np.array_equal(split_reduce_scalar(pm, ps, po, run=32),
                              split_reduce_scalar(pm, ps, po, run=128))
