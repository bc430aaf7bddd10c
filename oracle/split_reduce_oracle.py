"""CPU oracle for the flash-attention decode split reduce (the second workload).

TEST INFRASTRUCTURE. Only the test suite, the smoke check in
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this module. The product never imports, calls
or links it, and it imports nothing from the product.

Source: 1bit-MONSTER llama.cpp pull request 30 (flash attention decode split,
multipass reduce), sections "What" and "Changes", and its review:

  [PR30-W]  "What": the reduce ends with an output pass over every KV block;
            the per-block scale is exp(partial_max[block] - maximum), computed
            once per (row, block) rather than once per (block, element).
  [PR30-C]  "Changes": the lane-strided sum pass computes the per-block scale,
            stores it in a per-row stage and publishes each row's sum; the
            output pass accumulates fp32 over the blocks from fp16 partial
            outputs, four channels per work item; the per-channel accumulation
            order over blocks is what makes the result bit-identical.
  [PR30-R]  the review: the scale stage must be bounded (tile the output pass
            over block chunks with a fixed-size stage); value_head_size must be
            a multiple of 4.

The reduce, per group g and row r (float64 definition, split_reduce_f64):

    maximum[r] = max_b partial_max[r, b]
    scale[r,b] = exp(partial_max[r, b] - maximum[r])
    sum[r]     = sum_b scale[r,b] * partial_sum[r, b]
    out[r, c]  = (sum_b scale[r,b] * partial_out[r, b, c]) / sum[r]

which is the softmax-weighted output over every token of every block (pinned
in the tests against a direct softmax over the tokens).

Readings where the pages are silent (each also listed in the design notes):
  S1  Layouts: partial_max, partial_sum f32 [G, R, B]; partial_out f16
      [G, R, B, C] (C contiguous); out f32 [G, R, C].
  S2  The fp32 procedure is pinned (split_reduce_f32), in this order: the
      blocks are taken in chunks of CHUNK = 128 (the bounded stage), each
      chunk in runs of RUN = 32 consecutive blocks; inside a run, sum and
      output accumulate block by block from 0, each term rounded
      (fl(scale * x)) and then added (no fused multiply-add); a chunk's runs
      are added in order from 0, then the chunk partials in chunk order from
      0; out = fl(O / sum). Every operation is IEEE binary32
      round-to-nearest-even. (Runs let four thread groups share a chunk.)
  S3  The scale's exponential is one pinned fp32 routine (exp_f32): Cody and
      Waite's range reduction exp(x) = 2^n exp(x - n ln 2), with ln 2 split
      into a 16-bit high part and a low part so that n * LN2_HI is exact,
      and the degree-7 Taylor polynomial of exp on |t| <= ln2/2 in Horner
      form, each step one rounded multiply and one rounded add. Arguments
      below -86 (results below 2^-124) give 0. The routine is pinned against
      math.exp (at most 3 ulp).
  S4  B >= 1. A row whose sum is 0 cannot occur (every scale of the maximal
      block is 1 and partial sums are >= 1 in the workloads).

Parity: the CUDA kernel follows S2/S3 operation for operation, so it must
equal split_reduce_f32 bit for bit; split_reduce_f32 itself is checked against
split_reduce_f64 within error_bound (derived in its docstring).
"""
from __future__ import annotations

import math

import numpy as np

CHUNK = 128  # S2: blocks per chunk (the fixed-size scale stage)
RUN = 32     # S2: blocks per run inside a chunk

# S3: Cody-Waite split of ln 2 (high part with 16 significant bits) and the
# Taylor coefficients 1/k! for k = 7..0, all as float32.
LOG2E_F32 = np.float32(1.4426950408889634)
LN2_HI_F32 = np.float32(0.693145751953125)
LN2_LO_F32 = np.float32(math.log(2.0) - 0.693145751953125)
TAYLOR_F32 = [np.float32(1.0 / math.factorial(k)) for k in range(7, -1, -1)]
EXP_FLUSH_BELOW = np.float32(-86.0)


# ------------------------------------------------------------- exponential
def exp_f32(x) -> np.ndarray:
    """S3: the pinned fp32 exponential for x <= 0 (float32 in, float32 out)."""
    x = np.asarray(x, dtype=np.float32)
    xc = np.maximum(x, np.float32(-87.0))                   # flushed below; keeps the steps finite
    n = np.rint(xc * LOG2E_F32).astype(np.float32)         # round half to even
    t = (xc - n * LN2_HI_F32) - n * LN2_LO_F32              # n * LN2_HI is exact
    p = np.full_like(t, TAYLOR_F32[0])
    for c in TAYLOR_F32[1:]:
        p = p * t + c
    ni = np.clip(n, -126, 0).astype(np.int32)
    two_n = ((ni + 127).astype(np.uint32) << np.uint32(23)).view(np.float32)
    return np.where(x < EXP_FLUSH_BELOW, np.float32(0.0), p * two_n).astype(np.float32)


# ------------------------------------------------------------ the reduce
def split_reduce_f64(pm, ps, po) -> np.ndarray:
    """The definition in float64 (inputs converted exactly). Returns
    out [G, R, C] float64."""
    pm = np.asarray(pm, np.float64)
    ps = np.asarray(ps, np.float64)
    po = np.asarray(po, np.float64)
    maximum = pm.max(axis=2, keepdims=True)
    scale = np.exp(pm - maximum)
    s = (scale * ps).sum(axis=2)
    o = np.einsum("grb,grbc->grc", scale, po)
    return o / s[..., None]


def split_reduce_f32(pm, ps, po, chunk: int = CHUNK) -> np.ndarray:
    """S2: the pinned fp32 procedure. Returns out [G, R, C] float32."""
    pm = np.asarray(pm, np.float32)
    ps = np.asarray(ps, np.float32)
    po32 = np.asarray(po).astype(np.float32)   # fp16 -> fp32 is exact
    G, R, B = pm.shape
    C = po32.shape[3]
    maximum = pm.max(axis=2)                                 # exact
    scale = exp_f32(pm - maximum[..., None])                 # fl(pm - M), then exp_f32
    total_s = np.zeros((G, R), np.float32)
    total_o = np.zeros((G, R, C), np.float32)
    for b0 in range(0, B, chunk):
        part_s = np.zeros((G, R), np.float32)
        part_o = np.zeros((G, R, C), np.float32)
        for r0 in range(b0, min(B, b0 + chunk), RUN):
            run_s = np.zeros((G, R), np.float32)
            run_o = np.zeros((G, R, C), np.float32)
            for b in range(r0, min(B, r0 + RUN)):
                sc = scale[:, :, b]
                run_s = run_s + sc * ps[:, :, b]
                run_o = run_o + sc[..., None] * po32[:, :, b, :]
            part_s = part_s + run_s
            part_o = part_o + run_o
        total_s = total_s + part_s
        total_o = total_o + part_o
    return (total_o / total_s[..., None]).astype(np.float32)


def error_bound(pm, ps, po, chunk: int = CHUNK) -> np.ndarray:
    """Per-element bound on |split_reduce_f32 - split_reduce_f64|.

    With u = 2^-24 and delta = pm - maximum (exact), the fp32 argument
    fl(delta) has relative error <= u, which moves exp by a relative
    |delta| u; exp_f32 adds at most 3 ulp (<= 3 * 2^-23 relative). So each
    scale is S (1 + e), |e| <= eta = |delta| u + 3 * 2^-23 (to first order),
    or exactly 0 where delta < -86 (an absolute loss of S <= e^-86). Each
    term fl(scale * x) adds u. Every sum is a tree of at most
    h = RUN + chunk / RUN + ceil(B / chunk) additions along any path, so it adds at most
    gamma_h = h u / (1 - h u) of the sum of the terms' magnitudes. Hence
    |dO| <= A = sum_b S_b |po_b| (eta_b + u + gamma_h) + flushed terms, and
    |dSum| <= sum * eps_s with eps_s the same weight on the (positive) sum
    terms. The division adds u |out|. To first order
    |out32 - out64| <= A / sum + |out| eps_s + u |out|; the returned bound
    multiplies this by 1.01 to cover the second-order terms.
    """
    pm = np.asarray(pm, np.float64)
    ps = np.asarray(ps, np.float64)
    po = np.asarray(po, np.float64)
    u = 2.0 ** -24
    B = pm.shape[2]
    h = RUN + chunk // RUN + -(-B // chunk)
    gamma = h * u / (1.0 - h * u)
    maximum = pm.max(axis=2, keepdims=True)
    delta = pm - maximum
    S = np.exp(delta)
    flushed = delta < float(EXP_FLUSH_BELOW)
    eta = np.abs(delta) * u + 3.0 * 2.0 ** -23
    w = np.where(flushed, 1.0, eta + u + gamma)     # a flushed term is lost whole
    s = (S * ps).sum(axis=2)
    eps_s = (S * ps * w).sum(axis=2) / s
    A = np.einsum("grb,grbc->grc", S * w, np.abs(po))
    out = np.einsum("grb,grbc->grc", S, po) / s[..., None]
    return 1.01 * (A / s[..., None] + np.abs(out) * eps_s[..., None] + u * np.abs(out))


def bound_report(out32, out_ref, bound) -> dict:
    """Largest error relative to the bound (<= 1 passes)."""
    err = np.abs(np.asarray(out32, np.float64) - out_ref)
    util = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    return {"ok": bool(np.all(err <= bound)), "worst_util": float(util.max()) if util.size else 0.0,
            "max_abs_err": float(err.max()) if err.size else 0.0}


def n_chunks(B: int, chunk: int = CHUNK) -> int:
    """Number of block chunks (kernel CTAs per group)."""
    return -(-B // chunk)
