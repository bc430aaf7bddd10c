"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Scores of full blocks must lie within the pages' bound B of the float64
oracle; the tail column must equal the oracle's fp32 tail bit for bit; the
select must equal the oracle's top-k of the same GPU scores bit for bit, and
agree with the oracle's top-k of the exact scores except where the k-th /
(k+1)-th gap is below 2B; the fp16 conversion must be bitwise.
"""
import numpy as np
import pytest

import qsa_inputs as qi
from oracle import qsa_oracle as orc

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tbs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from top_block_selection_gb300 import _build
    _build.build()
    import top_block_selection_gb300 as m
    m.load_library()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


UTIL = {}


def check_case(tbs, q, kb, n_kv, block, k, name, exact=False):
    s_gpu, ids_gpu = tbs.qsa_score_select(dev(q), dev(kb), n_kv, k, block)
    torch.cuda.synchronize()
    s = s_gpu.cpu().numpy()
    ids = ids_gpu.cpu().numpy()
    s_ref, S, B, tail = orc.reference_scores(q, kb, n_kv, block)
    assert s.shape == s_ref.shape and s.dtype == np.float32
    if exact:
        assert np.array_equal(s.astype(np.float64), s_ref), name
    rep = orc.bound_report(s, s_ref, B)
    assert rep["ok"], (name, rep)
    UTIL[name] = rep["worst_util"]
    if tail is not None:
        assert s[:, -1].view(np.uint32).tolist() == tail.view(np.uint32).tolist(), name
    # exact select of the GPU's own scores
    assert np.array_equal(ids, orc.select_topk(s, k)), name
    sel = orc.selection_report(ids, s_ref, B, k)
    assert sel["ok"], (name, sel)
    return rep, sel


@pytest.mark.parametrize("w", qi.WORKLOADS, ids=[w.name for w in qi.WORKLOADS])
def test_workload_parity(tbs, w):
    q, kb = qi.make_inputs(w)
    rep, sel = check_case(tbs, q, kb, w.n_kv, w.block, w.k, w.name)
    print(f"{w.name}: worst bound utilisation {rep['worst_util']:.4f}, "
          f"guarded rows {sel['guarded_rows']}, exact rows {sel['exact_rows']}")


@pytest.mark.parametrize("w", qi.DECODE_WORKLOADS, ids=[w.name for w in qi.DECODE_WORKLOADS])
def test_decode_shapes(tbs, w):
    q, kb = qi.make_inputs(w)
    check_case(tbs, q, kb, w.n_kv, w.block, w.k, w.name)
    q32, _ = qi.make_f32_inputs(w)
    _, s_gpu, ids_gpu = tbs.qsa_select_step(dev(q32), dev(kb), w.n_kv, w.k, w.block)
    torch.cuda.synchronize()
    s = s_gpu.cpu().numpy()
    s_ref, S, B, _ = orc.reference_scores(orc.f32_to_f16(q32), kb, w.n_kv, w.block)
    assert orc.bound_report(s, s_ref, B)["ok"]
    assert np.array_equal(ids_gpu.cpu().numpy(), orc.select_topk(s, w.k))


@pytest.mark.parametrize("tied", [False, True])
@pytest.mark.parametrize("nb,k", [(2, 1), (32, 31), (33, 33), (64, 8), (64, 67)])
def test_short_rows_one_warp_select(tbs, nb, k, tied):
    """Rows of at most 64 blocks take the one-warp select in the fused step:
    ids exact against the oracle on the GPU's scores, including k >= nb (ids
    past nb are -1) and rows whose full blocks all tie (the block-index
    tie-break)."""
    q, kb = qi.random_case(40, 8, 128, nb, seed=nb * 13 + k, scale=0.3)
    if tied:
        kb[:] = kb[0]
    check_case(tbs, q, kb, nb * 64 - 5, 64, k, f"short-{nb}-{k}-{tied}")


@pytest.mark.parametrize("H", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("D", [16, 64, 80, 128, 256])
def test_coordinate_coded_exact(tbs, H, D):
    nq, nb, block = 19, 300, 16
    q, kb = qi.coordinate_coded_case(nq, H, D, nb)
    check_case(tbs, q, kb, nb * block - 5, block, 7, f"coord-H{H}-D{D}", exact=True)


def test_one_hot_exact(tbs):
    q, kb = qi.one_hot_case(40, 8, 128, 260, seed=11)
    check_case(tbs, q, kb, 260 * 64, 64, 16, "one-hot", exact=True)


@pytest.mark.parametrize("nq", [1, 17, 129])
@pytest.mark.parametrize("nb,tail", [(1, False), (1, True), (63, True), (129, False), (129, True)])
def test_ragged_tiles(tbs, nq, nb, tail):
    block = 64
    n_kv = nb * block - (13 if tail else 0)
    q, kb = qi.random_case(nq, 8, 128, nb, seed=nq * 1000 + nb, scale=0.3)
    check_case(tbs, q, kb, n_kv, block, 8, f"ragged-{nq}-{nb}-{tail}")


@pytest.mark.parametrize("H,D", [(1, 64), (2, 256), (4, 48), (16, 128), (32, 32), (8, 192), (4, 160)])
def test_other_geometries(tbs, H, D):
    nq, nb = 45, 700
    q, kb = qi.random_case(nq, H, D, nb, seed=H * 7 + D, scale=0.5)
    check_case(tbs, q, kb, nb * 64 - 1, 64, 24, f"geom-H{H}-D{D}")


def test_x8_headroom(tbs):
    q, kb = qi.random_case(64, 8, 128, 200, seed=5, scale=8.0 / np.sqrt(128) * 4)
    check_case(tbs, q, kb, 200 * 64, 64, 32, "x8-headroom")


def test_empty_and_degenerate(tbs):
    q, kb = qi.random_case(5, 8, 128, 10, seed=1)
    s, ids = tbs.qsa_score_select(dev(q), dev(kb), 0, 4, 64)
    torch.cuda.synchronize()
    assert tuple(s.shape) == (5, 0) and ids.cpu().numpy().tolist() == [[-1] * 4] * 5
    # n_kv < block: only the tail block
    check_case(tbs, q, kb, 10, 64, 4, "tail-only")
    # nq == 0
    s, ids = tbs.qsa_score_select(dev(q[:0]), dev(kb), 640, 4, 64)
    assert tuple(s.shape) == (0, 10) and tuple(ids.shape) == (0, 4)


def test_write_set_canaries(tbs):
    nq, H, D, nb, k, block = 33, 8, 128, 150, 10, 64
    q, kb = qi.random_case(nq, H, D, nb, seed=77)
    n_kv = nb * block - 3
    guard = 64
    sbuf = torch.full((guard + nq * nb + guard,), float("nan"), dtype=torch.float32, device="cuda")
    sbuf.view(torch.int32).fill_(0x7FC0DEAD)
    ibuf = torch.full((guard + nq * k + guard,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    s_view = sbuf[guard:guard + nq * nb].view(nq, nb)
    i_view = ibuf[guard:guard + nq * k].view(nq, k)
    tbs.qsa_score_select(dev(q), dev(kb), n_kv, k, block, scores=s_view, ids=i_view)
    torch.cuda.synchronize()
    sb = sbuf.view(torch.int32).cpu().numpy()
    ib = ibuf.cpu().numpy()
    assert np.all(sb[:guard] == 0x7FC0DEAD) and np.all(sb[-guard:] == 0x7FC0DEAD)
    assert np.all(ib[:guard] == 0x5A5A5A5A) and np.all(ib[-guard:] == 0x5A5A5A5A)
    assert not np.any(sb[guard:-guard] == 0x7FC0DEAD)       # every entry written
    assert not np.any(ib[guard:-guard] == 0x5A5A5A5A)


@pytest.mark.parametrize("nq,H,nb,tail,k", [(9, 8, 3077, True, 40), (20, 4, 8 * 128 * 3, False, 64),
                                            (3, 8, 32768, True, 64), (37, 16, 1100, True, 100),
                                            (5, 1, 2500, False, 33), (70, 2, 1500, True, 1024)])
def test_many_tiles_per_cta(tbs, nq, H, nb, tail, k):
    """More than two 128-block tiles per CTA (the Kb stages and the TMEM
    accumulators are reused), partial query groups, and long rows."""
    q, kb = qi.random_case(nq, H, 128, nb, seed=nq * 13 + nb, scale=0.25)
    check_case(tbs, q, kb, nb * 64 - (21 if tail else 0), 64, k, f"tiles-{nq}-{H}-{nb}")


def test_fused_matches_separate_kernels(tbs):
    """The fused launch and the separate score + select kernels agree bit for bit."""
    for w in qi.WORKLOADS[:4]:
        q, kb = qi.make_inputs(w)
        qd, kd = dev(q), dev(kb)
        s_f, i_f = tbs.qsa_score_select(qd, kd, w.n_kv, w.k, w.block)
        s_u = tbs.qsa_block_scores(qd, kd, w.n_kv, w.block)
        i_u = tbs.qsa_select(s_u, w.k)
        torch.cuda.synchronize()
        assert torch.equal(s_f.view(torch.int32), s_u.view(torch.int32)), w.name
        assert torch.equal(i_f, i_u), w.name


def test_large_step_paths_agree(tbs):
    """On the 4096-query prefill shape every path gives the same bits: the
    single-batch step (whatever plan it takes), the batched entry point (the
    8-CTA fused kernel), and the separate stages called one by one
    (conversion, score + tail, select)."""
    w = qi.BY_NAME["prefill_nq4096_h16_d128_kv131073"]
    q32, _ = qi.make_f32_inputs(w)
    _, kb = qi.make_inputs(w)
    kd = dev(kb)
    q16_buf = torch.empty(q32.shape, dtype=torch.float16, device="cuda")
    q16_s, s_s, i_s = tbs.qsa_select_step(dev(q32), kd, w.n_kv, w.k, w.block, q16=q16_buf)
    _, s_f, i_f = tbs.qsa_select_step(dev(q32), kd, w.n_kv, w.k, w.block)
    s_b, i_b = tbs.qsa_score_select_batched(q16_s[None], kd, w.n_kv, w.k, w.block)
    s_1, i_1 = tbs.qsa_score_select(q16_s, kd, w.n_kv, w.k, w.block)
    q16_c = tbs.qsa_f32_to_f16(dev(q32))
    s_c = tbs.qsa_block_scores(q16_c, kd, w.n_kv, w.block)
    i_c = tbs.qsa_select(s_c, w.k)
    torch.cuda.synchronize()
    for s, i in ((s_f, i_f), (s_b[0], i_b[0]), (s_1, i_1), (s_c, i_c)):
        assert torch.equal(s.view(torch.int32), s_s.view(torch.int32))
        assert torch.equal(i, i_s)
    assert np.array_equal(q16_s.cpu().numpy().view(np.uint16), orc.f32_to_f16(q32).view(np.uint16))


def test_arm_reports_the_plan_that_ran(tbs):
    """qsa_arm() names the kernels the last call on this thread launched: the
    8-CTA fused kernel for the 128K step and for a batched launch, and the
    chain of separate kernels for a step too large for the fused launch;
    qsa_select_step_launches agrees."""
    h = qi.BY_NAME["long128k_nq256_h8_d128_kv131072"]
    q32, _ = qi.make_f32_inputs(h)
    _, kb = qi.make_inputs(h)
    tbs.qsa_select_step(dev(q32), dev(kb), h.n_kv, h.k, h.block)
    arm = tbs.qsa_arm()
    assert "last call on this thread: 1 launch: fused_step_kernel" in arm, arm
    assert tbs.qsa_select_step_launches(h.nq, h.H, h.D, h.n_kv, h.k, h.block, with_q16=False) == 1
    tbs.qsa_select_step_batched(dev(q32[None]), dev(kb), h.n_kv, h.k, h.block)
    assert "1 launch: fused_step_kernel" in tbs.qsa_arm()
    # 4096 queries of 16 heads over 3000 blocks: more than 16 tiles of 128
    # blocks per query group and too many 8-CTA clusters -> the chain
    nq, H, nb = 4096, 16, 3000
    q, kb2 = qi.random_case_f32(nq, H, 128, nb, seed=77, scale=0.25)
    q16 = torch.empty(q.shape, dtype=torch.float16, device="cuda")
    tbs.qsa_select_step(dev(q), dev(kb2), nb * 64, 64, 64, q16=q16)
    torch.cuda.synchronize()
    arm = tbs.qsa_arm()
    assert ("3 launches: convert_vec8_kernel -> score_tc_persistent_kernel -> "
            "select_warp_kernel") in arm, arm
    assert tbs.qsa_select_step_launches(nq, H, 128, nb * 64, 64, 64, with_q16=True) == 3


@pytest.mark.parametrize("nq,H,n_kv", [(1000, 8, 2500 * 64 + 5), (600, 16, 1900 * 64)])
def test_large_scorer_ragged(tbs, nq, H, n_kv):
    """Shapes large enough for the persistent score kernel (many 128 x 256
    tiles), ragged in both directions: qsa_block_scores within the bound,
    the tail bitwise, and bit for bit with the fused kernel's scores."""
    q, kb = qi.random_case(nq, H, 128, -(-n_kv // 64), seed=nq + H, scale=0.25)
    qd, kd = dev(q), dev(kb)
    s_p = tbs.qsa_block_scores(qd, kd, n_kv, 64)
    s_f, _ = tbs.qsa_score_select_batched(qd[None], kd, n_kv, 8, 64)
    torch.cuda.synchronize()
    assert torch.equal(s_p.view(torch.int32), s_f[0].view(torch.int32))
    s = s_p.cpu().numpy()
    s_ref, S, B, tail = orc.reference_scores(q, kb, n_kv, 64)
    assert orc.bound_report(s, s_ref, B)["ok"]
    if tail is not None:
        assert s[:, -1].view(np.uint32).tolist() == tail.view(np.uint32).tolist()


@pytest.mark.parametrize("nq,H,n_kv,k", [(1300, 8, 700 * 64 + 5, 32), (1100, 32, 300 * 64 + 1, 64)])
def test_chain_with_tail_in_select(tbs, nq, H, n_kv, k):
    """Steps too large for one fused launch, with a tail block and at least
    1024 rows: the chain's one-warp-per-row select scores the tail itself
    (H lanes, one per head). Bit for bit with the fused kernel, the tail
    bitwise against the oracle, the ids the oracle's top-k of the same
    scores."""
    q, kb = qi.random_case(nq, H, 128, -(-n_kv // 64), seed=nq * 7 + H, scale=0.25)
    qd, kd = dev(q), dev(kb)
    s_c, i_c = tbs.qsa_score_select(qd, kd, n_kv, k, 64)
    torch.cuda.synchronize()
    arm = tbs.qsa_arm()
    assert "select_warp_kernel (tail block scored in)" in arm and "tail_kernel" not in arm, arm
    s_f, i_f = tbs.qsa_score_select_batched(qd[None], kd, n_kv, k, 64)
    torch.cuda.synchronize()
    assert torch.equal(s_c.view(torch.int32), s_f[0].view(torch.int32))
    assert torch.equal(i_c, i_f[0])
    s = s_c.cpu().numpy()
    s_ref, S, B, tail = orc.reference_scores(q, kb, n_kv, 64)
    assert orc.bound_report(s, s_ref, B)["ok"]
    assert s[:, -1].view(np.uint32).tolist() == tail.view(np.uint32).tolist()
    assert np.array_equal(i_c.cpu().numpy(), orc.select_topk(s, k))


def test_select_step_without_q16_output(tbs):
    w = qi.WORKLOADS[0]
    q32, _ = qi.make_f32_inputs(w)
    _, kb = qi.make_inputs(w)
    q16 = torch.empty(q32.shape, dtype=torch.float16, device="cuda")
    a = tbs.qsa_select_step(dev(q32), dev(kb), w.n_kv, w.k, w.block, q16=q16)
    b = tbs.qsa_select_step(dev(q32), dev(kb), w.n_kv, w.k, w.block)
    torch.cuda.synchronize()
    assert b[0] is None
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32)) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("shared_kb", [True, False])
@pytest.mark.parametrize("w", [qi.WORKLOADS[0], qi.WORKLOADS[2]], ids=["tiny", "mid"])
def test_batched_step_equals_single_steps(tbs, w, shared_kb):
    """n batches in one launch give exactly the single-batch results."""
    B = 3
    q32 = np.stack([qi.make_f32_inputs(w, variant=v)[0] for v in range(B)])
    kbs = np.stack([qi.make_inputs(w, variant=v)[1] for v in range(B)])
    kb_arg = dev(kbs[0]) if shared_kb else dev(kbs)
    q16b, sb, ib = tbs.qsa_select_step_batched(dev(q32), kb_arg, w.n_kv, w.k, w.block,
                                               q16=torch.empty(q32.shape, dtype=torch.float16,
                                                               device="cuda"))
    torch.cuda.synchronize()
    for b in range(B):
        kb_b = kbs[0] if shared_kb else kbs[b]
        q16s, ss, is_ = tbs.qsa_select_step(dev(q32[b]), dev(kb_b), w.n_kv, w.k, w.block,
                                            q16=torch.empty(q32.shape[1:], dtype=torch.float16,
                                                            device="cuda"))
        torch.cuda.synchronize()
        assert torch.equal(sb[b].view(torch.int32), ss.view(torch.int32)), b
        assert torch.equal(ib[b], is_), b
        assert torch.equal(q16b[b].view(torch.int16), q16s.view(torch.int16)), b
    # and batch 1 against the oracle
    kb_1 = kbs[0] if shared_kb else kbs[1]
    q16 = orc.f32_to_f16(q32[1])
    s_ref, S, B_, tail = orc.reference_scores(q16, kb_1, w.n_kv, w.block)
    s1 = sb[1].cpu().numpy()
    assert orc.bound_report(s1, s_ref, B_)["ok"]
    assert np.array_equal(ib[1].cpu().numpy(), orc.select_topk(s1, w.k))


def test_batched_per_batch_kb_chain(tbs):
    """Eight batches of the 128K workload, each with its own kb, and a q16
    buffer: past a few waves of the fused kernel they run as the chain
    (conversion, persistent scores over every batch's tiles, one select over
    every batch's rows). Bit for bit with single-batch steps."""
    w = qi.BY_NAME["long128k_nq256_h8_d128_kv131072"]
    B = 8
    q32 = np.stack([qi.make_f32_inputs(w, variant=v)[0] for v in range(B)])
    kbs = np.stack([qi.make_inputs(w, variant=v)[1] for v in range(B)])
    q16b, sb, ib = tbs.qsa_select_step_batched(dev(q32), dev(kbs), w.n_kv, w.k, w.block,
                                               q16=torch.empty(q32.shape, dtype=torch.float16,
                                                               device="cuda"))
    torch.cuda.synchronize()
    arm = tbs.qsa_arm()
    assert "score_tc_persistent_kernel" in arm and "select_warp_kernel" in arm, arm
    for b in (0, 5, 7):
        q16s, ss, is_ = tbs.qsa_select_step(dev(q32[b]), dev(kbs[b]), w.n_kv, w.k, w.block,
                                            q16=torch.empty(q32.shape[1:], dtype=torch.float16,
                                                            device="cuda"))
        torch.cuda.synchronize()
        assert torch.equal(sb[b].view(torch.int32), ss.view(torch.int32)), b
        assert torch.equal(ib[b], is_), b
        assert torch.equal(q16b[b].view(torch.int16), q16s.view(torch.int16)), b


@pytest.mark.parametrize("nq,H,n_kv,B", [(256, 16, 700 * 64 + 9, 8), (512, 8, 1000 * 64 + 1, 5),
                                        (300, 8, 1500 * 64 + 3, 8)])
def test_batched_per_batch_kb_chain_with_tail(tbs, nq, H, n_kv, B):
    """The per-batch-kb chain with a tail block: each batch's tail is scored
    by the select with that batch's key row. Bit for bit with the fused
    kernel on each batch; tails bitwise against the oracle."""
    nb = -(-n_kv // 64)
    qs, kbs = zip(*[qi.random_case(nq, H, 128, nb, seed=31 * b + nq, scale=0.25) for b in range(B)])
    q, kb = np.stack(qs), np.stack(kbs)
    s_c, i_c = tbs.qsa_score_select_batched(dev(q), dev(kb), n_kv, 64, 64)
    torch.cuda.synchronize()
    arm = tbs.qsa_arm()
    assert "select_warp_kernel (tail block scored in)" in arm, arm
    for b in range(B):
        s_f, i_f = tbs.qsa_score_select_batched(dev(q[b])[None], dev(kb[b]), n_kv, 64, 64)
        torch.cuda.synchronize()
        assert torch.equal(s_c[b].view(torch.int32), s_f[0].view(torch.int32)), b
        assert torch.equal(i_c[b], i_f[0]), b
    s_ref, S, B_, tail = orc.reference_scores(q[B - 1], kb[B - 1], n_kv, 64)
    s = s_c[B - 1].cpu().numpy()
    assert s[:, -1].view(np.uint32).tolist() == tail.view(np.uint32).tolist()
    assert orc.bound_report(s, s_ref, B_)["ok"]


@pytest.mark.parametrize("nq,nb,n_batches", [(256, 2048, 3), (64, 3000, 6)])
def test_batched_lean_form(tbs, nq, nb, n_batches):
    """Launches of several waves take the lean form (one Kb stage, capped
    registers); its bits equal the single-batch launches' (the regular form),
    with two tiles per CTA and with three (the stage refilled between tiles)."""
    H, D, k = 8, 128, 64
    n_kv = nb * 64 - 5
    cases = [qi.random_case_f32(nq, H, D, nb, seed=7000 + 31 * b + nb, scale=0.25) for b in range(n_batches)]
    q32 = np.stack([c[0] for c in cases])
    kbs = np.stack([c[1] for c in cases])
    _, sb, ib = tbs.qsa_select_step_batched(dev(q32), dev(kbs), n_kv, k, 64)
    torch.cuda.synchronize()
    for b in range(n_batches):
        _, ss, is_ = tbs.qsa_select_step(dev(q32[b]), dev(kbs[b]), n_kv, k, 64)
        torch.cuda.synchronize()
        assert torch.equal(sb[b].view(torch.int32), ss.view(torch.int32)), b
        assert torch.equal(ib[b], is_), b
    q16 = orc.f32_to_f16(q32[-1])
    s_ref, S, B_, tail = orc.reference_scores(q16, kbs[-1], n_kv, 64)
    s_last = sb[-1].cpu().numpy()
    assert orc.bound_report(s_last, s_ref, B_)["ok"]
    assert s_last[:, -1].view(np.uint32).tolist() == tail.view(np.uint32).tolist()
    assert np.array_equal(ib[-1].cpu().numpy(), orc.select_topk(s_last, k))


def test_batched_score_select_fp16(tbs):
    w = qi.WORKLOADS[1]
    B = 4
    qs = np.stack([qi.make_inputs(w, variant=v)[0] for v in range(B)])
    kb = qi.make_inputs(w)[1]
    sb, ib = tbs.qsa_score_select_batched(dev(qs), dev(kb), w.n_kv, w.k, w.block)
    torch.cuda.synchronize()
    for b in range(B):
        ss, is_ = tbs.qsa_score_select(dev(qs[b]), dev(kb), w.n_kv, w.k, w.block)
        torch.cuda.synchronize()
        assert torch.equal(sb[b].view(torch.int32), ss.view(torch.int32)), b
        assert torch.equal(ib[b], is_), b
    s_ref, S, B_, _ = orc.reference_scores(qs[2], kb, w.n_kv, w.block)
    assert orc.bound_report(sb[2].cpu().numpy(), s_ref, B_)["ok"]


def test_determinism_double_launch(tbs):
    w = qi.WORKLOADS[3]
    q, kb = qi.make_inputs(w)
    qd, kd = dev(q), dev(kb)
    s1, i1 = tbs.qsa_score_select(qd, kd, w.n_kv, w.k, w.block)
    s2, i2 = tbs.qsa_score_select(qd, kd, w.n_kv, w.k, w.block)
    torch.cuda.synchronize()
    assert torch.equal(s1.view(torch.int32), s2.view(torch.int32))
    assert torch.equal(i1, i2)


@pytest.mark.parametrize("kind", ["normal", "ties", "signed0", "const"])
@pytest.mark.parametrize("nb,k", [(1, 1), (5, 8), (33, 8), (64, 63), (64, 70), (65, 8), (100, 64),
                                  (1000, 100), (2049, 64), (4096, 1024), (32768, 64), (300, 300)])
def test_select_exact(tbs, kind, nb, k):
    nq = 3 if nb >= 4096 else 23
    s = qi.random_scores(nq, nb, seed=nb * 31 + k, kind=kind)
    ids = tbs.qsa_select(dev(s), k)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), orc.select_topk(s, k))


@pytest.mark.parametrize("kind", ["normal", "ties", "signed0", "const"])
@pytest.mark.parametrize("nb,k", [(1, 1), (5, 8), (100, 64), (129, 128), (2049, 64), (4096, 128)])
def test_select_exact_many_rows(tbs, kind, nb, k):
    """Launches of many rows take the one-warp-per-row select: exact against
    the oracle on score rows, ties, signed zeros and constant rows (the last
    two take its bisection path)."""
    nq = 1100
    s = qi.random_scores(nq, nb, seed=nb * 17 + k, kind=kind)
    ids = tbs.qsa_select(dev(s), k)
    torch.cuda.synchronize()
    assert "select_warp_kernel" in tbs.qsa_arm()
    assert np.array_equal(ids.cpu().numpy(), orc.select_topk(s, k))


def _threshold_rows(k, extras, nb=1024, threads=256):
    """Score rows that steer the CTA-per-row threshold select to a chosen
    number of candidates. Thread t of the 256-thread select holds the keys of
    indices t + 256 j; warp w = t // 32 takes the ceil(k/8)-th largest of its
    threads' maxima. Each warp gets exactly ceil(k/8) threads with a high
    maximum (>= 100, except one of warp 0's at 10.0), so the bound is 10.0 and
    the keys >= it are those 8 ceil(k/8) maxima plus `extras` further keys in
    (10, 99) placed in the high threads' other slots; every other key is below
    1. All values are distinct. The oracle decides the expected ids, so a row
    stays a valid exactness case whatever path the kernel takes."""
    q = -(-k // 8)
    rng = np.random.default_rng(1000 * k + extras)
    row = (rng.permutation(nb).astype(np.float64) * 1e-4).astype(np.float32)
    slots = []
    for w in range(threads // 32):
        for i in range(q):
            t = 32 * w + i
            row[t] = 10.0 if (w == 0 and i == q - 1) else np.float32(100.0 + 0.01 * t)
            if not (w == 0 and i == q - 1):
                slots += [t + threads * j for j in range(1, nb // threads)]
    assert extras <= len(slots)
    for e, idx in enumerate(rng.permutation(slots)[:extras]):
        row[idx] = np.float32(11.0 + 0.01 * e)
    return row


@pytest.mark.parametrize("k,extras", [(64, 0), (64, 1), (64, 3), (64, 189), (128, 1), (128, 127),
                                      (128, 128), (128, 129)])
def test_select_threshold_candidate_counts(tbs, k, extras):
    """The threshold select around its limits: an odd number of candidates
    (the ranking reads one padding entry past them), exactly 255 and 256
    candidates (the most it ranks) and 257 (more: the window select takes the
    row)."""
    rows = np.stack([_threshold_rows(k, extras), _threshold_rows(k, extras)[::-1].copy()])
    ids = tbs.qsa_select(dev(rows), k)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), orc.select_topk(rows, k))


def test_select_empty_rows(tbs):
    ids = tbs.qsa_select(torch.zeros((4, 0), dtype=torch.float32, device="cuda"), 3)
    torch.cuda.synchronize()
    assert ids.cpu().numpy().tolist() == [[-1] * 3] * 4


def test_convert_bitwise(tbs):
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e6, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, np.inf, -np.inf]),
        rng.normal(size=100003) * np.exp2(rng.integers(-30, 17, size=100003))]).astype(np.float32)
    out = tbs.qsa_f32_to_f16(dev(vals)).cpu().numpy()
    assert np.array_equal(out.view(np.uint16), orc.f32_to_f16(vals).view(np.uint16))
    # an unaligned view takes the scalar path
    x = dev(vals)[1:]
    out2 = tbs.qsa_f32_to_f16(x.contiguous())
    assert np.array_equal(out2.cpu().numpy().view(np.uint16), orc.f32_to_f16(vals[1:]).view(np.uint16))
    nan = tbs.qsa_f32_to_f16(dev(np.array([np.nan] * 9, np.float32))).cpu().numpy()
    assert np.all(np.isnan(nan))


@pytest.mark.parametrize("w", qi.WORKLOADS[:4], ids=[w.name for w in qi.WORKLOADS[:4]])
def test_select_step_from_f32(tbs, w):
    """Start from f32 queries and keys: the conversion runs on the GPU and the
    scores are compared with the float64 oracle on the f32 ORIGINALS, which
    exercises the 2^-9.5 * S operand-rounding term of the bound."""
    q32, kb32 = qi.make_f32_inputs(w)
    kb16_gpu = tbs.qsa_f32_to_f16(dev(kb32))
    q16_buf = torch.empty(q32.shape, dtype=torch.float16, device="cuda")
    q16_gpu, s_gpu, ids_gpu = tbs.qsa_select_step(dev(q32), kb16_gpu, w.n_kv, w.k, w.block,
                                                  q16=q16_buf)
    torch.cuda.synchronize()
    kb16 = orc.f32_to_f16(kb32)
    assert np.array_equal(kb16_gpu.cpu().numpy().view(np.uint16), kb16.view(np.uint16))
    q16 = q16_gpu.cpu().numpy()
    assert np.array_equal(q16.view(np.uint16), orc.f32_to_f16(q32).view(np.uint16))
    s = s_gpu.cpu().numpy()
    s_ref32 = orc.scores_f64(q32.astype(np.float64), kb32.astype(np.float64), w.n_kv, w.block)
    S32 = orc.abs_product_sum_f64(q32.astype(np.float64), kb32.astype(np.float64), w.n_kv, w.block)
    B32 = orc.error_bound(S32, s_ref32)
    full = slice(0, w.n_full)
    rep = orc.bound_report(s[:, full], s_ref32[:, full], B32[:, full])
    assert rep["ok"], rep
    UTIL[w.name + "-f32"] = rep["worst_util"]
    tail = orc.tail_scores_f32(q16, kb16, w.n_kv, w.block)
    if tail is not None:
        assert s[:, -1].view(np.uint32).tolist() == tail.view(np.uint32).tolist()
    assert np.array_equal(ids_gpu.cpu().numpy(), orc.select_topk(s, w.k))


@pytest.mark.parametrize("nq,H,D,nb,tail", [(1, 8, 128, 129, True), (9, 8, 128, 129, False),
                                          (17, 8, 128, 63, True), (129, 8, 128, 300, True),
                                          (45, 1, 64, 700, True), (45, 2, 256, 700, True),
                                          (45, 4, 48, 700, True), (45, 16, 128, 700, False),
                                          (45, 32, 32, 700, True), (45, 8, 192, 700, True),
                                          (45, 4, 160, 700, True)])
def test_f32_step_ragged_and_geometries(tbs, nq, H, D, nb, tail):
    """fp32 queries through the step (in the fused kernel the eight CTAs of a
    cluster each round a slice of the query tile and deliver it to all eight):
    the rounded queries, the scores and the ids are bit-identical to the fp16
    path on the same rounded queries, and the scores lie within the bound."""
    block = 64
    n_kv = nb * block - (13 if tail else 0)
    k = 24
    q32, kb = qi.random_case_f32(nq, H, D, nb, seed=nq * 131 + H * 7 + D, scale=0.5)
    q16_buf = torch.empty(q32.shape, dtype=torch.float16, device="cuda")
    q16_gpu, s_gpu, ids_gpu = tbs.qsa_select_step(dev(q32), dev(kb), n_kv, k, block, q16=q16_buf)
    _, s_nq, ids_nq = tbs.qsa_select_step(dev(q32), dev(kb), n_kv, k, block)
    q16 = orc.f32_to_f16(q32)
    s_h, ids_h = tbs.qsa_score_select(dev(q16), dev(kb), n_kv, k, block)
    torch.cuda.synchronize()
    assert np.array_equal(q16_gpu.cpu().numpy().view(np.uint16), q16.view(np.uint16))
    for s_x, i_x in ((s_gpu, ids_gpu), (s_nq, ids_nq)):
        assert torch.equal(s_x.view(torch.int32), s_h.view(torch.int32))
        assert torch.equal(i_x, ids_h)
    s = s_gpu.cpu().numpy()
    s_ref, S, B, tail_ref = orc.reference_scores(q16, kb, n_kv, block)
    rep = orc.bound_report(s, s_ref, B)
    assert rep["ok"], rep
    if tail_ref is not None:
        assert s[:, -1].view(np.uint32).tolist() == tail_ref.view(np.uint32).tolist()
    assert np.array_equal(ids_gpu.cpu().numpy(), orc.select_topk(s, k))


def test_select_step_host_matches_device(tbs):
    w = qi.WORKLOADS[2]
    q32, kb16 = qi.make_f32_inputs(w)[0], qi.make_inputs(w)[1]
    q32h = torch.from_numpy(q32).pin_memory()
    kbh = torch.from_numpy(kb16).pin_memory()
    sh = torch.empty((w.nq, w.nb), dtype=torch.float32).pin_memory()
    ih = torch.empty((w.nq, w.k), dtype=torch.int32).pin_memory()
    bufs = (torch.empty_like(q32h, device="cuda"), torch.empty(q32.shape, dtype=torch.float16, device="cuda"),
            torch.empty_like(kbh, device="cuda"), torch.empty_like(sh, device="cuda"),
            torch.empty_like(ih, device="cuda"))
    tbs.qsa_select_step_host(q32h, kbh, w.n_kv, w.k, w.block, sh, ih, bufs)
    torch.cuda.synchronize()
    _, s_d, i_d = tbs.qsa_select_step(dev(q32), dev(kb16), w.n_kv, w.k, w.block)
    torch.cuda.synchronize()
    assert np.array_equal(sh.numpy().view(np.uint32), s_d.cpu().numpy().view(np.uint32))
    assert np.array_equal(ih.numpy(), i_d.cpu().numpy())
    assert np.array_equal(bufs[1].cpu().numpy().view(np.uint16), orc.f32_to_f16(q32).view(np.uint16))


def test_select_step_host_packed_buffers(tbs):
    """The packed host step (one copy each way) gives the same bits as the
    device step, with the scores copied back or left on the device, and the
    separate-buffer host step may leave the scores on the device too."""
    w = qi.WORKLOADS[2]
    q32, kb16 = qi.make_f32_inputs(w)[0], qi.make_inputs(w)[1]
    _, s_d, i_d = tbs.qsa_select_step(dev(q32), dev(kb16), w.n_kv, w.k, w.block)
    torch.cuda.synchronize()
    for with_scores in (True, False):
        step = tbs.HostStep(w.nq, w.H, w.D, w.n_kv, w.k, w.block, with_scores=with_scores,
                            with_q16=True)
        buf = step.new_input()
        step.q32_view(buf).copy_(torch.from_numpy(q32))
        step.kb_view(buf).copy_(torch.from_numpy(kb16))
        step.ids_host.fill_(-7)
        step(buf)
        torch.cuda.synchronize()
        assert np.array_equal(step.ids_host.numpy(), i_d.cpu().numpy())
        assert torch.equal(step.scores_dev.view(torch.int32), s_d.view(torch.int32))
        assert torch.equal(step.ids_dev, i_d)
        assert np.array_equal(step.q16_dev.cpu().numpy().view(np.uint16),
                              orc.f32_to_f16(q32).view(np.uint16))
        if with_scores:
            assert np.array_equal(step.scores_host.numpy().view(np.uint32),
                                  s_d.cpu().numpy().view(np.uint32))
        else:
            assert step.scores_host is None
    # qsa_select_step_host with scores_host None: ids back, scores on the device
    ih = torch.full((w.nq, w.k), -7, dtype=torch.int32).pin_memory()
    bufs = (torch.empty(q32.shape, dtype=torch.float32, device="cuda"), None,
            torch.empty(kb16.shape, dtype=torch.float16, device="cuda"),
            torch.zeros((w.nq, w.nb), dtype=torch.float32, device="cuda"),
            torch.empty((w.nq, w.k), dtype=torch.int32, device="cuda"))
    tbs.qsa_select_step_host(torch.from_numpy(q32).pin_memory(), torch.from_numpy(kb16).pin_memory(),
                             w.n_kv, w.k, w.block, None, ih, bufs)
    torch.cuda.synchronize()
    assert np.array_equal(ih.numpy(), i_d.cpu().numpy())
    assert torch.equal(bufs[3].view(torch.int32), s_d.view(torch.int32))


def test_negative_control_on_gpu_scores(tbs):
    w = qi.WORKLOADS[0]
    q, kb = qi.make_inputs(w)
    s = tbs.qsa_block_scores(dev(q), dev(kb), w.n_kv, w.block).cpu().numpy()
    s_ref, S, B, _ = orc.reference_scores(q, kb, w.n_kv, w.block)
    assert orc.bound_report(s, s_ref, B)["ok"]
    bad = s.astype(np.float64) + 2.5 * B
    assert not orc.bound_report(bad, s_ref, B)["ok"]


def test_bounded_wait_timeout_is_reported(tbs):
    """A wait that nothing completes gives up after its bound, sets the
    status word, and leaves the context usable."""
    st, bits = tbs.qsa_device_status(clear=True)
    assert st == 0 and bits == 0
    tbs.qsa_selftest_bounded_wait(2_000_000)          # 2 ms
    st, bits = tbs.qsa_device_status(clear=False)
    assert st == 6 and bits == (1 << 31)               # QSA_ERR_TIMEOUT, self-test bit
    st, bits = tbs.qsa_device_status(clear=True)      # read and clear
    assert st == 6
    st, bits = tbs.qsa_device_status(clear=True)
    assert st == 0 and bits == 0
    # the context still works
    w = qi.WORKLOADS[0]
    q, kb = qi.make_inputs(w)
    check_case(tbs, q, kb, w.n_kv, w.block, w.k, "after-timeout")


def test_device_status_clear(tbs):
    st, bits = tbs.qsa_device_status(clear=True)
    assert st == 0 and bits == 0


def test_report_bound_utilisation():
    if UTIL:
        worst = max(UTIL.values())
        print("worst bound utilisation over GPU cases: %.4f (%s)" % (worst, max(UTIL, key=UTIL.get)))
        assert worst <= 1.0
