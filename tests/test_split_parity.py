"""GPU parity of the flash-attention decode split reduce (qsa_split_reduce)
against the CPU oracle: bit for bit with the pinned fp32 procedure, and
within the derived bound of the float64 definition."""
import numpy as np
import pytest

import qsa_inputs as qi
from oracle import split_reduce_oracle as sro

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


def check(tbs, pm, ps, po, name, workspace=None):
    out = tbs.qsa_split_reduce(dev(pm), dev(ps), dev(po), workspace=workspace)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want32 = sro.split_reduce_f32(pm, ps, po)
    assert np.array_equal(got.view(np.uint32), want32.view(np.uint32)), \
        (name, int((got != want32).sum()), float(np.abs(got - want32).max()))
    rep = sro.bound_report(got, sro.split_reduce_f64(pm, ps, po), sro.error_bound(pm, ps, po))
    assert rep["ok"], (name, rep)
    return got


@pytest.mark.parametrize("w", qi.SPLIT_WORKLOADS, ids=[w.name for w in qi.SPLIT_WORKLOADS])
def test_split_workloads(tbs, w):
    pm, ps, po = qi.make_split_partials(w)
    check(tbs, pm, ps, po, w.name)


@pytest.mark.parametrize("G,R,B,C", [(1, 1, 1, 4), (3, 8, 1, 128), (2, 3, 63, 8), (1, 8, 64, 128),
                                     (2, 8, 65, 128), (1, 32, 129, 128), (3, 16, 300, 256),
                                     (1, 5, 700, 12), (2, 8, 4097, 64), (1, 2, 5000, 4),
                                     (1, 4, 200, 1024), (2, 32, 129, 128)])
def test_split_shapes(tbs, G, R, B, C):
    pm, ps, po = qi.split_random_case(G, R, B, C, seed=G * 1000 + B)
    check(tbs, pm, ps, po, f"{G}x{R}x{B}x{C}")


def test_split_extreme_scales(tbs):
    """Maxima 100 apart: most scales flush to 0 or are tiny; one block dominates."""
    pm, ps, po = qi.split_random_case(2, 8, 200, 128, seed=9, pm_sd=40.0)
    check(tbs, pm, ps, po, "extreme")


def test_split_workspace_reused_across_calls(tbs):
    """One zero-filled workspace serves many calls (the arrival counters are
    left at zero), also for shapes of different sizes."""
    w = qi.SPLIT_BY_NAME["split_g4_r8_c128_b2048"]
    need = tbs.qsa_split_reduce_workspace_bytes(w.G, w.R, w.B, w.C)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for v in range(3):
        pm, ps, po = qi.make_split_partials(w, variant=v)
        check(tbs, pm, ps, po, f"reuse-{v}", workspace=ws)
    pm, ps, po = qi.split_random_case(2, 8, 300, 128, seed=4)
    check(tbs, pm, ps, po, "reuse-small", workspace=ws)
    head = ws[:16].cpu().numpy().view(np.uint32)
    assert np.all(head == 0)


def test_split_deterministic(tbs):
    w = qi.SPLIT_BY_NAME["split_g2_r16_c128_b4096"]
    pm, ps, po = (dev(a) for a in qi.make_split_partials(w))
    a = tbs.qsa_split_reduce(pm, ps, po)
    b = tbs.qsa_split_reduce(pm, ps, po)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_split_empty_groups(tbs):
    out = tbs.qsa_split_reduce(torch.zeros((0, 8, 10), device="cuda"),
                               torch.zeros((0, 8, 10), device="cuda"),
                               torch.zeros((0, 8, 10, 128), dtype=torch.float16, device="cuda"))
    assert out.shape == (0, 8, 128)
