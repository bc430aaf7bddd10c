"""qsa_split_reduce_static, the split reduce that allocates nothing (its
scratch is a fixed device array inside the library), called through the C
ABI: two calls in a row, of different shapes, each bit-identical to
qsa_split_reduce with a caller workspace. Named to be collected last; it
also passes alone."""
import ctypes

import numpy as np
import pytest

import qsa_inputs as qi
from oracle import split_reduce_oracle as sro

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

UNSUPPORTED = 2
STATIC_BYTES = 4 << 20


@pytest.fixture(scope="module")
def tbs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from top_block_selection_gb300 import _build
    _build.build()
    import top_block_selection_gb300 as m
    m.load_library()
    return m


def static_call(lib, pm, ps, po, out):
    G, R, B = pm.shape
    C = po.shape[3]
    v = ctypes.c_void_p
    return lib.qsa_split_reduce_static(v(pm.data_ptr()), v(ps.data_ptr()), v(po.data_ptr()), G, R, B,
                                       C, v(out.data_ptr()),
                                       v(torch.cuda.current_stream().cuda_stream))


def test_static_entry_point_matches_the_workspace_one(tbs):
    lib = tbs.load_library()
    cases = [qi.make_split_partials(qi.SPLIT_BY_NAME["split_g4_r8_c128_b2048"]),
             qi.split_random_case(3, 16, 300, 64, seed=77),
             qi.make_split_partials(qi.SPLIT_BY_NAME["split_g2_r8_c128_b33"])]
    for pm, ps, po in cases:          # consecutive calls, shapes changing
        d = [torch.from_numpy(a).cuda() for a in (pm, ps, po)]
        G, R, B = pm.shape
        C = po.shape[3]
        assert tbs.qsa_split_reduce_workspace_bytes(G, R, B, C) <= STATIC_BYTES
        out_s = torch.empty((G, R, C), dtype=torch.float32, device="cuda")
        assert static_call(lib, *d, out_s) == 0
        out_w = tbs.qsa_split_reduce(*d)
        torch.cuda.synchronize()
        assert torch.equal(out_s.view(torch.int32), out_w.view(torch.int32))
        assert np.array_equal(out_s.cpu().numpy().view(np.uint32),
                              sro.split_reduce_f32(pm, ps, po).view(np.uint32))


def test_static_entry_point_rejects_shapes_beyond_its_array(tbs):
    lib = tbs.load_library()
    G, R, B, C = 64, 8, 4096, 128
    assert tbs.qsa_split_reduce_workspace_bytes(G, R, B, C) > STATIC_BYTES
    v = ctypes.c_void_p
    A = v(1 << 20)  # never dereferenced: the size check comes first
    assert lib.qsa_split_reduce_static(A, A, A, G, R, B, C, A, None) == UNSUPPORTED
