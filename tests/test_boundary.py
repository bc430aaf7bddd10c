"""CPU tests of the C ABI: the library builds and loads, exports every symbol
that include/qsa.h declares, and rejects bad arguments on the host (before
any CUDA call, so these run without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

import top_block_selection_gb300 as tbs
from top_block_selection_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")

OK, INVALID, GEOM, ARCH, MISALIGNED, CUDA, TIMEOUT = range(7)


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tbs.load_library()


def header_functions():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(qsa_\w+)\s*\(", txt, re.M)))


def test_header_declares_the_binding_symbols():
    assert header_functions() == sorted(tbs.EXPORTED_SYMBOLS)


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", tbs.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (qsa_\w+)$", out, re.M))
    assert set(header_functions()) <= exported


def test_library_has_no_cuda_driver_link_dependency(lib):
    # the runtime is linked statically and loads the driver lazily, so the
    # library loads on a machine without a GPU
    out = subprocess.run(["ldd", tbs.library_path()], capture_output=True, text=True).stdout
    assert "libcudart" not in out


def test_host_only_helpers(lib):
    assert tbs.qsa_abi_version() == 1
    assert tbs.qsa_num_blocks(4000, 64) == 63
    assert tbs.qsa_num_blocks(131072, 64) == 2048
    assert tbs.qsa_num_blocks(131073, 64) == 2049
    assert tbs.qsa_num_blocks(0, 64) == 0
    assert tbs.qsa_num_blocks(-1, 64) == -1 and tbs.qsa_num_blocks(5, 0) == -1
    for s in range(7):
        assert tbs.qsa_status_str(s) == tbs.STATUS_NAMES[s]
    assert "tcgen05" in tbs.qsa_arm()


def _scores(lib, q=16, kb=16, nq=4, H=8, D=128, n_kv=1000, block=64, out=16):
    return lib.qsa_block_scores(ctypes.c_void_p(q), ctypes.c_void_p(kb), nq, H, D, n_kv, block,
                                ctypes.c_void_p(out), None)


def test_block_scores_rejects_bad_arguments_on_host(lib):
    A = 1 << 20  # a fake, 16-byte aligned address; never dereferenced
    assert _scores(lib, A, A, nq=-1, out=A) == INVALID
    assert _scores(lib, A, A, block=0, out=A) == INVALID
    assert _scores(lib, A, A, n_kv=-5, out=A) == INVALID
    assert _scores(lib, A, A, H=3, out=A) == GEOM
    assert _scores(lib, A, A, H=64, out=A) == GEOM
    assert _scores(lib, A, A, D=72, out=A) == GEOM
    assert _scores(lib, A, A, D=272, out=A) == GEOM
    assert _scores(lib, A, A, D=0, out=A) == INVALID
    assert _scores(lib, 0, A, out=A) == INVALID
    assert _scores(lib, A, 0, out=A) == INVALID
    assert _scores(lib, A, A, out=0) == INVALID
    assert _scores(lib, A + 8, A, out=A) == MISALIGNED
    assert _scores(lib, A, A + 2, out=A) == MISALIGNED
    assert _scores(lib, A, A, out=A + 4) == MISALIGNED
    # empty work succeeds without touching the device (null pointers allowed)
    assert _scores(lib, 0, 0, nq=0, out=0) == OK
    assert _scores(lib, 0, 0, n_kv=0, out=0) == OK


def test_select_rejects_bad_arguments_on_host(lib):
    A = 1 << 20
    sel = lambda s, nq, nb, k, ids: lib.qsa_select(ctypes.c_void_p(s), nq, nb, k, ctypes.c_void_p(ids), None)
    assert sel(A, 4, 100, 0, A) == INVALID
    assert sel(A, -1, 100, 8, A) == INVALID
    assert sel(A, 4, -1, 8, A) == INVALID
    assert sel(A, 4, 100, 1025, A) == GEOM
    assert sel(A, 4, 32769, 8, A) == GEOM
    assert sel(0, 4, 100, 8, A) == INVALID
    assert sel(A, 4, 100, 8, 0) == INVALID
    assert sel(A + 2, 4, 100, 8, A) == MISALIGNED
    assert sel(A, 4, 100, 8, A + 1) == MISALIGNED
    assert sel(0, 0, 100, 8, 0) == OK


def test_convert_and_step_reject_bad_arguments_on_host(lib):
    A = 1 << 20
    assert lib.qsa_f32_to_f16(ctypes.c_void_p(A), ctypes.c_void_p(A), -1, None) == INVALID
    assert lib.qsa_f32_to_f16(ctypes.c_void_p(0), ctypes.c_void_p(A), 8, None) == INVALID
    assert lib.qsa_f32_to_f16(ctypes.c_void_p(A + 1), ctypes.c_void_p(A), 8, None) == MISALIGNED
    assert lib.qsa_f32_to_f16(ctypes.c_void_p(A), ctypes.c_void_p(A + 1), 8, None) == MISALIGNED
    assert lib.qsa_f32_to_f16(ctypes.c_void_p(0), ctypes.c_void_p(0), 0, None) == OK
    step = lambda q32, q16: lib.qsa_select_step(ctypes.c_void_p(q32), ctypes.c_void_p(q16), ctypes.c_void_p(A),
                                                4, 8, 128, 1000, 64, 8, ctypes.c_void_p(A), ctypes.c_void_p(A), None)
    assert step(0, A) == INVALID
    assert step(A, A + 2) == MISALIGNED
    assert step(A + 2, A) == MISALIGNED


def test_packed_host_step_rejects_bad_arguments_on_host(lib):
    A = 1 << 20
    v = ctypes.c_void_p
    pk = lambda nq, H, D, n_kv, k, in_h, out_h, in_d, out_d: lib.qsa_select_step_host_packed(
        v(in_h), nq, H, D, n_kv, 64, k, v(out_h), 0, v(in_d), None, v(out_d), None)
    assert pk(-1, 8, 128, 1000, 8, A, A, A, A) == INVALID
    assert pk(4, 0, 128, 1000, 8, A, A, A, A) == INVALID
    assert pk(4, 8, 120, 1000, 8, A, A, A, A) == GEOM          # D not a multiple of 16
    assert pk(4, 8, 128, 1000, 8, A, A, 0, A) == INVALID       # no device input buffer
    assert pk(4, 8, 128, 1000, 8, A, A, A + 2, A) == MISALIGNED
    assert pk(4, 8, 128, 1000, 8, 0, A, A, A) == INVALID       # no host input buffer
    assert pk(4, 8, 128, 1000, 8, A, 0, A, A) == INVALID       # no host output buffer
    assert pk(0, 8, 128, 1000, 8, 0, 0, A, A) == OK            # nothing to do


def test_batched_rejects_bad_arguments_on_host(lib):
    A = 1 << 20
    v = ctypes.c_void_p
    step = lambda stride, nb_: lib.qsa_select_step_batched(v(A), None, v(A), stride, nb_, 4, 8, 128,
                                                           1000, 64, 8, v(A), v(A), None)
    assert step(0, -1) == INVALID
    assert step(-8, 2) == INVALID
    assert step(8, 2) == INVALID            # stride below nb * D
    assert step(16 * 128 + 4, 2) == MISALIGNED
    assert step(0, 0) == OK                 # no batches: nothing to do
    ss = lambda stride, nb_: lib.qsa_score_select_batched(v(A), v(A), stride, nb_, 4, 8, 128, 1000,
                                                          64, 8, v(A), v(A), None)
    assert ss(0, -1) == INVALID and ss(0, 0) == OK


def test_step_launches_host_rules(lib):
    n = lambda nq, H, D, n_kv, block, k, q16: lib.qsa_select_step_launches(nq, H, D, n_kv, block, k, q16)
    assert n(4, 3, 128, 1000, 64, 8, 1) == -1        # unsupported head count
    assert n(4, 8, 120, 1000, 64, 8, 1) == -1        # D not a multiple of 16
    assert n(4, 8, 128, 1000, 64, 2000, 1) == -1     # k above the select limit
    assert n(4, 8, 128, 64 * 40000, 64, 8, 1) == -1  # nb above the select limit
    assert n(-1, 8, 128, 1000, 64, 8, 1) == -1
    assert n(0, 8, 128, 1000, 64, 8, 1) == 0         # nothing to compute
    assert n(4, 8, 128, 0, 64, 8, 1) == 0


def test_split_reduce_host_rules(lib):
    ws = lambda G, R, B, C: lib.qsa_split_reduce_workspace_bytes(G, R, B, C)
    assert ws(4, 8, 128, 128) == 0                 # one chunk: no workspace
    assert ws(0, 8, 2048, 128) == 0
    # counters (one per group and row, 16-byte padded), chunk sums, chunk outputs
    assert ws(4, 8, 2048, 128) == 128 + 4 * 16 * 8 * 4 + 4 * 16 * 8 * 128 * 4
    assert ws(3, 16, 129, 4) == 192 + 3 * 2 * 16 * 4 + 3 * 2 * 16 * 4 * 4
    assert ws(1, 33, 100, 128) == 0                # unsupported: 33 rows
    A = 1 << 20
    v = ctypes.c_void_p
    call = lambda G, R, B, C, pm=A, ps=A, po=A, out=A, w=A, wsz=1 << 30: lib.qsa_split_reduce(
        v(pm), v(ps), v(po), G, R, B, C, v(out), v(w), wsz, None)
    assert call(0, 8, 100, 128) == OK              # no groups: nothing to do
    assert call(-1, 8, 100, 128) == INVALID
    assert call(1, 0, 100, 128) == INVALID
    assert call(1, 8, 0, 128) == INVALID
    assert call(1, 33, 100, 128) == GEOM
    assert call(1, 8, 100, 126) == GEOM            # C not a multiple of 4
    assert call(1, 32, 100, 256) == GEOM           # R * C above 4096
    assert call(1, 8, 100, 128, pm=0) == INVALID
    assert call(1, 8, 200, 128, w=0) == INVALID    # two chunks need a workspace
    assert call(1, 8, 200, 128, wsz=64) == INVALID
    assert call(1, 8, 100, 128, po=A + 4) == MISALIGNED
    assert call(1, 8, 100, 128, out=A + 8) == MISALIGNED
    assert call(1, 8, 200, 128, w=A + 8) == MISALIGNED


def test_split_reduce_static_host_rules(lib):
    A = 1 << 20
    v = ctypes.c_void_p
    call = lambda G, R, B, C, pm=A, out=A: lib.qsa_split_reduce_static(v(pm), v(A), v(A), G, R, B, C,
                                                                      v(out), None)
    assert call(0, 8, 2048, 128) == OK                 # no groups
    assert call(64, 8, 4096, 128) == GEOM              # needs more than the fixed 4 MiB
    assert call(1, 33, 100, 128) == GEOM
    assert call(1, 8, 300, 128, pm=0) == INVALID
    assert call(1, 8, 300, 128, out=A + 8) == MISALIGNED


def test_selftest_rejects_bad_timeout_on_host(lib):
    assert lib.qsa_selftest_bounded_wait(0, None) == INVALID
    assert lib.qsa_selftest_bounded_wait(2_000_000_000, None) == INVALID


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(tbs, "_LIB", None)
    monkeypatch.setenv("QSA_LIBRARY", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        tbs.load_library()
