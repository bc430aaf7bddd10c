"""Python binding of libqsa: QSA block scores and top-k block selection on
GB300 (sm_103a).

Argument marshalling only: every function checks dtypes, devices, shapes and
contiguity, allocates outputs with PyTorch when none are given, and calls the
C entry point of the same name (include/qsa.h) on the current CUDA stream.
All computation runs in the library's CUDA kernels; there is no other path.
If libqsa.so is missing or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "QsaError", "load_library", "library_path", "qsa_abi_version", "qsa_status_str",
    "qsa_last_cuda_error", "qsa_arm",
    "qsa_num_blocks", "qsa_f32_to_f16", "qsa_block_scores", "qsa_select", "qsa_score_select",
    "qsa_select_step", "qsa_select_step_host", "qsa_select_step_host_packed", "HostStep",
    "qsa_device_status", "qsa_selftest_bounded_wait",
    "qsa_select_step_batched", "qsa_score_select_batched", "qsa_select_step_launches",
    "qsa_split_reduce", "qsa_split_reduce_workspace_bytes", "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

# Every symbol declared in include/qsa.h.
EXPORTED_SYMBOLS = (
    "qsa_abi_version", "qsa_status_str", "qsa_last_cuda_error", "qsa_arm", "qsa_num_blocks",
    "qsa_f32_to_f16", "qsa_block_scores", "qsa_select", "qsa_score_select", "qsa_select_step",
    "qsa_select_step_host", "qsa_select_step_host_packed", "qsa_device_status",
    "qsa_selftest_bounded_wait", "qsa_select_step_batched", "qsa_score_select_batched", "qsa_select_step_launches",
    "qsa_split_reduce_workspace_bytes", "qsa_split_reduce", "qsa_split_reduce_static",
)

STATUS_NAMES = {0: "QSA_OK", 1: "QSA_ERR_INVALID_ARG", 2: "QSA_ERR_UNSUPPORTED_GEOMETRY",
                3: "QSA_ERR_UNSUPPORTED_ARCH", 4: "QSA_ERR_MISALIGNED", 5: "QSA_ERR_CUDA",
                6: "QSA_ERR_TIMEOUT"}


class QsaError(RuntimeError):
    """A libqsa entry point returned a status other than QSA_OK."""

    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


def library_path() -> str:
    return os.environ.get("QSA_LIBRARY", os.path.join(_HERE, "lib", "libqsa.so"))


def load_library():
    """Load libqsa.so once and declare the C signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libqsa.so not found at {path}: build it with "
                           "`python -m top_block_selection_gb300._build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, u32p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint32)
    sig = {
        "qsa_abi_version": (ctypes.c_int, []),
        "qsa_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "qsa_arm": (ctypes.c_char_p, []),
        "qsa_last_cuda_error": (ctypes.c_char_p, []),
        "qsa_num_blocks": (i64, [i64, i32]),
        "qsa_f32_to_f16": (ctypes.c_int, [vp, vp, i64, vp]),
        "qsa_block_scores": (ctypes.c_int, [vp, vp, i32, i32, i32, i64, i32, vp, vp]),
        "qsa_select": (ctypes.c_int, [vp, i32, i32, i32, vp, vp]),
        "qsa_score_select": (ctypes.c_int, [vp, vp, i32, i32, i32, i64, i32, i32, vp, vp, vp]),
        "qsa_select_step": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i64, i32, i32, vp, vp, vp]),
        "qsa_select_step_host": (ctypes.c_int, [vp, vp, i32, i32, i32, i64, i32, i32, vp, vp,
                                                vp, vp, vp, vp, vp, vp]),
        "qsa_select_step_host_packed": (ctypes.c_int, [vp, i32, i32, i32, i64, i32, i32, vp, i32,
                                                       vp, vp, vp, vp]),
        "qsa_device_status": (ctypes.c_int, [ctypes.c_int, u32p, vp]),
        "qsa_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint64, vp]),
        "qsa_select_step_batched": (ctypes.c_int, [vp, vp, vp, i64, i32, i32, i32, i32, i64, i32,
                                                   i32, vp, vp, vp]),
        "qsa_score_select_batched": (ctypes.c_int, [vp, vp, i64, i32, i32, i32, i32, i64, i32, i32,
                                                    vp, vp, vp]),
        "qsa_select_step_launches": (i32, [i32, i32, i32, i64, i32, i32, i32]),
        "qsa_split_reduce_workspace_bytes": (ctypes.c_size_t, [i32, i32, i32, i32]),
        "qsa_split_reduce": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, vp, vp, ctypes.c_size_t,
                                            vp]),
        "qsa_split_reduce_static": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


# ------------------------------------------------------------------ helpers
def _check(status: int, where: str):
    if status != 0:
        detail = _LIB.qsa_last_cuda_error().decode() if status == 5 and _LIB is not None else ""
        raise QsaError(status, where, detail)


def _torch():
    import torch
    return torch


def _stream_of(t):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t, dtype, ndim, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D CUDA {dtype} tensor, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t.numel() else 0)


# -------------------------------------------------------------- entry points
def qsa_abi_version() -> int:
    return load_library().qsa_abi_version()


def qsa_status_str(status: int) -> str:
    return load_library().qsa_status_str(status).decode()


def qsa_last_cuda_error() -> str:
    return load_library().qsa_last_cuda_error().decode()


def qsa_arm() -> str:
    return load_library().qsa_arm().decode()


def qsa_num_blocks(n_kv: int, block: int = 64) -> int:
    return int(load_library().qsa_num_blocks(n_kv, block))


def qsa_f32_to_f16(x, out=None):
    """fp32 -> fp16 (round to nearest even) of a CUDA float32 tensor."""
    torch = _torch()
    if not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    elif out.shape != x.shape or out.dtype != torch.float16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float16 tensor shaped like x")
    lib = load_library()
    with torch.cuda.device(x.device):
        _check(lib.qsa_f32_to_f16(_ptr(x), _ptr(out), x.numel(), _stream_of(x)), "qsa_f32_to_f16")
    return out


def _score_args(q, kb, n_kv, block):
    torch = _torch()
    _need(q, torch.float16, 3, "q")
    _need(kb, torch.float16, 2, "kb")
    nq, H, D = q.shape
    if kb.shape[1] != D:
        raise ValueError(f"kb has D={kb.shape[1]}, q has D={D}")
    nb = qsa_num_blocks(n_kv, block)
    if nb < 0:
        raise ValueError("n_kv must be >= 0 and block >= 1")
    if kb.shape[0] < nb:
        raise ValueError(f"kb must hold nb={nb} rows, has {kb.shape[0]}")
    if kb.device != q.device:
        raise ValueError("q and kb must be on the same device")
    return nq, H, D, nb


def qsa_block_scores(q, kb, n_kv: int, block: int = 64, out=None):
    """scores f32 [nq, nb]: full blocks on the tensor cores, the tail block
    (if any) by the fp32 tail kernel with the +1e9 bonus."""
    torch = _torch()
    nq, H, D, nb = _score_args(q, kb, n_kv, block)
    if out is None:
        out = torch.empty((nq, nb), dtype=torch.float32, device=q.device)
    else:
        _need(out, torch.float32, 2, "out")
        if tuple(out.shape) != (nq, nb):
            raise ValueError(f"out must be [{nq}, {nb}]")
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.qsa_block_scores(_ptr(q), _ptr(kb), nq, H, D, n_kv, block, _ptr(out),
                                    _stream_of(q)), "qsa_block_scores")
    return out


def qsa_select(scores, k: int, out=None):
    """ids int32 [nq, k]: top-k blocks per row, descending score, smaller index
    first on ties, -1 padding when nb < k."""
    torch = _torch()
    _need(scores, torch.float32, 2, "scores")
    nq, nb = scores.shape
    if out is None:
        out = torch.empty((nq, k), dtype=torch.int32, device=scores.device)
    else:
        _need(out, torch.int32, 2, "out")
        if tuple(out.shape) != (nq, k):
            raise ValueError(f"out must be [{nq}, {k}]")
    lib = load_library()
    with torch.cuda.device(scores.device):
        _check(lib.qsa_select(_ptr(scores), nq, nb, k, _ptr(out), _stream_of(scores)), "qsa_select")
    return out


def qsa_score_select(q, kb, n_kv: int, k: int, block: int = 64, scores=None, ids=None):
    """(scores [nq, nb] f32, ids [nq, k] int32) in one call."""
    torch = _torch()
    nq, H, D, nb = _score_args(q, kb, n_kv, block)
    if scores is None:
        scores = torch.empty((nq, nb), dtype=torch.float32, device=q.device)
    if ids is None:
        ids = torch.empty((nq, k), dtype=torch.int32, device=q.device)
    _need(scores, torch.float32, 2, "scores")
    _need(ids, torch.int32, 2, "ids")
    if tuple(scores.shape) != (nq, nb) or tuple(ids.shape) != (nq, k):
        raise ValueError("scores must be [nq, nb] and ids [nq, k]")
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.qsa_score_select(_ptr(q), _ptr(kb), nq, H, D, n_kv, block, k, _ptr(scores),
                                    _ptr(ids), _stream_of(q)), "qsa_score_select")
    return scores, ids


def qsa_select_step(q32, kb, n_kv: int, k: int, block: int = 64, q16=None, scores=None, ids=None):
    """One selection step from f32 queries in one fused launch: fp16
    conversion, scores, select. q16, if given, receives the converted
    queries; otherwise they stay on chip. Returns (q16 or None, scores, ids)."""
    torch = _torch()
    _need(q32, torch.float32, 3, "q32")
    _need(kb, torch.float16, 2, "kb")
    nq, H, D = q32.shape
    nb = qsa_num_blocks(n_kv, block)
    if nb < 0 or kb.shape[1] != D or kb.shape[0] < nb:
        raise ValueError("kb must be [>= nb, D] and n_kv >= 0, block >= 1")
    if scores is None:
        scores = torch.empty((nq, nb), dtype=torch.float32, device=q32.device)
    if ids is None:
        ids = torch.empty((nq, k), dtype=torch.int32, device=q32.device)
    if q16 is not None:
        _need(q16, torch.float16, 3, "q16")
        if tuple(q16.shape) != (nq, H, D):
            raise ValueError("q16 must be shaped like q32")
    _need(scores, torch.float32, 2, "scores")
    _need(ids, torch.int32, 2, "ids")
    if tuple(scores.shape) != (nq, nb) or tuple(ids.shape) != (nq, k):
        raise ValueError("scores must be [nq, nb] and ids [nq, k]")
    lib = load_library()
    with torch.cuda.device(q32.device):
        _check(lib.qsa_select_step(_ptr(q32), _ptr(q16) if q16 is not None else None, _ptr(kb), nq,
                                   H, D, n_kv, block, k, _ptr(scores), _ptr(ids), _stream_of(q32)),
               "qsa_select_step")
    return q16, scores, ids


def qsa_select_step_host(q32_host, kb_host, n_kv: int, k: int, block: int, scores_host, ids_host,
                         dev_buffers, stream=None):
    """qsa_select_step from host (CPU, ideally pinned) tensors. dev_buffers =
    (q32_dev, q16_dev or None, kb_dev, scores_dev, ids_dev) CUDA tensors. Enqueued on
    `stream` (default: current stream); synchronize before reading outputs.
    scores_host None leaves the scores in scores_dev. Buffers from
    host_step_buffers() are packed, so each direction is one copy."""
    torch = _torch()
    q32_dev, q16_dev, kb_dev, scores_dev, ids_dev = dev_buffers
    for t, name in ((q32_host, "q32_host"), (kb_host, "kb_host"), (scores_host, "scores_host"),
                    (ids_host, "ids_host")):
        if t is None and name == "scores_host":
            continue
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    nq, H, D = q32_host.shape
    if stream is None:
        stream = torch.cuda.current_stream(q32_dev.device)
    lib = load_library()
    with torch.cuda.device(q32_dev.device):
        _check(lib.qsa_select_step_host(
            _ptr(q32_host), _ptr(kb_host), nq, H, D, n_kv, block, k,
            _ptr(scores_host) if scores_host is not None else None,
            _ptr(ids_host), _ptr(q32_dev), _ptr(q16_dev) if q16_dev is not None else None,
            _ptr(kb_dev), _ptr(scores_dev),
            _ptr(ids_dev), ctypes.c_void_p(stream.cuda_stream)), "qsa_select_step_host")


def qsa_select_step_host_packed(in_host, nq: int, H: int, D: int, n_kv: int, k: int, block: int,
                                out_host, in_dev, out_dev, q16_dev=None, with_scores: bool = False,
                                stream=None):
    """The step from packed byte buffers (uint8 tensors): in_host / in_dev =
    q32 [nq,H,D] f32 then kb [nb,D] f16; out_dev = scores [nq,nb] f32 then
    ids [nq,k] int32; out_host = the same (with_scores) or ids only. One copy
    each way, enqueued on `stream` (default: current stream)."""
    torch = _torch()
    nb = qsa_num_blocks(n_kv, block)
    if nb < 0:
        raise ValueError("n_kv >= 0 and block >= 1 required")
    in_bytes = nq * H * D * 4 + nb * D * 2
    out_dev_bytes = nq * nb * 4 + nq * k * 4
    out_host_bytes = out_dev_bytes if with_scores else nq * k * 4
    for t, cuda, size, name in ((in_host, False, in_bytes, "in_host"), (in_dev, True, in_bytes, "in_dev"),
                                (out_dev, True, out_dev_bytes, "out_dev"),
                                (out_host, False, out_host_bytes, "out_host")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or t.is_cuda != cuda \
                or not t.is_contiguous() or t.numel() < size:
            raise ValueError(f"{name} must be a contiguous {'CUDA' if cuda else 'host'} uint8 tensor "
                             f"of at least {size} bytes")
    if q16_dev is not None:
        _need(q16_dev, torch.float16, 3, "q16_dev")
    if stream is None:
        stream = torch.cuda.current_stream(in_dev.device)
    lib = load_library()
    with torch.cuda.device(in_dev.device):
        _check(lib.qsa_select_step_host_packed(
            _ptr(in_host), nq, H, D, n_kv, block, k, _ptr(out_host), 1 if with_scores else 0,
            _ptr(in_dev), _ptr(q16_dev) if q16_dev is not None else None, _ptr(out_dev),
            ctypes.c_void_p(stream.cuda_stream)), "qsa_select_step_host_packed")


class HostStep:
    """A selection step fed from and read back to the host, bound to fixed
    sizes, its own packed device buffers and a stream (a serving loop's
    per-step state): one copy in (queries then keys), the step, one copy out
    (the ids, or scores then ids). Checks and pointer marshalling of the fixed
    parts are done once; a call marshals only the input buffer.

        step = HostStep(nq, H, D, n_kv, k, block)
        buf = step.new_input()            # pinned; fill step.q32_view(buf), step.kb_view(buf)
        step(buf)                         # enqueue; then synchronize the stream
        step.ids_host / step.scores_host  # results (scores_host: with_scores=True)
    """

    def __init__(self, nq: int, H: int, D: int, n_kv: int, k: int, block: int = 64, device=None,
                 with_scores: bool = False, with_q16: bool = False, stream=None):
        torch = _torch()
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        nb = qsa_num_blocks(n_kv, block)
        if nb < 0 or nq < 0 or H < 1 or D < 1 or k < 1:
            raise ValueError("bad step sizes")
        self.nq, self.H, self.D, self.nb, self.k = nq, H, D, nb, k
        self.n_kv, self.block, self.with_scores = n_kv, block, with_scores
        self._qb, self._kbb = nq * H * D * 4, nb * D * 2
        self._sb, self._ib = nq * nb * 4, nq * k * 4
        self.in_dev = torch.empty(self._qb + self._kbb, dtype=torch.uint8, device=self.device)
        self.out_dev = torch.empty(self._sb + self._ib, dtype=torch.uint8, device=self.device)
        self.q16_dev = (torch.empty((nq, H, D), dtype=torch.float16, device=self.device)
                        if with_q16 else None)
        self.out_host = torch.empty(self._sb + self._ib if with_scores else self._ib,
                                    dtype=torch.uint8).pin_memory()
        self.stream = torch.cuda.current_stream(self.device) if stream is None else stream
        self._fn = load_library().qsa_select_step_host_packed
        self._fixed_tail = (_ptr(self.out_host), 1 if with_scores else 0, _ptr(self.in_dev),
                            _ptr(self.q16_dev) if self.q16_dev is not None else None,
                            _ptr(self.out_dev), ctypes.c_void_p(self.stream.cuda_stream))
        self._dims = (nq, H, D, n_kv, block, k)

    def new_input(self):
        """A pinned input buffer for this step's sizes."""
        return _torch().empty(self._qb + self._kbb, dtype=_torch().uint8).pin_memory()

    def q32_view(self, buf):
        return buf[:self._qb].view(_torch().float32).view(self.nq, self.H, self.D)

    def kb_view(self, buf):
        return buf[self._qb:self._qb + self._kbb].view(_torch().float16).view(self.nb, self.D)

    @property
    def ids_host(self):
        off = self._sb if self.with_scores else 0
        return self.out_host[off:off + self._ib].view(_torch().int32).view(self.nq, self.k)

    @property
    def scores_host(self):
        if not self.with_scores:
            return None
        return self.out_host[:self._sb].view(_torch().float32).view(self.nq, self.nb)

    @property
    def scores_dev(self):
        return self.out_dev[:self._sb].view(_torch().float32).view(self.nq, self.nb)

    @property
    def ids_dev(self):
        return self.out_dev[self._sb:self._sb + self._ib].view(_torch().int32).view(self.nq, self.k)

    def __call__(self, in_host):
        torch = _torch()
        if in_host.dtype != torch.uint8 or in_host.is_cuda or in_host.numel() < self._qb + self._kbb \
                or not in_host.is_contiguous():
            raise ValueError("in_host must be a contiguous host uint8 buffer from new_input()")
        if torch.cuda.current_device() != self.device.index:
            with torch.cuda.device(self.device):
                return self(in_host)
        nq, H, D, n_kv, block, k = self._dims
        _check(self._fn(_ptr(in_host), nq, H, D, n_kv, block, k, *self._fixed_tail),
               "qsa_select_step_host_packed")


def qsa_device_status(clear: bool = True, device=None):
    """Synchronize the current stream and return (status, bits) of the device
    status word (nonzero bits = a kernel gave up a bounded wait)."""
    torch = _torch()
    lib = load_library()
    bits = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib.qsa_device_status(1 if clear else 0, ctypes.byref(bits),
                                   ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    return st, bits.value


def qsa_selftest_bounded_wait(timeout_ns: int = 1_000_000, device=None):
    """Run the bounded-wait self-test kernel on the current stream (it gives
    up after timeout_ns and records a timeout in the status word)."""
    torch = _torch()
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib.qsa_selftest_bounded_wait(timeout_ns,
                                             ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)),
               "qsa_selftest_bounded_wait")


def qsa_select_step_launches(nq: int, H: int, D: int, n_kv: int, k: int, block: int = 64,
                             with_q16: bool = True, device=None) -> int:
    """Kernel launches one qsa_select_step call of these sizes makes on the
    device (1 = the fused launch); raises for sizes the step rejects."""
    torch = _torch()
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        n = int(lib.qsa_select_step_launches(nq, H, D, n_kv, block, k, 1 if with_q16 else 0))
    if n < 0:
        raise QsaError(1, "qsa_select_step_launches")
    return n


def _batched_kb(kb, nb, D, n_batches):
    """(kb_batch_stride in elements) for a shared [>= nb, D] kb or a
    per-batch [n_batches, >= nb, D] kb."""
    torch = _torch()
    if kb.dtype != torch.float16 or not kb.is_cuda or not kb.is_contiguous():
        raise ValueError("kb must be a contiguous CUDA float16 tensor")
    if kb.dim() == 2:
        if kb.shape[1] != D or kb.shape[0] < nb:
            raise ValueError("shared kb must be [>= nb, D]")
        return 0
    if kb.dim() == 3:
        if kb.shape[0] != n_batches or kb.shape[2] != D or kb.shape[1] < nb:
            raise ValueError("per-batch kb must be [n_batches, >= nb, D]")
        return kb.shape[1] * D
    raise ValueError("kb must be 2-D (shared) or 3-D (per batch)")


def _batched_out(dev, n_batches, nq, nb, k, scores, ids):
    torch = _torch()
    if scores is None:
        scores = torch.empty((n_batches, nq, nb), dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty((n_batches, nq, k), dtype=torch.int32, device=dev)
    _need(scores, torch.float32, 3, "scores")
    _need(ids, torch.int32, 3, "ids")
    if tuple(scores.shape) != (n_batches, nq, nb) or tuple(ids.shape) != (n_batches, nq, k):
        raise ValueError("scores must be [n_batches, nq, nb] and ids [n_batches, nq, k]")
    return scores, ids


def qsa_select_step_batched(q32, kb, n_kv: int, k: int, block: int = 64, q16=None, scores=None,
                            ids=None):
    """The step for q32 [n_batches, nq, H, D]; kb shared ([nb, D]: one step
    over every batch's queries) or per batch ([n_batches, nb, D]: one launch).
    Returns (q16, scores, ids)."""
    torch = _torch()
    _need(q32, torch.float32, 4, "q32")
    B, nq, H, D = q32.shape
    nb = qsa_num_blocks(n_kv, block)
    if nb < 0:
        raise ValueError("n_kv must be >= 0 and block >= 1")
    stride = _batched_kb(kb, nb, D, B)
    scores, ids = _batched_out(q32.device, B, nq, nb, k, scores, ids)
    if q16 is not None:
        _need(q16, torch.float16, 4, "q16")
        if tuple(q16.shape) != tuple(q32.shape):
            raise ValueError("q16 must be shaped like q32")
    lib = load_library()
    with torch.cuda.device(q32.device):
        _check(lib.qsa_select_step_batched(_ptr(q32), _ptr(q16) if q16 is not None else None,
                                           _ptr(kb), stride, B, nq, H, D, n_kv, block, k,
                                           _ptr(scores), _ptr(ids), _stream_of(q32)),
               "qsa_select_step_batched")
    return q16, scores, ids


def qsa_score_select_batched(q, kb, n_kv: int, k: int, block: int = 64, scores=None, ids=None):
    """Scores and top-k for fp16 q [n_batches, nq, H, D] in one launch; kb
    shared or per batch as for qsa_select_step_batched."""
    torch = _torch()
    _need(q, torch.float16, 4, "q")
    B, nq, H, D = q.shape
    nb = qsa_num_blocks(n_kv, block)
    if nb < 0:
        raise ValueError("n_kv must be >= 0 and block >= 1")
    stride = _batched_kb(kb, nb, D, B)
    scores, ids = _batched_out(q.device, B, nq, nb, k, scores, ids)
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.qsa_score_select_batched(_ptr(q), _ptr(kb), stride, B, nq, H, D, n_kv, block, k,
                                            _ptr(scores), _ptr(ids), _stream_of(q)),
               "qsa_score_select_batched")
    return scores, ids


# ------------------------------------------------------- split reduce
def qsa_split_reduce_workspace_bytes(G: int, R: int, B: int, C: int) -> int:
    """Bytes of workspace qsa_split_reduce needs (0 when B <= 64)."""
    return int(load_library().qsa_split_reduce_workspace_bytes(G, R, B, C))


def qsa_split_reduce(partial_max, partial_sum, partial_out, out=None, workspace=None):
    """Flash-attention decode split reduce: partial_max / partial_sum f32
    [G, R, B], partial_out f16 [G, R, B, C] -> out f32 [G, R, C].

    workspace: a CUDA uint8 tensor of at least qsa_split_reduce_workspace_bytes
    bytes whose counter area is zero (torch.zeros once; every call leaves it
    zero). Allocated here when not given."""
    torch = _torch()
    _need(partial_max, torch.float32, 3, "partial_max")
    _need(partial_sum, torch.float32, 3, "partial_sum")
    _need(partial_out, torch.float16, 4, "partial_out")
    G, R, B = partial_max.shape
    C = partial_out.shape[3]
    if tuple(partial_sum.shape) != (G, R, B) or tuple(partial_out.shape[:3]) != (G, R, B):
        raise ValueError("partial_sum must be [G, R, B] and partial_out [G, R, B, C]")
    dev = partial_max.device
    if out is None:
        out = torch.empty((G, R, C), dtype=torch.float32, device=dev)
    _need(out, torch.float32, 3, "out")
    if tuple(out.shape) != (G, R, C):
        raise ValueError(f"out must be [{G}, {R}, {C}]")
    lib = load_library()
    with torch.cuda.device(dev):
        need = int(lib.qsa_split_reduce_workspace_bytes(G, R, B, C))
        if workspace is None:
            workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
        if workspace.dtype != torch.uint8 or not workspace.is_cuda or workspace.numel() < need:
            raise ValueError(f"workspace must be a CUDA uint8 tensor of at least {need} bytes")
        _check(lib.qsa_split_reduce(_ptr(partial_max), _ptr(partial_sum), _ptr(partial_out), G, R, B,
                                    C, _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream_of(partial_max)), "qsa_split_reduce")
    return out
