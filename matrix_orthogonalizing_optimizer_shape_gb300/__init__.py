"""Dion3 optimizer step on one GB300 (sm_103a): Python binding of the C ABI.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libdion3.so`` (declared in ``include/dion3.h``).  PyTorch tensors provide
device memory and the current stream; nothing here computes on them.  There is
no CPU fallback: if the library is missing, :func:`load_library` raises.

Typical use::

    import matrix_orthogonalizing_optimizer_shape_gb300 as d3
    hp = d3.HParams(f=0.25, mu=0.95, lr=0.02)
    groups = [d3.Group(params=[W...], grads=[G...], momentum=[M...])]
    ws = d3.alloc_workspace(d3.workspace_size(groups, hp))
    d3.step(groups, hp, ws)
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional, Sequence

from ._build import LIB_PATH, build  # noqa: F401

ABI_VERSION = 1

F32, BF16, F16 = 0, 1, 2

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_CHECK = range(7)

#: Muon's quintic Newton-Schulz coefficients.
MUON_QUINTIC = (3.4445, -4.7750, 2.0315)

#: Every exported symbol of include/dion3.h.
EXPORTED = (
    "dion3_abi_version", "dion3_status_string", "dion3_last_error", "dion3_num_selected",
    "dion3_useful_flops", "dion3_select_workspace_size", "dion3_select_rows",
    "dion3_gram_ns_workspace_size", "dion3_gram_ns_batched", "dion3_workspace_size",
    "dion3_step", "dion3_device_status", "dion3_gemm_f16", "dion3_trace_enable",
    "dion3_trace_collect", "dion3_select_rows_noalloc", "dion3_ns_useful_flops",
    "dion3_ns_workspace_size", "dion3_ns_batched", "dion3_step_lazy", "dion3_flush_row_scale",
    "dion3_step_normuon", "dion3_wait_probe", "dion3_set_overlap",
)


class Dion3Error(RuntimeError):
    """A C-ABI call returned a status other than DION3_OK."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class _HParams(ctypes.Structure):
    _fields_ = [("f", ctypes.c_float), ("mu", ctypes.c_float), ("lr", ctypes.c_float),
                ("eps", ctypes.c_float), ("ns_steps", ctypes.c_int32),
                ("restart_iter", ctypes.c_int32), ("a", ctypes.c_float), ("b", ctypes.c_float),
                ("c", ctypes.c_float), ("ns_dtype", ctypes.c_int32)]


class _Group(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("cols", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("param_dtype", ctypes.c_int32), ("grad_dtype", ctypes.c_int32),
                ("params", ctypes.POINTER(ctypes.c_void_p)),
                ("grads", ctypes.POINTER(ctypes.c_void_p)),
                ("momentum", ctypes.POINTER(ctypes.c_void_p))]


class _NormuonParams(ctypes.Structure):
    _fields_ = [("beta2", ctypes.c_float), ("eps", ctypes.c_float), ("rms", ctypes.c_float)]


class _TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double), ("useful_flops", ctypes.c_double),
                ("algo_bytes", ctypes.c_double)]


_vp, _sz, _i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
_SIGS = {
    "dion3_abi_version": (ctypes.c_size_t, []),
    "dion3_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dion3_last_error": (ctypes.c_char_p, []),
    "dion3_num_selected": (_i32, [ctypes.c_float, _i32]),
    "dion3_useful_flops": (ctypes.c_double, [_i32, _i32, ctypes.POINTER(_HParams)]),
    "dion3_select_workspace_size": (ctypes.c_int, [_i32, _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "dion3_select_rows": (ctypes.c_int, [_i32, _i32, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "dion3_gram_ns_workspace_size": (ctypes.c_int, [_i32, _i32, _i32, ctypes.POINTER(_HParams),
                                                    ctypes.POINTER(_sz)]),
    "dion3_gram_ns_batched": (ctypes.c_int, [_i32, _i32, _i32, _vp, _vp, ctypes.POINTER(_HParams),
                                             _vp, _sz, _vp]),
    "dion3_workspace_size": (ctypes.c_int, [ctypes.POINTER(_Group), _i32, ctypes.POINTER(_HParams),
                                            ctypes.POINTER(_sz)]),
    "dion3_step": (ctypes.c_int, [ctypes.POINTER(_Group), _i32, ctypes.POINTER(_HParams), _vp, _sz,
                                  ctypes.POINTER(_vp), _vp]),
    "dion3_device_status": (ctypes.c_int, [_vp]),
    "dion3_step_lazy": (ctypes.c_int, [ctypes.POINTER(_Group), _i32, ctypes.POINTER(_HParams),
                                       ctypes.POINTER(_vp), _vp, _sz, ctypes.POINTER(_vp), _vp]),
    "dion3_flush_row_scale": (ctypes.c_int, [_i32, _i32, _i32, ctypes.POINTER(_vp), _vp, _vp]),
    "dion3_step_normuon": (ctypes.c_int, [ctypes.POINTER(_Group), _i32, ctypes.POINTER(_HParams),
                                          ctypes.POINTER(_NormuonParams), ctypes.POINTER(_vp), _vp, _sz,
                                          ctypes.POINTER(_vp), _vp]),
    "dion3_gemm_f16": (ctypes.c_int, [_i32, _i32, _i32, _i32, _i32,
                                      _vp, _i32, ctypes.c_int64, _vp, _i32, ctypes.c_int64,
                                      _vp, _i32, ctypes.c_int64, _vp, _i32, ctypes.c_int64,
                                      _vp, _i32, ctypes.c_int64,
                                      ctypes.c_float, ctypes.c_float, ctypes.c_float, _vp]),
    "dion3_trace_enable": (ctypes.c_int, [_i32]),
    "dion3_ns_useful_flops": (ctypes.c_double, [_i32, _i32, _i32, ctypes.POINTER(_HParams)]),
    "dion3_ns_workspace_size": (ctypes.c_int, [_i32, _i32, _i32, _i32, ctypes.POINTER(_HParams),
                                               ctypes.POINTER(_sz)]),
    "dion3_ns_batched": (ctypes.c_int, [_i32, _i32, _i32, _i32, _vp, _vp, ctypes.POINTER(_HParams),
                                        _vp, _sz, _vp]),
    "dion3_select_rows_noalloc": (ctypes.c_int, [_i32, _i32, _i32, ctypes.POINTER(_vp),
                                                 ctypes.POINTER(_vp), _i32, _i32, _vp, _vp, _vp]),
    "dion3_trace_collect": (ctypes.c_int, [ctypes.POINTER(_TraceEntry), _i32, ctypes.POINTER(_i32)]),
    "dion3_wait_probe": (ctypes.c_int, [_i32, ctypes.c_int64, _vp]),
    "dion3_set_overlap": (ctypes.c_int, [_i32]),
}

_LIB = None


def load_library(path: Optional[str] = None):
    """Load libdion3.so (built by :func:`build`); raises if it is missing."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -m "
                           "matrix_orthogonalizing_optimizer_shape_gb300._build)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.dion3_abi_version() != ABI_VERSION:
        raise RuntimeError("libdion3.so ABI version mismatch")
    if path is None:
        _LIB = lib
    return lib


def _check(status: int):
    if status != OK:
        lib = load_library()
        raise Dion3Error(status, (lib.dion3_status_string(status) or b"").decode() + ": "
                         + (lib.dion3_last_error() or b"").decode())


# ---------------------------------------------------------------------------
# Marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t) -> int:
    """Device address of a tensor (or an int address)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _dtype_code(t) -> int:
    import torch
    return {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}[t.dtype]


@dataclass
class HParams:
    """Hyperparameters of one step (mirrors ``dion3_hparams``)."""
    f: float = 1.0
    mu: float = 0.95
    lr: float = 0.02
    eps: float = 1e-7
    ns_steps: int = 5
    restart_iter: int = 3
    coeffs: tuple = MUON_QUINTIC
    ns_dtype: int = F16

    def c_struct(self) -> _HParams:
        a, b, c = self.coeffs
        return _HParams(self.f, self.mu, self.lr, self.eps, self.ns_steps, self.restart_iter,
                        a, b, c, self.ns_dtype)


@dataclass
class Group:
    """A shape group: same-shape parameter, gradient and momentum tensors."""
    params: Sequence
    grads: Sequence
    momentum: Sequence
    _keep: list = field(default_factory=list, repr=False)

    def c_struct(self) -> _Group:
        n = len(self.params)
        if not (len(self.grads) == len(self.momentum) == n) or n == 0:
            raise ValueError("params, grads and momentum must be non-empty and of equal length")
        rows, cols = self.params[0].shape
        arr = ctypes.c_void_p * n
        P = arr(*[_ptr(t) for t in self.params])
        G = arr(*[_ptr(t) for t in self.grads])
        M = arr(*[_ptr(t) for t in self.momentum])
        self._keep = [P, G, M]
        return _Group(rows, cols, n, _dtype_code(self.params[0]), _dtype_code(self.grads[0]),
                      ctypes.cast(P, ctypes.POINTER(ctypes.c_void_p)),
                      ctypes.cast(G, ctypes.POINTER(ctypes.c_void_p)),
                      ctypes.cast(M, ctypes.POINTER(ctypes.c_void_p)))


def alloc_workspace(nbytes: int, device=None):
    """A device byte tensor of at least ``nbytes`` bytes (256-byte aligned)."""
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def num_selected(f: float, rows: int) -> int:
    return int(load_library().dion3_num_selected(f, rows))


def useful_flops(k: int, m: int, hp: HParams) -> float:
    hs = hp.c_struct()
    return float(load_library().dion3_useful_flops(k, m, ctypes.byref(hs)))


def select_workspace_size(rows: int, cols: int, batch: int, k: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().dion3_select_workspace_size(rows, cols, batch, k, ctypes.byref(out)))
    return out.value


def gram_ns_workspace_size(k: int, m: int, batch: int, hp: HParams) -> int:
    out = ctypes.c_size_t(0)
    hs = hp.c_struct()
    _check(load_library().dion3_gram_ns_workspace_size(k, m, batch, ctypes.byref(hs),
                                                       ctypes.byref(out)))
    return out.value


def workspace_size(groups: Sequence[Group], hp: HParams) -> int:
    out = ctypes.c_size_t(0)
    cg = (_Group * len(groups))(*[g.c_struct() for g in groups])
    hs = hp.c_struct()
    _check(load_library().dion3_workspace_size(cg, len(groups), ctypes.byref(hs), ctypes.byref(out)))
    return out.value


def select_rows(momentum: Sequence, grads: Optional[Sequence], k: int, idx_out, fro2_out, ws,
                stream=None, ws_bytes: Optional[int] = None):
    """Step (a): optional M += G, then top-k rows by l1 (see dion3_select_rows)."""
    n = len(momentum)
    rows, cols = momentum[0].shape
    M = (ctypes.c_void_p * n)(*[_ptr(t) for t in momentum])
    G = (ctypes.c_void_p * n)(*[_ptr(t) for t in grads]) if grads is not None else None
    gd = _dtype_code(grads[0]) if grads is not None else F32
    nbytes = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    _check(load_library().dion3_select_rows(
        rows, cols, n, M, G, gd, k, _ptr(idx_out), _ptr(fro2_out), _ptr(ws), nbytes,
        _stream(stream)))


#: Largest batch * rows dion3_select_rows_noalloc accepts (its static scratch).
NOALLOC_MAX_ROWS = 1 << 20


def select_rows_noalloc(momentum: Sequence, grads: Optional[Sequence], k: int, idx_out, fro2_out,
                        stream=None):
    """Step (a) without a workspace, for callers that may not allocate device
    memory while stepping (see dion3_select_rows_noalloc).  Uses a static
    8 MiB scratch inside the library: batch * rows <= NOALLOC_MAX_ROWS, and
    calls that overlap on the GPU race on it."""
    n = len(momentum)
    rows, cols = momentum[0].shape
    M = (ctypes.c_void_p * n)(*[_ptr(t) for t in momentum])
    G = (ctypes.c_void_p * n)(*[_ptr(t) for t in grads]) if grads is not None else None
    gd = _dtype_code(grads[0]) if grads is not None else F32
    _check(load_library().dion3_select_rows_noalloc(
        rows, cols, n, M, G, gd, k, _ptr(idx_out), _ptr(fro2_out), _stream(stream)))


def gram_ns_batched(X, O, hp: HParams, ws, stream=None, ws_bytes: Optional[int] = None):
    """Step (b): O = GramNS(X / (||X||_F + eps)) for X of shape [batch, k, m] in
    hp.ns_dtype (fp16 or bf16)."""
    if X.dim() == 2:
        batch, (k, m) = 1, X.shape
    else:
        batch, k, m = X.shape
    hs = hp.c_struct()
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(load_library().dion3_gram_ns_batched(k, m, batch, _ptr(X), _ptr(O), ctypes.byref(hs),
                                                _ptr(ws), nbytes, _stream(stream)))


def step(groups: Sequence[Group], hp: HParams, ws, sel_idx_out: Optional[Sequence] = None,
         stream=None, ws_bytes: Optional[int] = None):
    """The whole Dion3 step over shape groups (see dion3_step)."""
    cg = (_Group * len(groups))(*[g.c_struct() for g in groups])
    hs = hp.c_struct()
    sel = None
    if sel_idx_out is not None:
        sel = (ctypes.c_void_p * len(groups))(*[_ptr(t) for t in sel_idx_out])
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(load_library().dion3_step(cg, len(groups), ctypes.byref(hs), _ptr(ws), nbytes, sel,
                                     _stream(stream)))


NS_GRAM, NS_GRAM_DENSE, NS_STANDARD, NS_STANDARD_DENSE = 0, 1, 2, 3


def ns_useful_flops(variant: int, k: int, m: int, hp: HParams) -> float:
    hs = hp.c_struct()
    return float(load_library().dion3_ns_useful_flops(variant, k, m, ctypes.byref(hs)))


def ns_workspace_size(variant: int, k: int, m: int, batch: int, hp: HParams) -> int:
    out = ctypes.c_size_t(0)
    hs = hp.c_struct()
    _check(load_library().dion3_ns_workspace_size(variant, k, m, batch, ctypes.byref(hs),
                                                  ctypes.byref(out)))
    return out.value


def ns_batched(variant: int, X, O, hp: HParams, ws, stream=None, ws_bytes: Optional[int] = None):
    """Newton-Schulz variant `variant` of X [batch, k, m] (hp.ns_dtype) into O (see
    dion3_ns_batched)."""
    if X.dim() == 2:
        batch, (k, m) = 1, X.shape
    else:
        batch, k, m = X.shape
    hs = hp.c_struct()
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(load_library().dion3_ns_batched(variant, k, m, batch, _ptr(X), _ptr(O), ctypes.byref(hs),
                                           _ptr(ws), nbytes, _stream(stream)))


GEMM_RECT, GEMM_SYM_LOWER = 0, 1
#: Mode flags for half-stored symmetric matrices (see dion3_gemm_f16): only the
#: 256 x 256 blocks below the block diagonal and the full diagonal blocks hold
#: valid values.
GEMM_OUT_HALF, GEMM_A_HALF, GEMM_B_HALF = 0x10, 0x20, 0x40
#: Mode flags for operands passed as their transpose (A stored [K][M], B [K][N]).
GEMM_A_TRANS, GEMM_B_TRANS = 0x100, 0x200


def gemm_f16(A, B, D=None, DT=None, C=None, *, mode: int = GEMM_RECT, alpha: float = 1.0,
             beta: float = 0.0, gamma: float = 0.0, stream=None):
    """V = alpha A B^T + beta C + gamma I on fp16 [batch, rows, cols] tensors
    (see dion3_gemm_f16); 2-D tensors are a batch of one.  Pitches and batch
    strides are taken from the tensors' strides.  With GEMM_A_TRANS (GEMM_B_TRANS)
    in `mode`, the tensor passed as A (B) holds A^T (B^T)."""
    def geom(t, rows_dim=-2):
        if t is None:
            return 0, 0, 0
        st = t.stride()
        return _ptr(t), st[-2], (st[0] if t.dim() == 3 else st[-2] * t.shape[-2])
    batch = A.shape[0] if A.dim() == 3 else 1
    M, K = (A.shape[-1], A.shape[-2]) if mode & GEMM_A_TRANS else (A.shape[-2], A.shape[-1])
    N = B.shape[-1] if mode & GEMM_B_TRANS else B.shape[-2]
    a, b, c, d, dt = geom(A), geom(B), geom(C), geom(D), geom(DT)
    _check(load_library().dion3_gemm_f16(mode, M, N, K, batch, *a, *b, *c, *d, *dt,
                                         alpha, beta, gamma, _stream(stream)))


def trace_enable(on: bool = True):
    """Start (or stop) recording per-launch CUDA events (see dion3_trace_enable)."""
    _check(load_library().dion3_trace_enable(1 if on else 0))


def trace_collect() -> dict:
    """{kernel: {launches, total_ms, useful_flops, algo_bytes}} since the last
    collect; waits for the recorded events."""
    lib = load_library()
    cap = 32
    buf = (_TraceEntry * cap)()
    n = ctypes.c_int32(0)
    _check(lib.dion3_trace_collect(buf, cap, ctypes.byref(n)))
    out = {}
    for i in range(min(n.value, cap)):
        e = buf[i]
        out[e.name.decode()] = {"launches": int(e.launches), "total_ms": float(e.total_ms),
                                "useful_flops": float(e.useful_flops),
                                "algo_bytes": float(e.algo_bytes)}
    return out


def step_lazy(groups: Sequence[Group], hp: HParams, row_scale: Sequence, ws,
              sel_idx_out: Optional[Sequence] = None, stream=None, ws_bytes: Optional[int] = None):
    """dion3_step with the selected rows' decay left pending in row_scale (one
    fp32 [batch, rows] tensor per group, all ones before the first call); see
    dion3_step_lazy."""
    cg = (_Group * len(groups))(*[g.c_struct() for g in groups])
    hs = hp.c_struct()
    rs = (ctypes.c_void_p * len(groups))(*[_ptr(t) for t in row_scale])
    sel = None
    if sel_idx_out is not None:
        sel = (ctypes.c_void_p * len(groups))(*[_ptr(t) for t in sel_idx_out])
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(load_library().dion3_step_lazy(cg, len(groups), ctypes.byref(hs), rs, _ptr(ws), nbytes, sel,
                                          _stream(stream)))


@dataclass
class NormuonParams:
    """Per-neuron normalisation of dion3_step_normuon (NorMuon form, a reading:
    the pages name it but do not define it)."""
    beta2: float = 0.95
    eps: float = 1e-8
    rms: float = 0.2

    def c_struct(self) -> _NormuonParams:
        return _NormuonParams(self.beta2, self.eps, self.rms)


def step_normuon(groups: Sequence[Group], hp: HParams, nm: NormuonParams, v: Sequence, ws,
                 sel_idx_out: Optional[Sequence] = None, stream=None, ws_bytes: Optional[int] = None):
    """dion3_step with the per-neuron normalisation (see dion3_step_normuon):
    one fp32 [batch, rows] state tensor per group in v, zeros before the first
    call."""
    cg = (_Group * len(groups))(*[g.c_struct() for g in groups])
    hs = hp.c_struct()
    ns = nm.c_struct()
    vs = (ctypes.c_void_p * len(groups))(*[_ptr(t) for t in v])
    sel = None
    if sel_idx_out is not None:
        sel = (ctypes.c_void_p * len(groups))(*[_ptr(t) for t in sel_idx_out])
    nbytes = ws_bytes if ws_bytes is not None else ws.numel() * ws.element_size()
    _check(load_library().dion3_step_normuon(cg, len(groups), ctypes.byref(hs), ctypes.byref(ns), vs,
                                             _ptr(ws), nbytes, sel, _stream(stream)))


def flush_row_scale(momentum: Sequence, row_scale, stream=None):
    """Apply pending lazy decays of one group in place (dion3_flush_row_scale)."""
    n = len(momentum)
    rows, cols = momentum[0].shape
    M = (ctypes.c_void_p * n)(*[_ptr(t) for t in momentum])
    _check(load_library().dion3_flush_row_scale(rows, cols, n, M, _ptr(row_scale), _stream(stream)))


def set_overlap(on: bool):
    """Overlap each shape group's accumulation with the previous group's
    Newton-Schulz GEMMs in :func:`step` (default on; see dion3_set_overlap)."""
    _check(load_library().dion3_set_overlap(1 if on else 0))


def wait_probe(arrive: bool, limit_ns: int, stream=None):
    """Run the library's bounded device-side wait on its own (dion3_wait_probe):
    with ``arrive`` False the wait runs out after ``limit_ns`` and the next
    :func:`device_status` raises the timeout."""
    _check(load_library().dion3_wait_probe(1 if arrive else 0, int(limit_ns), _stream(stream)))


def device_status(stream=None):
    """Synchronise and raise if a bounded device-side wait ran out."""
    _check(load_library().dion3_device_status(_stream(stream)))
