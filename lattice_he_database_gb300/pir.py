"""Thin Python binding of libpir.so (include/pir.h).

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  Functions carry the C names; tensors are torch CUDA tensors (used as
plain device buffers), streams are torch.cuda.Stream objects or None for the
current stream.  A non-zero return code raises PirError.  The library must
have been built (``lattice_he_database_gb300.build.build()``); there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

PIR_OK = 0
PIR_ERR_ARG = -1
PIR_ERR_CUDA = -2
PIR_ERR_UNSUPPORTED = -3
PIR_ERR_ALLOC = -4
PIR_STATUS_TIMEOUT = 1
PIR_SLAB = 128


class PirError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, pir_strerror(code) if _lib else "?", code))


_lib = None
_u32p = ctypes.POINTER(ctypes.c_uint32)
_vp = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """Load libpir.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libpir.so not built: run lattice_he_database_gb300.build.build()")
        L = ctypes.CDLL(_build.LIB)
        L.pir_params_check.restype = ctypes.c_int
        L.pir_params_check.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p]
        L.pir_primes.restype = ctypes.c_int
        L.pir_primes.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u32p]
        L.pir_ctx_create.restype = ctypes.c_int
        L.pir_ctx_create.argtypes = [ctypes.POINTER(_vp), ctypes.c_uint32, ctypes.c_uint32, _u32p, ctypes.c_int]
        L.pir_ctx_destroy.restype = None
        L.pir_ctx_destroy.argtypes = [_vp]
        L.pir_ctx_psi.restype = ctypes.c_int
        L.pir_ctx_psi.argtypes = [_vp, _u32p]
        for name in ("pir_ntt_fwd", "pir_ntt_inv", "pir_lift_ntt"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [_vp, _vp, _vp, ctypes.c_uint64, _vp]
        L.pir_db_bytes.restype = ctypes.c_uint64
        L.pir_db_bytes.argtypes = [_vp, ctypes.c_uint32, ctypes.c_uint32]
        L.pir_db_encode.restype = ctypes.c_int
        L.pir_db_encode.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                    _vp, _vp]
        L.pir_rowsel_workspace_bytes.restype = ctypes.c_uint64
        L.pir_rowsel_workspace_bytes.argtypes = [_vp, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        L.pir_rowsel.restype = ctypes.c_int
        L.pir_rowsel.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, _vp, ctypes.c_uint32, _vp, _vp,
                                 ctypes.c_uint64, _vp]
        L.pir_scalar_workspace_bytes.restype = ctypes.c_uint64
        L.pir_exppack.restype = ctypes.c_int
        L.pir_exppack.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, _vp, _vp, ctypes.c_uint32, _vp, _vp,
                                  ctypes.c_uint64, _vp]
        L.pir_server_create.restype = ctypes.c_int
        L.pir_server_create.argtypes = [ctypes.POINTER(_vp), _vp, _vp, ctypes.c_uint32, ctypes.c_uint32,
                                        ctypes.c_uint32]
        L.pir_server_destroy.restype = None
        L.pir_server_destroy.argtypes = [_vp]
        L.pir_server_submit.restype = ctypes.c_int
        L.pir_server_submit.argtypes = [_vp, _vp, _vp, ctypes.POINTER(ctypes.c_uint64)]
        L.pir_server_wait.restype = ctypes.c_int
        L.pir_server_wait.argtypes = [_vp, ctypes.c_uint64]
        L.pir_server_mark.restype = ctypes.c_int
        L.pir_server_mark.argtypes = [_vp, ctypes.c_int]
        L.pir_server_elapsed_ms.restype = ctypes.c_int
        L.pir_server_elapsed_ms.argtypes = [_vp, ctypes.POINTER(ctypes.c_float)]
        L.pir_scalar_workspace_bytes.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        L.pir_scalar_scan.restype = ctypes.c_int
        L.pir_scalar_scan.argtypes = [_vp, _vp, ctypes.c_uint64, ctypes.c_uint64, _vp, ctypes.c_uint32, _vp,
                                      _vp, ctypes.c_uint64, _vp]
        L.pir_coltor_workspace_bytes.restype = ctypes.c_uint64
        L.pir_coltor_workspace_bytes.argtypes = [_vp, ctypes.c_uint64, ctypes.c_uint32]
        for name in ("pir_coltor_stage", "pir_coltor"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, _vp, ctypes.c_uint64, _vp, _vp,
                          ctypes.c_uint64, _vp]
        L.pir_expand_workspace_bytes.restype = ctypes.c_uint64
        L.pir_expand_workspace_bytes.argtypes = [_vp, ctypes.c_uint64, ctypes.c_uint32]
        L.pir_expand_stage.restype = ctypes.c_int
        L.pir_expand_stage.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _vp,
                                       ctypes.c_uint64, _vp, _vp, ctypes.c_uint64, _vp]
        L.pir_expand.restype = ctypes.c_int
        L.pir_expand.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _vp, _vp, _vp,
                                 ctypes.c_uint64, _vp]
        L.pir_coltor_batch_workspace_bytes.restype = ctypes.c_uint64
        L.pir_coltor_batch_workspace_bytes.argtypes = [_vp, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
        L.pir_coltor_batch.restype = ctypes.c_int
        L.pir_coltor_batch.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, _vp, ctypes.c_uint64,
                                       ctypes.c_uint64, _vp, _vp, ctypes.c_uint64, _vp]
        L.pir_expand_batch.restype = ctypes.c_int
        L.pir_expand_batch.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, _vp,
                                       ctypes.c_uint64, _vp, _vp, ctypes.c_uint64, _vp]
        L.pir_rgsw_convert_workspace_bytes.restype = ctypes.c_uint64
        L.pir_rgsw_convert_workspace_bytes.argtypes = [_vp, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
        L.pir_rgsw_convert.restype = ctypes.c_int
        L.pir_rgsw_convert.argtypes = [_vp, _vp, ctypes.c_uint32, ctypes.c_uint32, _vp, ctypes.c_uint64,
                                       ctypes.c_uint64, ctypes.c_uint64, _vp, _vp, ctypes.c_uint64, _vp]
        L.pir_status.restype = ctypes.c_int
        L.pir_status.argtypes = [_vp, _u32p, ctypes.c_int]
        L.pir_ctx_set_wait_limit.restype = ctypes.c_int
        L.pir_ctx_set_wait_limit.argtypes = [_vp, ctypes.c_uint64]
        L.pir_ctx_set_test_hook.restype = ctypes.c_int
        L.pir_ctx_set_test_hook.argtypes = [_vp, ctypes.c_uint32]
        L.pir_strerror.restype = ctypes.c_char_p
        L.pir_strerror.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def pir_strerror(code: int) -> str:
    return lib().pir_strerror(code).decode()


def _check(rc: int, what: str):
    if rc != PIR_OK:
        raise PirError(rc, what)


def _qarr(qs):
    arr = (ctypes.c_uint32 * max(1, len(qs)))(*[int(q) for q in qs])
    return arr


def _dev_ptr(t: torch.Tensor, itemsize: int, what: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if t.element_size() != itemsize:
        raise ValueError("%s must have %d-byte elements" % (what, itemsize))
    return t.data_ptr()


def _host_ptr(t: torch.Tensor, nbytes: int, what: str) -> int:
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError("%s must be a host tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    if t.numel() * t.element_size() < nbytes:
        raise ValueError("%s holds %d bytes, needs %d" % (what, t.numel() * t.element_size(), nbytes))
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- context
def pir_params_check(N: int, qs) -> int:
    return lib().pir_params_check(N, len(qs), _qarr(qs))


def pir_primes(N: int, L: int) -> list[int]:
    """The L largest primes < 2^29 with q = 1 mod 2N (descending)."""
    out = (ctypes.c_uint32 * max(1, L))()
    _check(lib().pir_primes(N, L, out), "pir_primes")
    return [int(v) for v in out[:L]]


class Ctx:
    """Owning handle of a pir_ctx (destroyed on close/GC)."""

    def __init__(self, handle: int, N: int, qs, device: int):
        self.handle = handle
        self.N = N
        self.qs = [int(q) for q in qs]
        self.L = len(self.qs)
        self.device = device

    def close(self):
        if self.handle:
            lib().pir_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def _as_parameter_(self):
        return _vp(self.handle)


def pir_ctx_create(N: int, qs, device: int = 0) -> Ctx:
    h = _vp()
    _check(lib().pir_ctx_create(ctypes.byref(h), N, len(qs), _qarr(qs), device), "pir_ctx_create")
    return Ctx(h.value, N, qs, device)


def pir_ctx_destroy(ctx: Ctx):
    ctx.close()


def pir_ctx_psi(ctx: Ctx) -> list[int]:
    out = (ctypes.c_uint32 * ctx.L)()
    _check(lib().pir_ctx_psi(ctx, out), "pir_ctx_psi")
    return [int(v) for v in out]


def pir_status(ctx: Ctx, clear: bool = True) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib().pir_status(ctx, ctypes.byref(flags), int(clear)), "pir_status")
    return int(flags.value)


PIR_HOOK_NONE = 0
PIR_HOOK_WITHHOLD_LAST_COPY = 1


def pir_ctx_set_wait_limit(ctx: Ctx, ns: int):
    """Limit of the kernels' ordinary device waits (0 = the default 2 s)."""
    _check(lib().pir_ctx_set_wait_limit(ctx, ns), "pir_ctx_set_wait_limit")


def pir_ctx_set_test_hook(ctx: Ctx, hook: int):
    """Failure-path test hook (PIR_HOOK_*); PIR_HOOK_NONE in normal use."""
    _check(lib().pir_ctx_set_test_hook(ctx, hook), "pir_ctx_set_test_hook")


# ---------------------------------------------------------------- NTT
def pir_ntt_fwd(ctx: Ctx, inp: torch.Tensor, out: torch.Tensor, cnt: int, stream=None):
    _check(lib().pir_ntt_fwd(ctx, _dev_ptr(inp, 4, "in"), _dev_ptr(out, 4, "out"), cnt, _stream(stream)),
           "pir_ntt_fwd")


def pir_ntt_inv(ctx: Ctx, inp: torch.Tensor, out: torch.Tensor, cnt: int, stream=None):
    _check(lib().pir_ntt_inv(ctx, _dev_ptr(inp, 4, "in"), _dev_ptr(out, 4, "out"), cnt, _stream(stream)),
           "pir_ntt_inv")


def pir_lift_ntt(ctx: Ctx, raw: torch.Tensor, out: torch.Tensor, cnt: int, stream=None):
    """out[i][l] = NTT(raw[i] mod q_l): [cnt][N] plain words -> [cnt][L][N]."""
    _check(lib().pir_lift_ntt(ctx, _dev_ptr(raw, 4, "raw"), _dev_ptr(out, 4, "out"), cnt, _stream(stream)),
           "pir_lift_ntt")


# ---------------------------------------------------------------- RowSel
def pir_db_bytes(ctx: Ctx, D0: int, D1: int) -> int:
    return int(lib().pir_db_bytes(ctx, D0, D1))


def pir_db_encode(ctx: Ctx, raw: torch.Tensor, k0: int, kcnt: int, D0: int, D1: int, db: torch.Tensor,
                  stream=None):
    _check(lib().pir_db_encode(ctx, _dev_ptr(raw, 4, "raw"), k0, kcnt, D0, D1, _dev_ptr(db, 4, "db"),
                               _stream(stream)), "pir_db_encode")


def pir_rowsel_workspace_bytes(ctx: Ctx, D0: int, D1: int, B: int) -> int:
    return int(lib().pir_rowsel_workspace_bytes(ctx, D0, D1, B))


def pir_rowsel(ctx: Ctx, db: torch.Tensor, D0: int, D1: int, query: torch.Tensor, B: int, out: torch.Tensor,
               workspace: torch.Tensor, stream=None):
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_rowsel(ctx, _dev_ptr(db, 4, "db"), D0, D1, _dev_ptr(query, 4, "query"), B,
                            _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                            _stream(stream)), "pir_rowsel")


def rowsel_workspace(ctx: Ctx, D0: int, D1: int, B: int, device="cuda") -> torch.Tensor:
    """A device workspace sized for pir_rowsel(D0, D1, B)."""
    return torch.empty(pir_rowsel_workspace_bytes(ctx, D0, D1, B), dtype=torch.uint8, device=device)


def pir_exppack(ctx: Ctx, h_db: torch.Tensor, n: int, Dr: int, C: torch.Tensor, G: torch.Tensor, B: int,
                out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """out = H*C + (0|G) point-wise mod q (ring-packing GEMM); h_db encoded with D0 = n, D1 = Dr."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_exppack(ctx, _dev_ptr(h_db, 4, "h_db"), n, Dr, _dev_ptr(C, 4, "C"), _dev_ptr(G, 4, "G"), B,
             _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(), _stream(stream)),
           "pir_exppack")


# ---------------------------------------------------------------- ColTor
def pir_coltor_workspace_bytes(ctx: Ctx, n: int, ell: int) -> int:
    return int(lib().pir_coltor_workspace_bytes(ctx, n, ell))


def coltor_workspace(ctx: Ctx, n: int, ell: int, device="cuda") -> torch.Tensor:
    """A device workspace sized for pir_coltor / pir_coltor_stage over n ciphertexts."""
    return torch.empty(pir_coltor_workspace_bytes(ctx, n, ell), dtype=torch.uint8, device=device)


def pir_coltor_stage(ctx: Ctx, C: torch.Tensor, ell: int, w: int, cts: torch.Tensor, n: int, out: torch.Tensor,
                     workspace: torch.Tensor, stream=None):
    """out_i = ct_2i + C (x) (ct_2i+1 - ct_2i), i < ceil(n/2) (all NTT form)."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_coltor_stage(ctx, _dev_ptr(C, 4, "C"), ell, w, _dev_ptr(cts, 4, "in"), n,
                                  _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "pir_coltor_stage")


def pir_coltor(ctx: Ctx, C: torch.Tensor, ell: int, w: int, cts: torch.Tensor, n: int, out: torch.Tensor,
               workspace: torch.Tensor, stream=None):
    """The whole tournament over n ciphertexts; C holds ceil(log2 n) stages' RGSW ciphertexts."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_coltor(ctx, _dev_ptr(C, 4, "C"), ell, w, _dev_ptr(cts, 4, "in"), n,
                            _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                            _stream(stream)), "pir_coltor")


def pir_coltor_batch_workspace_bytes(ctx: Ctx, n: int, G: int, ell: int) -> int:
    return int(lib().pir_coltor_batch_workspace_bytes(ctx, n, G, ell))


def coltor_batch_workspace(ctx: Ctx, n: int, G: int, ell: int, device="cuda") -> torch.Tensor:
    """A device workspace sized for pir_coltor_batch: G tournaments of n ciphertexts."""
    return torch.empty(pir_coltor_batch_workspace_bytes(ctx, n, G, ell), dtype=torch.uint8, device=device)


def pir_coltor_batch(ctx: Ctx, C: torch.Tensor, ell: int, w: int, cts: torch.Tensor, n: int, G: int,
                     out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """G tournaments of n ciphertexts each ([G][n] in, [G] out); C holds each
    client's ceil(log2 n) stages' RGSW ciphertexts, client after client."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_coltor_batch(ctx, _dev_ptr(C, 4, "C"), ell, w, _dev_ptr(cts, 4, "in"), n, G,
                                  _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "pir_coltor_batch")


# ---------------------------------------------------------------- ExpandQuery
def pir_expand_workspace_bytes(ctx: Ctx, M: int, ell: int) -> int:
    return int(lib().pir_expand_workspace_bytes(ctx, M, ell))


def expand_workspace(ctx: Ctx, M: int, ell: int, device="cuda") -> torch.Tensor:
    """A device workspace for expansion stages of up to M input ciphertexts."""
    return torch.empty(pir_expand_workspace_bytes(ctx, M, ell), dtype=torch.uint8, device=device)


def pir_expand_stage(ctx: Ctx, evk: torch.Tensor, ell: int, w: int, j: int, cts: torch.Tensor, M: int,
                     out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """Stage j of ExpandQuery: M ciphertexts -> 2M (NTT form)."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_expand_stage(ctx, _dev_ptr(evk, 4, "evk"), ell, w, j, _dev_ptr(cts, 4, "in"), M,
                                  _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "pir_expand_stage")


def pir_expand(ctx: Ctx, evks: torch.Tensor, ell: int, w: int, stages: int, ct: torch.Tensor, out: torch.Tensor,
               workspace: torch.Tensor, stream=None):
    """ExpandQuery: one ciphertext -> 2^stages ciphertexts (NTT form)."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_expand(ctx, _dev_ptr(evks, 4, "evks"), ell, w, stages, _dev_ptr(ct, 4, "ct"),
                            _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                            _stream(stream)), "pir_expand")


def pir_expand_batch(ctx: Ctx, evks: torch.Tensor, ell: int, w: int, stages: int, ct: torch.Tensor, G: int,
                     out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """G expansions ([G] query ciphertexts in, [G][2^stages] out); evks holds
    each client's stages' keys, client after client.  The workspace is
    expand_workspace(ctx, G * 2^(stages-1), ell)."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_expand_batch(ctx, _dev_ptr(evks, 4, "evks"), ell, w, stages, _dev_ptr(ct, 4, "ct"), G,
                                  _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "pir_expand_batch")


# ---------------------------------------------------------------- scalar scan
def pir_scalar_workspace_bytes(C: int, B: int) -> int:
    return int(lib().pir_scalar_workspace_bytes(C, B))


def pir_scalar_scan(ctx: Ctx, db: torch.Tensor, R: int, C: int, Q: torch.Tensor, B: int, out: torch.Tensor,
                    workspace: torch.Tensor, stream=None):
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_scalar_scan(ctx, _dev_ptr(db, 1, "db"), R, C, _dev_ptr(Q, 4, "Q"), B, _dev_ptr(out, 4, "out"),
                                 ws, workspace.numel() * workspace.element_size(), _stream(stream)),
           "pir_scalar_scan")


def pir_scalar_scan_noalloc(ctx: Ctx, db: torch.Tensor, R: int, C: int, Q: torch.Tensor, B: int,
                            out: torch.Tensor, stream=None):
    """pir_scalar_scan without a workspace argument: the library stages the
    split query in its own static device array (C <= 16384), allocating
    nothing.  For callers that cannot allocate device memory per call."""
    f = lib().pir_scalar_scan_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [_vp, _vp, ctypes.c_uint64, ctypes.c_uint64, _vp, ctypes.c_uint32, _vp, _vp]
    _check(f(ctx, _dev_ptr(db, 1, "db"), R, C, _dev_ptr(Q, 4, "Q"), B, _dev_ptr(out, 4, "out"), _stream(stream)),
           "pir_scalar_scan_noalloc")


# ---------------------------------------------------------------- helpers
def empty_u32(n, device="cuda") -> torch.Tensor:
    """A flat device buffer of n uint32 words (int32 storage)."""
    return torch.empty(int(n), dtype=torch.int32, device=device)


def db_layout_offset(N: int, L: int, D0: int, D1: int, p, k, n):
    """Word offset of (evaluation point p, DB row k, DB column n) in the encoded DB
    (numpy/int arrays broadcast).  Mirrors the layout documented in pir.h."""
    import numpy as np
    D1p = (D1 + 3) // 4 * 4
    S = (D1 + PIR_SLAB - 1) // PIR_SLAB
    Wl = D1p - PIR_SLAB * (S - 1)
    p = np.asarray(p, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    n = np.asarray(n, dtype=np.int64)
    s = n // PIR_SLAB
    Ws = np.where(s == S - 1, Wl, PIR_SLAB)
    return p * D0 * D1p + s * D0 * PIR_SLAB + k * Ws + (n - PIR_SLAB * s)


class RowselServer:
    """RowSel serving path: an encoded DB resident in HBM, answering query
    batches given in coefficient form (host or device), through the C ABI:
    forward NTT of the query, the scan, inverse NTT of the result."""

    def __init__(self, ctx: Ctx, db: torch.Tensor, D0: int, D1: int, B: int, stream=None):
        self.ctx, self.db, self.D0, self.D1, self.B = ctx, db, D0, D1, B
        P = ctx.L * ctx.N
        self.q_words = B * D0 * 2 * P
        self.o_words = B * D1 * 2 * P
        dev = db.device
        self.q_coef = empty_u32(self.q_words, dev)
        self.q_ntt = empty_u32(self.q_words, dev)
        self.o_ntt = empty_u32(self.o_words, dev)
        self.o_coef = empty_u32(self.o_words, dev)
        self.ws = rowsel_workspace(ctx, D0, D1, B, dev)
        self.stream = stream or torch.cuda.current_stream(dev)
        self.launches_per_answer = 3

    def answer_device(self, q_coef: torch.Tensor | None = None):
        """Device-resident query (coefficient form) -> device result (coefficient form)."""
        q = self.q_coef if q_coef is None else q_coef
        c = self.ctx
        pir_ntt_fwd(c, q, self.q_ntt, self.B * self.D0 * 2, self.stream)
        pir_rowsel(c, self.db, self.D0, self.D1, self.q_ntt, self.B, self.o_ntt, self.ws, self.stream)
        pir_ntt_inv(c, self.o_ntt, self.o_coef, self.B * self.D1 * 2, self.stream)
        return self.o_coef

    def answer_host(self, q_host: torch.Tensor, o_host: torch.Tensor):
        """Pinned host query in, pinned host result out (copies on the same stream)."""
        with torch.cuda.stream(self.stream):
            self.q_coef.copy_(q_host, non_blocking=True)
            self.answer_device()
            o_host.copy_(self.o_coef, non_blocking=True)
        return o_host


class PirServer:
    """Pipelined query stream over a resident RowSel DB (pir_server_*): host
    queries in coefficient form go in, host results in coefficient form come
    out; copies overlap the scans of neighbouring queries."""

    def __init__(self, ctx: Ctx, db: torch.Tensor, D0: int, D1: int, B: int):
        self.ctx, self.db, self.D0, self.D1, self.B = ctx, db, D0, D1, B
        P = ctx.L * ctx.N
        self.q_bytes = B * D0 * 2 * P * 4
        self.o_bytes = B * D1 * 2 * P * 4
        h = _vp()
        _check(lib().pir_server_create(ctypes.byref(h), ctx, _dev_ptr(db, 4, "db"), D0, D1, B), "pir_server_create")
        self.handle = h.value
        self._keep = {}

    def close(self):
        if self.handle:
            lib().pir_server_destroy(self.handle)
            self.handle = None
            self._keep.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def submit(self, q_host: torch.Tensor, o_host: torch.Tensor) -> int:
        t = ctypes.c_uint64()
        _check(lib().pir_server_submit(self.handle, _host_ptr(q_host, self.q_bytes, "query"),
                                       _host_ptr(o_host, self.o_bytes, "result"), ctypes.byref(t)),
               "pir_server_submit")
        self._keep[t.value % 2] = (q_host, o_host)   # host buffers stay referenced while in flight
        return t.value

    def wait(self, ticket: int):
        _check(lib().pir_server_wait(self.handle, ticket), "pir_server_wait")

    def mark(self, which: int):
        _check(lib().pir_server_mark(self.handle, which), "pir_server_mark")

    def elapsed_ms(self) -> float:
        ms = ctypes.c_float()
        _check(lib().pir_server_elapsed_ms(self.handle, ctypes.byref(ms)), "pir_server_elapsed_ms")
        return float(ms.value)


# ---------------------------------------------------------------- RGSW from the expanded query
def pir_rgsw_convert_workspace_bytes(ctx: Ctx, n: int, G: int, ell: int) -> int:
    return int(lib().pir_rgsw_convert_workspace_bytes(ctx, n, G, ell))


def rgsw_convert_workspace(ctx: Ctx, n: int, G: int, ell: int, device="cuda") -> torch.Tensor:
    """A device workspace for pir_rgsw_convert of G clients x n RGSW ciphertexts."""
    return torch.empty(pir_rgsw_convert_workspace_bytes(ctx, n, G, ell), dtype=torch.uint8, device=device)


def pir_rgsw_convert(ctx: Ctx, ksk: torch.Tensor, ell: int, w: int, cts: torch.Tensor, n: int, G: int,
                     out: torch.Tensor, workspace: torch.Tensor, stream=None, in_stride: int = 0):
    """RGSW ciphertexts [G][n][2 ell][2][L][N] from the expanded gadget
    ciphertexts (client b's n ell of them at b * in_stride ciphertexts,
    in_stride = 0: contiguous) and each client's key-switching key of s^2
    ([G][ell][2][L][N]), all NTT form."""
    ws = _dev_ptr(workspace, workspace.element_size(), "workspace")
    _check(lib().pir_rgsw_convert(ctx, _dev_ptr(ksk, 4, "ksk"), ell, w, _dev_ptr(cts, 4, "in"), in_stride, n, G,
                                  _dev_ptr(out, 4, "out"), ws, workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "pir_rgsw_convert")
