"""ctypes binding of libubgemm (include/ub.h): argument marshalling only.

Every step of the AG-GEMM and GEMM-RS path runs in the library's kernels and copy
engine calls; this module checks tensor dtypes, devices and shapes, passes raw
device pointers and the current CUDA stream, and turns error codes into exceptions.
There is no fallback: if ``libubgemm.so`` is missing, the first call raises.

API modelled on "Support dynamic token counts in TP communication/GEMM overlap"
(TransformerEngine issue #3564), "Proposed API": ``initialize_ub([max_tokens,
hidden], tp_size, dtype=torch.bfloat16)`` registers a buffer at capacity, and
``set_ub_active_shape([T, hidden])`` sets the active shape before each microbatch.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libubgemm.so")
_lib = None

UB_OK = 0
ERRORS = {
    -1: "UB_ERR_ARG", -2: "UB_ERR_DTYPE", -3: "UB_ERR_RANK", -4: "UB_ERR_ZERO",
    -5: "UB_ERR_CAPACITY", -6: "UB_ERR_HIDDEN", -7: "UB_ERR_DIVISIBLE", -8: "UB_ERR_ALIGN",
    -9: "UB_ERR_CUDA", -10: "UB_ERR_TIMEOUT",
}
CODES = {v: k for k, v in ERRORS.items()}
OPTIONS = {"sm_margin": 1, "timeout_ns": 2, "self_rank": 3, "drop_flag": 4, "profile": 5,
           "cta_pair": 6, "streamk": 7, "copy_streams": 8, "gather_kernel": 9, "skinny": 10, "pdl": 11,
           "bulk_beside": 12, "gather_chain": 13}
OPS = {"ag": 0, "rs": 1, "ag_swiglu": 2, "ag_kn": 3, "rs_kn": 4, "wgrad": 5, "reduce_scatter": 6}
MAX_TP = 8
EXPORTS = [
    "ub_create", "ub_destroy", "ub_set_active_shape", "ub_set_active_shape_nd",
    "ub_validate_active_shape", "ub_get_active_shape", "ub_get_capacity", "ub_get_tp",
    "ub_buffer", "ag_gemm", "gemm_rs", "ub_set_option", "ub_get_option", "ub_query_status",
    "ub_clear_status", "ub_get_counters", "ub_kernel_time", "ub_grid_ctas", "ub_last_error",
    "ag_gemm_noalloc", "ag_gemm_swiglu", "ag_gemm_kn", "gemm_rs_kn", "ub_wgrad",
    "ub_allgather", "ub_reduce_scatter", "ub_plan_tail_split", "ub_plan_path",
    "ub_plan_ag_self_head", "ag_gemm_from_buffer", "ub_plan_gather_parts", "ub_stream_read",
    "ub_plan_ag_group_m",
]
NOALLOC_MAX_ELEMS = 16 * 1024 * 1024


class UbError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("%s (%d): %s" % (ERRORS.get(code, "UB_ERR?"), code, msg))
        self.code = code
        self.name = ERRORS.get(code, "UB_ERR?")


class Counters(ctypes.Structure):
    _fields_ = [("ag_calls", ctypes.c_int64), ("rs_calls", ctypes.c_int64),
                ("device_allocations", ctypes.c_int64), ("last_T", ctypes.c_int64),
                ("tensor_map_encodes", ctypes.c_int64), ("last_kernel", ctypes.c_int64),
                ("last_pieces", ctypes.c_int64), ("last_gather", ctypes.c_int64)]


KERNELS = {0: "single", 1: "pair", 2: "few_token"}
GATHERS = {-1: "none", 0: "copies", 1: "gather_kernel", 2: "in_gemm"}


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libubgemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("libubgemm.so is not built (%s); run __graft_entry__.build()" % _LIB_PATH)
    L = ctypes.CDLL(_LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    PP = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "ub_create": [I64, I64, I, I, ctypes.POINTER(P)],
        "ub_destroy": [P],
        "ub_set_active_shape": [P, I64, I64],
        "ub_set_active_shape_nd": [P, I, ctypes.POINTER(I64)],
        "ub_validate_active_shape": [I, ctypes.POINTER(I64), I64, I64, I],
        "ub_get_active_shape": [P, ctypes.POINTER(I64), ctypes.POINTER(I64)],
        "ub_get_capacity": [P, ctypes.POINTER(I64), ctypes.POINTER(I64)],
        "ub_get_tp": [P, ctypes.POINTER(I)],
        "ub_buffer": [P, PP, ctypes.POINTER(ctypes.c_size_t)],
        "ag_gemm": [P, PP, P, I64, P, P],
        "ag_gemm_swiglu": [P, PP, P, I64, P, P],
        "ag_gemm_kn": [P, PP, P, I64, P, P],
        "gemm_rs_kn": [P, PP, PP, I64, PP, P],
        "ub_wgrad": [P, P, I64, I, P, P],
        "ub_allgather": [P, PP, P],
        "ub_reduce_scatter": [P, PP, PP, P],
        "ub_stream_read": [P, P, I64, P],
        "gemm_rs": [P, PP, PP, I64, PP, P],
        "ub_set_option": [P, I, I64],
        "ub_get_option": [P, I, ctypes.POINTER(I64)],
        "ub_query_status": [P],
        "ub_clear_status": [P],
        "ub_get_counters": [P, ctypes.POINTER(Counters)],
        "ub_kernel_time": [P, I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)],
        "ub_grid_ctas": [P, ctypes.POINTER(I)],
        "ub_last_error": [],
        "ag_gemm_noalloc": [PP, I, I64, I64, P, I64, P, P],
        "ag_gemm_from_buffer": [P, P, I64, I64, P, P],
        "ub_plan_tail_split": [I64, I64, I64, I, I],
        "ub_plan_path": [I64, I64, I64, I64, I64, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)],
        "ub_plan_ag_self_head": [I64, I, I, I64, I64],
        "ub_plan_ag_group_m": [I64, I, I, I64, I64],
        "ub_plan_gather_parts": [I, I, I64, I64, ctypes.POINTER(I), ctypes.POINTER(I64), ctypes.POINTER(I64),
                                 ctypes.POINTER(I)],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        if name == "ub_last_error":
            fn.restype = ctypes.c_char_p
        elif name in ("ub_plan_tail_split", "ub_plan_ag_self_head"):
            fn.restype = ctypes.c_int64
        else:
            fn.restype = ctypes.c_int
    _lib = L
    return L


def last_error() -> str:
    return load().ub_last_error().decode(errors="replace")


# ---------------------------------------------------------------- planning queries (host only)

def _plan_check(v: int) -> int:
    if v < 0:
        _check(int(v))
    return int(v)


def plan_tail_split(tiles: int, pairs: int, k_blocks: int, widest: bool = False, gathered: bool = False) -> int:
    """k-pieces per tile of the CTA-pair kernel's last, partial wave (1: whole tiles);
    `gathered` for an AG-GEMM whose rows come through the all-gather."""
    return _plan_check(load().ub_plan_tail_split(tiles, pairs, k_blocks, 1 if widest else 0, 1 if gathered else 0))


def plan_path(single_tiles: int, pair_tiles: int, k_blocks: int, slots: int, pairs: int,
              cta_pair: int = -1, streamk: int = -1, gathered: bool = False) -> tuple:
    """(pair, split) for a tile-kernel call: CTA pairs or single CTAs, split last wave."""
    pr, sp = ctypes.c_int(0), ctypes.c_int(0)
    rc = load().ub_plan_path(single_tiles, pair_tiles, k_blocks, slots, pairs, cta_pair, streamk,
                             1 if gathered else 0, ctypes.byref(pr), ctypes.byref(sp))
    _check(rc)
    return bool(pr.value), bool(sp.value)


def plan_gather_parts(tp: int, self_rank: int, c: int, head: int) -> list:
    """The gather's copies in issue order: (chunk, row_lo, row_hi, publishes_flag)."""
    n_max = MAX_TP + 1
    ch = (ctypes.c_int * n_max)()
    lo = (ctypes.c_int64 * n_max)()
    hi = (ctypes.c_int64 * n_max)()
    fl = (ctypes.c_int * n_max)()
    n = load().ub_plan_gather_parts(tp, self_rank, c, head, ch, lo, hi, fl)
    if n < 0:
        _check(n)
    return [(ch[i], lo[i], hi[i], bool(fl[i])) for i in range(n)]


def plan_ag_self_head(T: int, tp: int, self_rank: int, n_tiles: int, pairs: int) -> int:
    """Rows of the self chunk the CTA-pair AG kernel reads in place."""
    return _plan_check(load().ub_plan_ag_self_head(T, tp, self_rank, n_tiles, pairs))


def plan_ag_group_m(T: int, tp: int, self_rank: int, n_tiles: int, pairs: int) -> int:
    """Tile rows per group of a CTA-pair AG call's tile order (0: N fastest)."""
    return _plan_check(load().ub_plan_ag_group_m(T, tp, self_rank, n_tiles, pairs))


def _check(rc: int):
    if rc != UB_OK:
        raise UbError(rc, last_error())
    return rc


def validate_active_shape(shape, max_tokens: int, hidden: int, tp: int) -> int:
    """UB_OK or the UB_ERR_* code of the first violated active-shape constraint."""
    dims = (ctypes.c_int64 * max(1, len(shape)))(*[int(d) for d in shape])
    return load().ub_validate_active_shape(len(shape), dims, max_tokens, hidden, tp)


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptrs(tensors):
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def _bf16_cuda(t: torch.Tensor, name: str, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError("%s must be a CUDA bfloat16 tensor, got %s on %s" % (name, t.dtype, t.device))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the user buffer on %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


class _DeviceArray:
    """Exposes the registered buffer to torch through __cuda_array_interface__."""

    def __init__(self, owner, ptr: int, shape):
        self._owner = owner
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": "<i2",
                                         "data": (ptr, False), "version": 3, "strides": None}


class UserBuffer:
    """A user buffer registered at capacity [max_tokens, hidden] for tp virtual ranks."""

    def __init__(self, shape, tp_size: int, dtype=torch.bfloat16):
        if len(shape) != 2:
            raise UbError(CODES["UB_ERR_RANK"], "capacity shape must be [max_tokens, hidden]")
        if dtype != torch.bfloat16:
            raise UbError(CODES["UB_ERR_DTYPE"], "only torch.bfloat16 user buffers are supported")
        L = load()
        h = ctypes.c_void_p()
        _check(L.ub_create(int(shape[0]), int(shape[1]), int(tp_size), 0, ctypes.byref(h)))
        self._h = h
        self.max_tokens, self.hidden, self.tp = int(shape[0]), int(shape[1]), int(tp_size)
        self._active = None
        self.device = torch.device("cuda", torch.cuda.current_device())

    # -- lifetime
    def close(self):
        if getattr(self, "_h", None):
            load().ub_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- shapes
    def set_active_shape(self, shape):
        dims = (ctypes.c_int64 * max(1, len(shape)))(*[int(d) for d in shape])
        _check(load().ub_set_active_shape_nd(self._h, len(shape), dims))
        self._active = (int(shape[0]), int(shape[1]))

    @property
    def active_shape(self):
        """[T, hidden] as last set (kept on this side: every call reads it)."""
        if self._active is None:
            T, H = ctypes.c_int64(), ctypes.c_int64()
            _check(load().ub_get_active_shape(self._h, ctypes.byref(T), ctypes.byref(H)))
            self._active = (T.value, H.value)
        return self._active

    @property
    def capacity_shape(self):
        M, H = ctypes.c_int64(), ctypes.c_int64()
        _check(load().ub_get_capacity(self._h, ctypes.byref(M), ctypes.byref(H)))
        return (M.value, H.value)

    def buffer(self) -> torch.Tensor:
        """The whole registered buffer as a [max_tokens, hidden] bf16 CUDA tensor (a view)."""
        p = ctypes.c_void_p()
        n = ctypes.c_size_t()
        _check(load().ub_buffer(self._h, ctypes.byref(p), ctypes.byref(n)))
        arr = _DeviceArray(self, p.value, (self.max_tokens, self.hidden))
        return torch.as_tensor(arr, device=self.device).view(torch.bfloat16)

    def buffer_ptr(self) -> int:
        p = ctypes.c_void_p()
        _check(load().ub_buffer(self._h, ctypes.byref(p), None))
        return p.value

    # -- options / status
    def set_option(self, key: str, value: int):
        _check(load().ub_set_option(self._h, OPTIONS[key], int(value)))

    def get_option(self, key: str) -> int:
        v = ctypes.c_int64()
        _check(load().ub_get_option(self._h, OPTIONS[key], ctypes.byref(v)))
        return v.value

    def query_status(self) -> int:
        """Sticky device status (UB_OK or UB_ERR_*); synchronise the stream first."""
        return load().ub_query_status(self._h)

    def clear_status(self):
        _check(load().ub_clear_status(self._h))

    def counters(self) -> dict:
        c = Counters()
        _check(load().ub_get_counters(self._h, ctypes.byref(c)))
        return {f: getattr(c, f) for f, _ in Counters._fields_}

    def kernel_time(self, op: str):
        """(total_ms, launches) of the GEMM kernels of ``op`` since the last query
        (needs the ``profile`` option)."""
        ms, n = ctypes.c_double(), ctypes.c_int64()
        _check(load().ub_kernel_time(self._h, OPS[op], ctypes.byref(ms), ctypes.byref(n)))
        return ms.value, n.value

    def grid_ctas(self) -> int:
        g = ctypes.c_int()
        _check(load().ub_grid_ctas(self._h, ctypes.byref(g)))
        return g.value

    # -- the two operations
    def ag_gemm(self, shards, Wt: torch.Tensor, Y: torch.Tensor | None = None, stream=None):
        """Y[T, N] = concat_r(shards[r]) @ Wt.T; the gathered input stays in the buffer."""
        T, H = self.active_shape
        if len(shards) != self.tp:
            raise ValueError("expected %d shards, got %d" % (self.tp, len(shards)))
        c = T // self.tp
        for r, s in enumerate(shards):
            _bf16_cuda(s, "shards[%d]" % r, (c, H), device=self.device)
        _bf16_cuda(Wt, "Wt", device=self.device)
        if Wt.dim() != 2 or Wt.shape[1] != H:
            raise ValueError("Wt must be [N, %d], got %s" % (H, tuple(Wt.shape)))
        N = Wt.shape[0]
        if Y is None:
            Y = torch.empty((T, N), dtype=torch.bfloat16, device=Wt.device)
        _bf16_cuda(Y, "Y", device=self.device)
        if Y.dim() != 2 or Y.shape[0] < T or Y.shape[1] != N:
            raise ValueError("Y must be [>=%d, %d], got %s" % (T, N, tuple(Y.shape)))
        _check(load().ag_gemm(self._h, _ptrs(shards), ctypes.c_void_p(Wt.data_ptr()), N,
                              ctypes.c_void_p(Y.data_ptr()), _stream_ptr(stream)))
        return Y

    def ag_gemm_swiglu(self, shards, Wt: torch.Tensor, Z: torch.Tensor | None = None, stream=None):
        """Z[T, F] = silu(G @ Wt[:F].T) * (G @ Wt[F:].T), G = concat_r(shards[r]); Wt is
        [2F, hidden] with the gate rows first. The gathered input stays in the buffer."""
        T, H = self.active_shape
        if len(shards) != self.tp:
            raise ValueError("expected %d shards, got %d" % (self.tp, len(shards)))
        c = T // self.tp
        for r, s in enumerate(shards):
            _bf16_cuda(s, "shards[%d]" % r, (c, H), device=self.device)
        _bf16_cuda(Wt, "Wt", device=self.device)
        if Wt.dim() != 2 or Wt.shape[1] != H or Wt.shape[0] % 2:
            raise ValueError("Wt must be [2F, %d], got %s" % (H, tuple(Wt.shape)))
        F = Wt.shape[0] // 2
        if Z is None:
            Z = torch.empty((T, F), dtype=torch.bfloat16, device=Wt.device)
        _bf16_cuda(Z, "Z", device=self.device)
        if Z.dim() != 2 or Z.shape[0] < T or Z.shape[1] != F:
            raise ValueError("Z must be [>=%d, %d], got %s" % (T, F, tuple(Z.shape)))
        _check(load().ag_gemm_swiglu(self._h, _ptrs(shards), ctypes.c_void_p(Wt.data_ptr()), F,
                                     ctypes.c_void_p(Z.data_ptr()), _stream_ptr(stream)))
        return Z

    def ag_gemm_kn(self, shards, W: torch.Tensor, Y: torch.Tensor | None = None, stream=None):
        """Y[T, N] = concat_r(shards[r]) @ W with W stored [hidden, N] (e.g. the
        row-parallel input gradient dS @ Bt_j). The gathered input stays in the buffer."""
        T, H = self.active_shape
        if len(shards) != self.tp:
            raise ValueError("expected %d shards, got %d" % (self.tp, len(shards)))
        c = T // self.tp
        for r, s in enumerate(shards):
            _bf16_cuda(s, "shards[%d]" % r, (c, H), device=self.device)
        _bf16_cuda(W, "W", device=self.device)
        if W.dim() != 2 or W.shape[0] != H:
            raise ValueError("W must be [%d, N], got %s" % (H, tuple(W.shape)))
        N = W.shape[1]
        if Y is None:
            Y = torch.empty((T, N), dtype=torch.bfloat16, device=W.device)
        _bf16_cuda(Y, "Y", device=self.device)
        if Y.dim() != 2 or Y.shape[0] < T or Y.shape[1] != N:
            raise ValueError("Y must be [>=%d, %d], got %s" % (T, N, tuple(Y.shape)))
        _check(load().ag_gemm_kn(self._h, _ptrs(shards), ctypes.c_void_p(W.data_ptr()), N,
                                 ctypes.c_void_p(Y.data_ptr()), _stream_ptr(stream)))
        return Y

    def gemm_rs_kn(self, A, B, Y_shards=None, stream=None):
        """Y_shards[r] = rows [r*c, (r+1)*c) of sum_j A[j] @ B[j], B[j] stored [K, hidden]
        (e.g. the column-parallel input gradient sum_j dY_j @ Wt_j)."""
        T, H = self.active_shape
        if len(A) != self.tp or len(B) != self.tp:
            raise ValueError("expected %d A and B operands" % self.tp)
        K = A[0].shape[1] if A[0].dim() == 2 else -1
        for j in range(self.tp):
            _bf16_cuda(A[j], "A[%d]" % j, (T, K), device=self.device)
            _bf16_cuda(B[j], "B[%d]" % j, (K, H), device=self.device)
        c = T // self.tp
        if Y_shards is None:
            Y_shards = [torch.empty((c, H), dtype=torch.bfloat16, device=A[0].device)
                        for _ in range(self.tp)]
        for r, y in enumerate(Y_shards):
            _bf16_cuda(y, "Y_shards[%d]" % r, device=self.device)
            if y.dim() != 2 or y.shape[0] < c or y.shape[1] != H:
                raise ValueError("Y_shards[%d] must be [>=%d, %d]" % (r, c, H))
        _check(load().gemm_rs_kn(self._h, _ptrs(A), _ptrs(B), K, _ptrs(Y_shards),
                                 _stream_ptr(stream)))
        return Y_shards

    def wgrad(self, D: torch.Tensor, ub_is_a: bool = False, out: torch.Tensor | None = None,
              stream=None):
        """Weight gradient over the T active rows of the gathered buffer G:
        ub_is_a=False -> out [M, hidden] = D.T @ G; ub_is_a=True -> out [hidden, M] = G.T @ D."""
        T, H = self.active_shape
        _bf16_cuda(D, "D", device=self.device)
        if D.dim() != 2 or D.shape[0] != T:
            raise ValueError("D must be [%d, M], got %s" % (T, tuple(D.shape)))
        M = D.shape[1]
        shape = (H, M) if ub_is_a else (M, H)
        if out is None:
            out = torch.empty(shape, dtype=torch.bfloat16, device=D.device)
        _bf16_cuda(out, "out", shape, device=self.device)
        _check(load().ub_wgrad(self._h, ctypes.c_void_p(D.data_ptr()), M, int(bool(ub_is_a)),
                               ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)))
        return out

    def ag_gemm_from_buffer(self, Wt: torch.Tensor, Y: torch.Tensor | None = None, swiglu: bool = False,
                            stream=None):
        """Y[T, N] = UB[:T] @ Wt.T over the buffer as it stands (no gather, no flag wait);
        with swiglu, Wt is [2F, hidden] (gate rows first) and Y[T, F] = silu(gate) * up.
        The buffer must already hold the chunks: an allgather() of this active shape on
        this handle, ordered before this call (same stream, or an event)."""
        T, H = self.active_shape
        _bf16_cuda(Wt, "Wt", device=self.device)
        if Wt.dim() != 2 or Wt.shape[1] != H or (swiglu and Wt.shape[0] % 2):
            raise ValueError("Wt must be [%s, %d], got %s" % ("2F" if swiglu else "N", H, tuple(Wt.shape)))
        N = Wt.shape[0]
        n_out = N // 2 if swiglu else N
        if Y is None:
            Y = torch.empty((T, n_out), dtype=torch.bfloat16, device=Wt.device)
        _bf16_cuda(Y, "Y", device=self.device)
        if Y.dim() != 2 or Y.shape[0] < T or Y.shape[1] != n_out:
            raise ValueError("Y must be [>=%d, %d], got %s" % (T, n_out, tuple(Y.shape)))
        _check(load().ag_gemm_from_buffer(self._h, ctypes.c_void_p(Wt.data_ptr()), N, n_out if swiglu else 0,
                                          ctypes.c_void_p(Y.data_ptr()), _stream_ptr(stream)))
        return Y

    def allgather(self, shards, stream=None):
        """Bulk all-gather: UB[r*c + i] = shards[r][i] for the active shape, no GEMM."""
        T, H = self.active_shape
        if len(shards) != self.tp:
            raise ValueError("expected %d shards, got %d" % (self.tp, len(shards)))
        c = T // self.tp
        for r, s in enumerate(shards):
            _bf16_cuda(s, "shards[%d]" % r, (c, H), device=self.device)
        _check(load().ub_allgather(self._h, _ptrs(shards), _stream_ptr(stream)))

    def reduce_scatter(self, P, Y_shards=None, stream=None):
        """Bulk reduce-scatter: Y_shards[r] = rows [r*c, (r+1)*c) of sum_j P[j]."""
        T, H = self.active_shape
        if len(P) != self.tp:
            raise ValueError("expected %d partials" % self.tp)
        for j, x in enumerate(P):
            _bf16_cuda(x, "P[%d]" % j, (T, H), device=self.device)
        c = T // self.tp
        if Y_shards is None:
            Y_shards = [torch.empty((c, H), dtype=torch.bfloat16, device=P[0].device)
                        for _ in range(self.tp)]
        for r, y in enumerate(Y_shards):
            _bf16_cuda(y, "Y_shards[%d]" % r, device=self.device)
            if y.dim() != 2 or y.shape[0] < c or y.shape[1] != H:
                raise ValueError("Y_shards[%d] must be [>=%d, %d]" % (r, c, H))
        _check(load().ub_reduce_scatter(self._h, _ptrs(P), _ptrs(Y_shards), _stream_ptr(stream)))
        return Y_shards

    def stream_read(self, t: torch.Tensor, stream=None):
        """Read the bytes of contiguous CUDA tensor `t` once and discard them (ub_stream_read:
        the cost of one kernel reading them, the floor of a call whose work is that read)."""
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise TypeError("t must be a contiguous CUDA tensor")
        if t.device != self.device:
            raise ValueError("t is on %s, the user buffer on %s" % (t.device, self.device))
        _check(load().ub_stream_read(self._h, ctypes.c_void_p(t.data_ptr()), t.numel() * t.element_size(),
                                     _stream_ptr(stream)))

    def gemm_rs(self, A, Bt, Y_shards=None, stream=None):
        """Y_shards[r] = rows [r*c, (r+1)*c) of sum_j A[j] @ Bt[j].T (c = T / tp)."""
        T, H = self.active_shape
        if len(A) != self.tp or len(Bt) != self.tp:
            raise ValueError("expected %d A and Bt operands" % self.tp)
        K = A[0].shape[1] if A[0].dim() == 2 else -1
        for j in range(self.tp):
            _bf16_cuda(A[j], "A[%d]" % j, (T, K), device=self.device)
            _bf16_cuda(Bt[j], "Bt[%d]" % j, (H, K), device=self.device)
        c = T // self.tp
        if Y_shards is None:
            Y_shards = [torch.empty((c, H), dtype=torch.bfloat16, device=A[0].device)
                        for _ in range(self.tp)]
        if len(Y_shards) != self.tp:
            raise ValueError("expected %d output shards" % self.tp)
        for r, y in enumerate(Y_shards):
            _bf16_cuda(y, "Y_shards[%d]" % r, device=self.device)
            if y.dim() != 2 or y.shape[0] < c or y.shape[1] != H:
                raise ValueError("Y_shards[%d] must be [>=%d, %d]" % (r, c, H))
        _check(load().gemm_rs(self._h, _ptrs(A), _ptrs(Bt), K, _ptrs(Y_shards),
                              _stream_ptr(stream)))
        return Y_shards


def ag_gemm_noalloc(shards, Wt: torch.Tensor, Y: torch.Tensor | None = None, stream=None):
    """AG-GEMM through the allocation-free entry point (no handle): for callers that
    cannot allocate device memory. Uses the library's fixed 32 MiB device scratch, so
    T * hidden <= NOALLOC_MAX_ELEMS, and calls on one device must not overlap.

    The C entry point cannot see tensor sizes (it builds its tensor maps from T, hidden
    and N alone), so every shape and the device of every tensor are checked here, and
    the call runs with the tensors' device current: the library picks that device's
    copy of the scratch and launches there."""
    tp = len(shards)
    if not 1 <= tp <= MAX_TP:
        raise ValueError("expected 1..%d shards, got %d" % (MAX_TP, tp))
    _bf16_cuda(shards[0], "shards[0]")
    if shards[0].dim() != 2:
        raise ValueError("shards[0] must be [c, hidden], got %s" % (tuple(shards[0].shape),))
    c, H = shards[0].shape
    for r, s in enumerate(shards):
        _bf16_cuda(s, "shards[%d]" % r, (c, H))
    _bf16_cuda(Wt, "Wt")
    if Wt.dim() != 2 or Wt.shape[1] != H:
        raise ValueError("Wt must be [N, %d], got %s" % (H, tuple(Wt.shape)))
    N = Wt.shape[0]
    T = c * tp
    device = Wt.device
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.bfloat16, device=device)
    _bf16_cuda(Y, "Y")
    if Y.dim() != 2 or Y.shape[0] < T or Y.shape[1] != N:
        raise ValueError("Y must be [>=%d, %d], got %s" % (T, N, tuple(Y.shape)))
    for name, t in [("shards[%d]" % r, s) for r, s in enumerate(shards)] + [("Y", Y)]:
        if t.device != device:
            raise ValueError("%s is on %s, Wt on %s: all tensors must share one device" % (name, t.device, device))
    with torch.cuda.device(device):
        _check(load().ag_gemm_noalloc(_ptrs(shards), tp, T, H, ctypes.c_void_p(Wt.data_ptr()), N,
                                      ctypes.c_void_p(Y.data_ptr()), _stream_ptr(stream)))
    return Y


# ---------------------------------------------------------------- module-level manager

_default: UserBuffer | None = None


def initialize_ub(shape, tp_size: int, dtype=torch.bfloat16) -> UserBuffer:
    """Register the default user buffer at capacity ``shape`` = [max_tokens, hidden]."""
    global _default
    if _default is not None:
        _default.close()
    _default = UserBuffer(shape, tp_size, dtype)
    return _default


def set_ub_active_shape(shape):
    """Set the active shape [T, hidden] of the default user buffer."""
    if _default is None:
        raise RuntimeError("initialize_ub() has not been called")
    _default.set_active_shape(shape)


def get_ub() -> UserBuffer:
    if _default is None:
        raise RuntimeError("initialize_ub() has not been called")
    return _default


def destroy_ub():
    global _default
    if _default is not None:
        _default.close()
        _default = None
