"""CPU oracle for the active-shape AG-GEMM and GEMM-RS (test infrastructure only).

This package is the checker, not the product: only ``tests/``, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``
may import it. The GPU library never loads it and shares no code with it.

What it computes (fp64 accumulation of exactly widened bf16 inputs):

* ``allgather`` -- the concatenation of the tp token shards into rows
  ``[r*c, (r+1)*c)`` of a capacity buffer, ``c = T // tp``; rows ``>= T`` untouched.
  Source: "Support dynamic token counts in TP communication/GEMM overlap"
  (TransformerEngine issue #3564), "Implementation approach in the prototype" --
  active data is a contiguous prefix; chunk offsets come from the active first
  dimension.
* ``ag_gemm`` -- ``Y = concat_r(X_r) @ Wt.T`` (the column-parallel linear of the QKV /
  fc1 diagrams in "Do tp overlap support thd..." (Megatron-LM discussion #1240)).
* ``gemm_rs`` -- ``S = sum_j A_j @ Bt_j.T`` and ``Y_r = S[r*c:(r+1)*c]`` (the
  row-parallel linear of the MLP diagram on the same page: partial products summed
  over ranks, output split by rows).
* ``check_active_shape`` -- the five constraints of issue #3564, "Constrain the initial
  behavior".
* ``gemm_xw_rows`` / ``gemm_tn`` -- the weight in its K x N layout, and the
  contraction over the T active tokens: the products of the backward pass (input and
  weight gradients of both layers).
* ``reduce_scatter`` -- the "bulk" method's independent reduce-scatter of tp partial
  results ("How to setup TP Overlap configs", option "method": "bulk").
* ``swiglu`` -- the activation between fc1 and fc2 (the GELU/SwiGLU box of the MLP
  diagram in discussion #1240): fc1's row is [gate | up] and ``Z = silu(gate) * up``.

Weights are stored out x in (PyTorch ``nn.Linear`` layout): ``Wt`` is ``[N, H]``,
``Bt_j`` is ``[H, K]``. bf16 tensors cross the boundary as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (plain gcc, OpenMP, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_chunk_rows.restype = I64
        lib.oracle_chunk_rows.argtypes = [I64, ctypes.c_int]
        lib.oracle_chunk_offset.restype = I64
        lib.oracle_chunk_offset.argtypes = [I64, ctypes.c_int, ctypes.c_int]
        lib.oracle_allgather.argtypes = [ctypes.c_int, I64, I64, P, P]
        lib.oracle_gemm_xwt_rows.argtypes = [P, I64, P, I64, I64, P, I64, P]
        lib.oracle_ag_gemm.argtypes = [ctypes.c_int, I64, I64, I64, P, P, P, P]
        lib.oracle_gemm_rs.argtypes = [ctypes.c_int, I64, I64, I64, P, P, P, P]
        lib.oracle_gemm_rs_rows.argtypes = [ctypes.c_int, I64, I64, I64, P, P, P, I64,
                                            P, P, P]
        lib.oracle_gemm_xw_rows.argtypes = [P, I64, P, I64, I64, P, I64, P]
        lib.oracle_gemm_tn.argtypes = [P, I64, P, I64, I64, P]
        lib.oracle_reduce_scatter.argtypes = [ctypes.c_int, I64, I64, P, P]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_swiglu.argtypes = [P, I64, I64, P]
        lib.oracle_check_active_shape.restype = ctypes.c_int
        lib.oracle_check_active_shape.argtypes = [ctypes.c_int, I64, I64, I64, I64,
                                                  ctypes.c_int]
        _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle takes bf16 bit patterns as uint16, got %s" % a.dtype)
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return _load().oracle_threads()


def round_bf16(v: float) -> int:
    """Nearest bf16 bit pattern of a double, ties to even."""
    return int(_load().oracle_round_bf16(float(v)))


def chunk_rows(T: int, tp: int) -> int:
    return int(_load().oracle_chunk_rows(T, tp))


def chunk_offset(T: int, tp: int, r: int) -> int:
    return int(_load().oracle_chunk_offset(T, tp, r))


def check_active_shape(shape, cap_tokens: int, cap_hidden: int, tp: int) -> int:
    """0 if ``shape`` is an acceptable active shape, else the 1-based index of the
    first violated constraint (2-D, nonzero, <= capacity, hidden unchanged, T % tp)."""
    shape = list(shape)
    T = int(shape[0]) if len(shape) > 0 else 0
    hidden = int(shape[1]) if len(shape) > 1 else 0
    return int(_load().oracle_check_active_shape(len(shape), T, hidden, cap_tokens,
                                                 cap_hidden, tp))


def allgather(shards, G: np.ndarray, T: int) -> np.ndarray:
    """Write the shards into the capacity buffer G (in place) and return G."""
    shards = [_u16(s) for s in shards]
    tp = len(shards)
    H = G.shape[1]
    assert G.dtype == np.uint16 and G.flags.c_contiguous and G.shape[0] >= T
    for s in shards:
        assert s.shape == (T // tp, H)
    _load().oracle_allgather(tp, T, H, _ptr_array(shards), _ptr(G))
    return G


def ag_gemm(shards, Wt, G: np.ndarray | None = None, T: int | None = None):
    """Return (G, Y): the gathered capacity buffer and Y = G[:T] @ Wt.T in fp64."""
    shards = [_u16(s) for s in shards]
    Wt = _u16(Wt)
    tp = len(shards)
    c, H = shards[0].shape
    if T is None:
        T = c * tp
    if G is None:
        G = np.full((T, H), 0xFFFF, dtype=np.uint16)
    N = Wt.shape[0]
    assert Wt.shape == (N, H)
    Y = np.empty((T, N), dtype=np.float64)
    _load().oracle_ag_gemm(tp, T, H, N, _ptr_array(shards), _ptr(Wt), _ptr(G), _ptr(Y))
    return G, Y


def gemm_rows(X, Wt, rows):
    """Y[q] = X[rows[q]] @ Wt.T in fp64, for selected rows of X."""
    X = _u16(X)
    Wt = _u16(Wt)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    N, K = Wt.shape
    assert X.shape[1] == K
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < X.shape[0])
    Y = np.empty((rows.size, N), dtype=np.float64)
    _load().oracle_gemm_xwt_rows(_ptr(X), X.shape[1], _ptr(Wt), N, K, _ptr(rows),
                                 rows.size, _ptr(Y))
    return Y


def gemm_rs(A, Bt, with_S: bool = True):
    """Return (S, [Y_r]): S = sum_j A_j @ Bt_j.T (fp64) and its tp row blocks."""
    A = [_u16(a) for a in A]
    Bt = [_u16(b) for b in Bt]
    tp = len(A)
    T, K = A[0].shape
    H = Bt[0].shape[0]
    for a in A:
        assert a.shape == (T, K)
    for b in Bt:
        assert b.shape == (H, K)
    assert T % tp == 0
    c = T // tp
    S = np.empty((T, H), dtype=np.float64) if with_S else None
    Y = [np.empty((c, H), dtype=np.float64) for _ in range(tp)]
    yptrs = (ctypes.c_void_p * tp)(*[_ptr(y) for y in Y])
    _load().oracle_gemm_rs(tp, T, K, H, _ptr_array(A), _ptr_array(Bt),
                           _ptr(S) if S is not None else None, yptrs)
    return S, Y


def gemm_rs_rows(A_rows, Bt, rows, T: int):
    """For selected active rows t = rows[q] of a T-token GEMM-RS: (S[t], owner rank
    t // c, local row t - owner*c). ``A_rows[j]`` holds only the selected rows of A_j
    (``A_rows[j][q] = A_j[rows[q]]``), so full-size checks need not copy all of A_j."""
    A_rows = [_u16(a) for a in A_rows]
    Bt = [_u16(b) for b in Bt]
    tp = len(A_rows)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    K = Bt[0].shape[1]
    H = Bt[0].shape[0]
    for a in A_rows:
        assert a.shape == (rows.size, K)
    assert T % tp == 0
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < T)
    out = np.empty((rows.size, H), dtype=np.float64)
    owner = np.empty(rows.size, dtype=np.int32)
    local = np.empty(rows.size, dtype=np.int64)
    _load().oracle_gemm_rs_rows(tp, T, K, H, _ptr_array(A_rows), _ptr_array(Bt), _ptr(rows),
                                rows.size, _ptr(out), _ptr(owner), _ptr(local))
    return out, owner, local


def silu(x: float) -> float:
    """x / (1 + exp(-x)) in double."""
    return float(_load().oracle_silu(float(x)))


def swiglu(Y: np.ndarray) -> np.ndarray:
    """Z = silu(Y[:, :F]) * Y[:, F:] for fp64 rows Y = [gate | up] of width 2F."""
    Y = np.ascontiguousarray(Y, dtype=np.float64)
    rows, two_f = Y.shape
    assert two_f % 2 == 0
    F = two_f // 2
    Z = np.empty((rows, F), dtype=np.float64)
    _load().oracle_swiglu(_ptr(Y), rows, F, _ptr(Z))
    return Z


def gemm_xw_rows(X, W, rows):
    """Y[q] = X[rows[q]] @ W in fp64, W stored K x N row-major."""
    X = _u16(X)
    W = _u16(W)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    K, N = W.shape
    assert X.shape[1] == K
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < X.shape[0])
    Y = np.empty((rows.size, N), dtype=np.float64)
    _load().oracle_gemm_xw_rows(_ptr(X), X.shape[1], _ptr(W), N, K, _ptr(rows), rows.size, _ptr(Y))
    return Y


def gemm_tn(D, G):
    """out = D.T @ G in fp64 for D [T, M], G [T, N] (the sum runs over the T rows)."""
    D = _u16(D)
    G = _u16(G)
    T, M = D.shape
    assert G.shape[0] == T
    N = G.shape[1]
    out = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_tn(_ptr(D), M, _ptr(G), N, T, _ptr(out))
    return out


def reduce_scatter(P):
    """[Y_r]: rank r's row block of sum_j P[j] (fp64), P[j] [T, H] bf16 bit patterns."""
    P = [_u16(a) for a in P]
    tp = len(P)
    T, H = P[0].shape
    for a in P:
        assert a.shape == (T, H)
    assert T % tp == 0
    c = T // tp
    Y = [np.empty((c, H), dtype=np.float64) for _ in range(tp)]
    yptrs = (ctypes.c_void_p * tp)(*[_ptr(y) for y in Y])
    _load().oracle_reduce_scatter(tp, T, H, _ptr_array(P), yptrs)
    return Y
