"""ctypes front end of the fp64 oracle (oracle/lora_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by
bench.py's CPU-baseline leg.  The product path (lora_rank_adapter_gb300) never
imports this module.

Every function takes and returns dense row-major numpy float64 arrays that hold
the exact values of the inputs (bf16/fp32 inputs widened without rounding).
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liblora_oracle.so")

_lib = None


def build(force=False, src=_SRC, out=_LIB_PATH):
    """Compile the oracle with gcc (portable C, OpenMP); returns the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path=None):
    """Load (building first if needed) and return a ctypes handle."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    p = path or build()
    lib = ctypes.CDLL(p)
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
    P = ctypes.c_void_p
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_lora_forward.argtypes = [i64, i64, i64, i64, P, P, P, P, dbl, P]
    lib.oracle_lora_backward_dx_da.argtypes = [i64, i64, i64, i64, P, P, P, P, dbl, P, P]
    lib.oracle_lora_backward_db.argtypes = [i64, i64, i64, i64, P, P, P, dbl, P]
    lib.oracle_lora_group_by_slot.argtypes = [i64, i32, i32, P, P, P, P]
    lib.oracle_lora_group_by_slot.restype = i64
    lib.oracle_lora_shrink.argtypes = [i64, i64, i32, i32, i32, P, P, P, P, P]
    lib.oracle_lora_expand.argtypes = [i64, i32, i32, i32, P, P, P, P, P, P, P, P]
    lib.oracle_lora_apply_linear.argtypes = [i64, i64, i32, i32, i32, P, P, P, P, P, P, P, P, P]
    lib.oracle_lora_gather_shrink.argtypes = [i64, i64, i32, i32, P, P, P, P, P]
    if path is None:
        _lib = lib
    return lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads(lib=None):
    return (lib or load()).oracle_num_threads()


def set_num_threads(n, lib=None):
    (lib or load()).oracle_set_num_threads(int(n))


def forward(X, A, B, Y0, s, lib=None):
    X, A, B, Y0 = _f64(X), _f64(A), _f64(B), _f64(Y0)
    M, K = X.shape
    r, L = B.shape
    assert A.shape == (K, r) and Y0.shape == (M, L)
    Y = np.empty((M, L), np.float64)
    (lib or load()).oracle_lora_forward(M, K, L, r, _p(X), _p(A), _p(B), _p(Y0), float(s), _p(Y))
    return Y


def backward_dx_da(X, dY, A, B, s, lib=None):
    X, dY, A, B = _f64(X), _f64(dY), _f64(A), _f64(B)
    M, K = X.shape
    r, L = B.shape
    assert A.shape == (K, r) and dY.shape == (M, L)
    dX = np.empty((M, K), np.float64)
    dA = np.empty((K, r), np.float64)
    (lib or load()).oracle_lora_backward_dx_da(M, K, L, r, _p(X), _p(dY), _p(A), _p(B),
                                               float(s), _p(dX), _p(dA))
    return dX, dA


def backward_db(X, A, dY, s, lib=None):
    X, A, dY = _f64(X), _f64(A), _f64(dY)
    M, K = X.shape
    r = A.shape[1]
    L = dY.shape[1]
    assert A.shape == (K, r) and dY.shape[0] == M
    dB = np.empty((r, L), np.float64)
    (lib or load()).oracle_lora_backward_db(M, K, L, r, _p(X), _p(A), _p(dY), float(s), _p(dB))
    return dB


def backward_ex(X, dY, A, B, s, dX0=None, lib=None):
    """The backward with its output options ([NeMo lora_kernel] update wrappers,
    whose `dtype` picks the gradients' type; an accumulating dX): returns
    (dX0 + s*dY B^T A^T, or that update alone when dX0 is None), dA and dB in
    fp64.  The gradients' storage type is the caller's rounding, not the oracle's."""
    dX, dA = backward_dx_da(X, dY, A, B, s, lib)
    dB = backward_db(X, A, dY, s, lib)
    if dX0 is not None:
        dX = _f64(dX0) + dX
    return dX, dA, dB


def group_by_slot(slots, ranks, R, lib=None):
    slots, ranks = _i32(slots), _i32(ranks)
    T, S = slots.shape[0], ranks.shape[0]
    counts = np.empty(S, np.int32)
    perm = np.full(max(T, 1), -1, np.int32)
    n = (lib or load()).oracle_lora_group_by_slot(T, S, int(R), _p(slots), _p(ranks),
                                                  _p(counts), _p(perm))
    return counts, perm[:n].copy()


def shrink(x, a, slots, ranks, R, num_slices=1, lib=None):
    x, a, slots, ranks = _f64(x), _f64(a), _i32(slots), _i32(ranks)
    T, IN = x.shape
    S = ranks.shape[0]
    assert a.shape == (S, num_slices * R, IN)
    h = np.empty((T, num_slices * R), np.float64)
    (lib or load()).oracle_lora_shrink(T, IN, S, int(R), int(num_slices), _p(slots), _p(ranks),
                                       _p(x), _p(a), _p(h))
    return h


def expand(h, b, slots, ranks, scalings, Y0, out_slices, R, lib=None):
    h, b, Y0 = _f64(h), _f64(b), _f64(Y0)
    slots, ranks, scal = _i32(slots), _i32(ranks), _f64(scalings)
    osl = _i32(out_slices)
    n = osl.shape[0]
    T = h.shape[0]
    S = ranks.shape[0]
    O = int(osl.sum())
    assert h.shape == (T, n * R) and b.shape == (S, O, R) and Y0.shape == (T, O)
    Y = np.empty((T, O), np.float64)
    (lib or load()).oracle_lora_expand(T, S, int(R), n, _p(osl), _p(slots), _p(ranks), _p(scal),
                                       _p(h), _p(b), _p(Y0), _p(Y))
    return Y


def apply_linear(x, a, b, slots, ranks, scalings, Y0, out_slices, R, lib=None):
    x, a, b, Y0 = _f64(x), _f64(a), _f64(b), _f64(Y0)
    slots, ranks, scal = _i32(slots), _i32(ranks), _f64(scalings)
    osl = _i32(out_slices)
    n = osl.shape[0]
    T, IN = x.shape
    S = ranks.shape[0]
    O = int(osl.sum())
    assert a.shape == (S, n * R, IN) and b.shape == (S, O, R) and Y0.shape == (T, O)
    Y = np.empty((T, O), np.float64)
    (lib or load()).oracle_lora_apply_linear(T, IN, S, int(R), n, _p(osl), _p(slots), _p(ranks),
                                             _p(scal), _p(x), _p(a), _p(b), _p(Y0), _p(Y))
    return Y


def gather_shrink(ids, a, slots, ranks, R, lib=None):
    a, slots, ranks = _f64(a), _i32(slots), _i32(ranks)
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    T = slots.shape[0]
    S, RR, V = a.shape
    assert RR == R and ids.shape == (T,)
    h = np.empty((T, R), np.float64)
    (lib or load()).oracle_lora_gather_shrink(T, V, S, int(R), _p(slots), _p(ranks), _p(ids),
                                              _p(a), _p(h))
    return h
