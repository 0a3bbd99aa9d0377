"""Thin Python binding of liblora.so (include/lora.h): argument marshalling only.

Each function has the name of the C entry point it calls and takes torch
tensors that already live on the GPU; it reads their pointers, shapes and
strides, allocates the workspace the C side asks for (torch caching allocator)
and passes the current CUDA stream.  All arithmetic runs in the library's
CUDA kernels.  There is no fallback: if liblora.so has not been built, or a
call fails, an exception is raised.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liblora.so")

LORA_F32, LORA_BF16 = 0, 1
OP_FORWARD, OP_BACKWARD_DX_DA, OP_BACKWARD_DB, OP_GROUP_BY_SLOT = 0, 1, 2, 3
OP_SHRINK, OP_EXPAND, OP_APPLY_LINEAR, OP_GATHER_SHRINK = 4, 5, 6, 7
OP_BACKWARD = 8
BWD_DX_ACCUMULATE, BWD_GRAD_INPUT_DTYPE = 1, 2   # lora_backward_ex flags
STATUS = {0: "LORA_OK", 1: "LORA_ERR_INVALID_ARG", 2: "LORA_ERR_UNSUPPORTED", 3: "LORA_ERR_ALIGNMENT",
          4: "LORA_ERR_WORKSPACE", 5: "LORA_ERR_CUDA", 6: "LORA_ERR_DEVICE"}
EXPORTS = ["lora_workspace_size", "lora_forward", "lora_backward_dx_da", "lora_backward_db",
           "lora_group_by_slot", "lora_shrink", "lora_expand", "lora_apply_linear",
           "lora_gather_shrink", "lora_status_string", "lora_device_error", "lora_kernel_launches",
           "lora_version", "lora_backward_db_noalloc", "lora_forward_h", "lora_backward", "lora_backward_ex",
           "lora_schedule_size", "lora_build_schedule"]


class LoraError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn} failed: {text}")
        self.status = status


class LoraAddressing(ctypes.Structure):
    """lora_addressing_t: device slots pointer, the sizes T, S, R, and an optional
    prebuilt schedule (device pointer, or 0)."""
    _fields_ = [("slots", ctypes.c_void_p), ("num_tokens", ctypes.c_int32),
                ("num_slots", ctypes.c_int32), ("max_rank", ctypes.c_int32),
                ("schedule", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded liblora.so with its C signatures (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with lora_rank_adapter_gb300._build.build() "
                          "(nvcc, sm_103a); there is no CPU fallback")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, f32, P, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    AP = ctypes.POINTER(LoraAddressing)
    sig = {
        "lora_workspace_size": (sz, [i32, i32, i64, i64, i64, i32, i32]),
        "lora_forward": (i32, [i32, i64, i64, i64, i32, P, i64, P, i64, i64, P, i64, i64, P, i64, f32,
                               P, sz, P]),
        "lora_backward_dx_da": (i32, [i32, i64, i64, i64, i32, P, i64, P, i64, P, i64, i64, P, i64, i64,
                                      f32, P, i64, P, i64, i64, P, sz, P]),
        "lora_backward_db": (i32, [i32, i64, i64, i64, i32, P, i64, P, i64, i64, P, i64, f32, P, i64, i64,
                                   P, sz, P]),
        "lora_forward_h": (i32, [i32, i64, i64, i64, i32, P, i64, P, i64, i64, P, i64, i64, P, i64, f32,
                                 P, i64, P, sz, P]),
        "lora_backward": (i32, [i32, i64, i64, i64, i32, P, i64, P, i64, P, i64, i64, P, i64, i64, P, i64,
                                f32, P, i64, P, i64, i64, P, i64, i64, P, sz, P]),
        "lora_backward_ex": (i32, [i32, i64, i64, i64, i32, P, i64, P, i64, P, i64, i64, P, i64, i64, P, i64,
                                   f32, P, i64, P, i64, i64, P, i64, i64, ctypes.c_uint32, P, sz, P]),
        "lora_group_by_slot": (i32, [AP, P, P, P, P, P, sz, P]),
        "lora_schedule_size": (sz, [i32, i32]),
        "lora_build_schedule": (i32, [AP, P, P, sz, P]),
        "lora_shrink": (i32, [AP, P, i64, i32, P, i64, P, i64, i64, P, i64, P, sz, P]),
        "lora_expand": (i32, [AP, P, P, P, i32, P, i64, P, i64, i64, i64, P, i64, P, sz, P]),
        "lora_apply_linear": (i32, [AP, P, P, P, i32, i64, P, i64, P, i64, i64, P, i64, i64, i64, P, i64,
                                    P, sz, P]),
        "lora_gather_shrink": (i32, [AP, P, i64, P, P, i64, i64, i64, P, i64, P]),
        "lora_status_string": (ctypes.c_char_p, [i32]),
        "lora_device_error": (i32, [ctypes.POINTER(i32)]),
        "lora_kernel_launches": (ctypes.c_uint64, []),
        "lora_backward_db_noalloc": (i32, [i32, i64, i64, i64, i32, P, i64, P, i64, i64, P, i64, f32, P, i64, i64,
                                           P]),
        "lora_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status, fn):
    if status != 0:
        raise LoraError(fn, status, lib().lora_status_string(status).decode())


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return LORA_BF16
    if t.dtype == torch.float32:
        return LORA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None and t.numel() > 0 else 0)


def workspace(op, dtype, m_or_t, k_or_in, l_or_o, r_or_R, num_slots=0, device="cuda"):
    """A uint8 workspace tensor of lora_workspace_size() bytes (None when zero)."""
    n = lib().lora_workspace_size(op, dtype, m_or_t, k_or_in, l_or_o, r_or_R, num_slots)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def _ws_args(ws):
    return (_ptr(ws), ws.numel() if ws is not None else 0)


# ----------------------------------------------------------------------------- single adapter
def lora_forward(X, A, B, Y, scale, ws=None, stream=None):
    """Y += scale * (X @ A) @ B in place.  X [M,K], A [K,r], B [r,L], Y [M,L]."""
    M, K = X.shape
    r, L = B.shape
    assert A.shape == (K, r) and Y.shape == (M, L)
    dt = _dtype(X)
    if ws is None:
        ws = workspace(OP_FORWARD, dt, M, K, L, r, device=X.device)
    st = lib().lora_forward(dt, M, K, L, r, _ptr(X), X.stride(0), _ptr(A), A.stride(0), A.stride(1),
                            _ptr(B), B.stride(0), B.stride(1), _ptr(Y), Y.stride(0), float(scale),
                            *_ws_args(ws), _stream(stream))
    _check(st, "lora_forward")
    return Y


def lora_forward_h(X, A, B, Y, scale, h, ws=None, stream=None):
    """Y += scale * (X @ A) @ B in place, and h = X @ A (fp32 [M, r]) for lora_backward."""
    M, K = X.shape
    r, L = B.shape
    assert A.shape == (K, r) and Y.shape == (M, L) and h.shape == (M, r) and h.dtype == torch.float32
    assert h.stride(1) == 1
    dt = _dtype(X)
    if ws is None:
        ws = workspace(OP_FORWARD, dt, M, K, L, r, device=X.device)
    st = lib().lora_forward_h(dt, M, K, L, r, _ptr(X), X.stride(0), _ptr(A), A.stride(0), A.stride(1),
                              _ptr(B), B.stride(0), B.stride(1), _ptr(Y), Y.stride(0), float(scale),
                              _ptr(h), h.stride(0), *_ws_args(ws), _stream(stream))
    _check(st, "lora_forward_h")
    return Y, h


def lora_backward(X, dY, A, B, h, scale, dX, dA, dB, ws=None, stream=None):
    """dX, dA and dB in one call from the h that lora_forward_h saved (dA, dB fp32)."""
    M, K = X.shape
    r, L = B.shape
    assert dY.shape == (M, L) and A.shape == (K, r) and dX.shape == (M, K) and dA.shape == (K, r)
    assert dB.shape == (r, L) and h.shape == (M, r) and h.stride(1) == 1
    assert dA.dtype == torch.float32 and dB.dtype == torch.float32 and h.dtype == torch.float32
    dt = _dtype(X)
    if ws is None:
        ws = workspace(OP_BACKWARD, dt, M, K, L, r, device=X.device)
    st = lib().lora_backward(dt, M, K, L, r, _ptr(X), X.stride(0), _ptr(dY), dY.stride(0),
                             _ptr(A), A.stride(0), A.stride(1), _ptr(B), B.stride(0), B.stride(1),
                             _ptr(h), h.stride(0), float(scale), _ptr(dX), dX.stride(0),
                             _ptr(dA), dA.stride(0), dA.stride(1), _ptr(dB), dB.stride(0), dB.stride(1),
                             *_ws_args(ws), _stream(stream))
    _check(st, "lora_backward")
    return dX, dA, dB


def lora_backward_ex(X, dY, A, B, h, scale, dX, dA, dB, flags=0, ws=None, stream=None):
    """lora_backward with output options: flags BWD_DX_ACCUMULATE (dX += the
    update) and BWD_GRAD_INPUT_DTYPE (dA, dB in X's dtype instead of fp32)."""
    M, K = X.shape
    r, L = B.shape
    assert dY.shape == (M, L) and A.shape == (K, r) and dX.shape == (M, K) and dA.shape == (K, r)
    assert dB.shape == (r, L) and h.shape == (M, r) and h.stride(1) == 1 and h.dtype == torch.float32
    gdt = X.dtype if flags & BWD_GRAD_INPUT_DTYPE else torch.float32
    assert dA.dtype == gdt and dB.dtype == gdt, (dA.dtype, dB.dtype, gdt)
    dt = _dtype(X)
    if ws is None:
        ws = workspace(OP_BACKWARD, dt, M, K, L, r, device=X.device)
    st = lib().lora_backward_ex(dt, M, K, L, r, _ptr(X), X.stride(0), _ptr(dY), dY.stride(0),
                                _ptr(A), A.stride(0), A.stride(1), _ptr(B), B.stride(0), B.stride(1),
                                _ptr(h), h.stride(0), float(scale), _ptr(dX), dX.stride(0),
                                _ptr(dA), dA.stride(0), dA.stride(1), _ptr(dB), dB.stride(0), dB.stride(1),
                                int(flags), *_ws_args(ws), _stream(stream))
    _check(st, "lora_backward_ex")
    return dX, dA, dB


def lora_backward_dx_da(X, dY, A, B, scale, dX, dA, ws=None, stream=None):
    """dX = scale * dY @ B^T @ A^T and dA = scale * X^T @ (dY @ B^T) (dA fp32)."""
    M, K = X.shape
    r, L = B.shape
    assert dY.shape == (M, L) and A.shape == (K, r) and dX.shape == (M, K) and dA.shape == (K, r)
    assert dA.dtype == torch.float32
    dt = _dtype(X)
    if ws is None:
        ws = workspace(OP_BACKWARD_DX_DA, dt, M, K, L, r, device=X.device)
    st = lib().lora_backward_dx_da(dt, M, K, L, r, _ptr(X), X.stride(0), _ptr(dY), dY.stride(0),
                                   _ptr(A), A.stride(0), A.stride(1), _ptr(B), B.stride(0), B.stride(1),
                                   float(scale), _ptr(dX), dX.stride(0), _ptr(dA), dA.stride(0),
                                   dA.stride(1), *_ws_args(ws), _stream(stream))
    _check(st, "lora_backward_dx_da")
    return dX, dA


def lora_backward_db(X, A, dY, scale, dB, ws=None, stream=None):
    """dB = scale * (X @ A)^T @ dY (dB fp32)."""
    M, K = X.shape
    r = A.shape[1]
    L = dY.shape[1]
    assert A.shape == (K, r) and dY.shape == (M, L) and dB.shape == (r, L)
    assert dB.dtype == torch.float32
    dt = _dtype(X)
    if ws is None:
        ws = workspace(OP_BACKWARD_DB, dt, M, K, L, r, device=X.device)
    st = lib().lora_backward_db(dt, M, K, L, r, _ptr(X), X.stride(0), _ptr(A), A.stride(0), A.stride(1),
                                _ptr(dY), dY.stride(0), float(scale), _ptr(dB), dB.stride(0), dB.stride(1),
                                *_ws_args(ws), _stream(stream))
    _check(st, "lora_backward_db")
    return dB


# ----------------------------------------------------------------------------- multi adapter
def _addr(slots, S, R, schedule=None):
    assert slots.dtype == torch.int32
    return LoraAddressing(slots.data_ptr() if slots.numel() else 0, slots.numel(), S, R,
                          schedule.data_ptr() if schedule is not None and schedule.numel() else 0)


def lora_build_schedule(slots, ranks, R, stream=None):
    """The grouping of a batch's tokens by slot, built once on the device (a
    uint8 tensor) for the shrink / expand / apply_linear calls of that batch."""
    S, T = ranks.numel(), slots.numel()
    n = lib().lora_schedule_size(T, S)
    sched = torch.empty(max(n, 1), dtype=torch.uint8, device=slots.device)
    ad = _addr(slots, S, R)
    _check(lib().lora_build_schedule(ctypes.byref(ad), _ptr(ranks), _ptr(sched), sched.numel(), _stream(stream)),
           "lora_build_schedule")
    return sched


def lora_group_by_slot(slots, ranks, R, counts, perm, num_active, ws=None, stream=None):
    S = ranks.numel()
    T = slots.numel()
    if ws is None:
        ws = workspace(OP_GROUP_BY_SLOT, LORA_BF16, T, 0, 0, R, S, device=slots.device)
    ad = _addr(slots, S, R)
    st = lib().lora_group_by_slot(ctypes.byref(ad), _ptr(ranks), _ptr(counts), _ptr(perm), _ptr(num_active),
                                  *_ws_args(ws), _stream(stream))
    _check(st, "lora_group_by_slot")


def lora_shrink(x, a, slots, ranks, R, h, num_slices=1, ws=None, stream=None, schedule=None):
    """h[t, i*R + j] = x[t] . a[slot(t), i*R + j] for j < rank (h fp32 [T, n*R])."""
    T, IN = x.shape
    S = ranks.numel()
    assert a.dim() == 3 and a.shape[0] == S and a.shape[1] == num_slices * R and a.shape[2] == IN
    assert a.stride(2) == 1
    if ws is None:
        ws = workspace(OP_SHRINK, LORA_BF16, T, IN, num_slices * R, R, S, device=x.device)
    ad = _addr(slots, S, R, schedule)
    st = lib().lora_shrink(ctypes.byref(ad), _ptr(ranks), IN, num_slices, _ptr(x), x.stride(0), _ptr(a),
                           a.stride(0), a.stride(1), _ptr(h), h.stride(0), *_ws_args(ws), _stream(stream))
    _check(st, "lora_shrink")
    return h


def _slices(out_slices):
    n = len(out_slices)
    return (ctypes.c_int32 * n)(*[int(v) for v in out_slices]), n


def lora_expand(h, b, slots, ranks, scalings, y, out_slices, R, ws=None, stream=None, schedule=None):
    """y[t, slice i] += scalings[slot] * h[t, slice i] @ b[slot, slice i]^T (b [S, O, R])."""
    T = y.shape[0]
    S = ranks.numel()
    osl, n = _slices(out_slices)
    O = sum(int(v) for v in out_slices)
    assert b.dim() == 3 and b.shape[0] == S and b.shape[1] == O and b.shape[2] == R
    if ws is None:
        ws = workspace(OP_EXPAND, LORA_BF16, T, 0, O, R, S, device=y.device)
    ad = _addr(slots, S, R, schedule)
    st = lib().lora_expand(ctypes.byref(ad), _ptr(ranks), _ptr(scalings), osl, n, _ptr(h), h.stride(0),
                           _ptr(b), b.stride(0), b.stride(1), b.stride(2), _ptr(y), y.stride(0),
                           *_ws_args(ws), _stream(stream))
    _check(st, "lora_expand")
    return y


def lora_apply_linear(x, a, b, slots, ranks, scalings, y, out_slices, R, ws=None, stream=None, schedule=None):
    """Fused shrink + expand into y."""
    T, IN = x.shape
    S = ranks.numel()
    osl, n = _slices(out_slices)
    O = sum(int(v) for v in out_slices)
    assert a.dim() == 3 and a.shape == (S, n * R, IN) and a.stride(2) == 1
    assert b.dim() == 3 and b.shape[0] == S and b.shape[1] == O and b.shape[2] == R
    if ws is None:
        ws = workspace(OP_APPLY_LINEAR, LORA_BF16, T, IN, O, R, S, device=x.device)
    ad = _addr(slots, S, R, schedule)
    st = lib().lora_apply_linear(ctypes.byref(ad), _ptr(ranks), _ptr(scalings), osl, n, IN, _ptr(x),
                                 x.stride(0), _ptr(a), a.stride(0), a.stride(1), _ptr(b), b.stride(0),
                                 b.stride(1), b.stride(2), _ptr(y), y.stride(0), *_ws_args(ws),
                                 _stream(stream))
    _check(st, "lora_apply_linear")
    return y


def lora_gather_shrink(ids, a, slots, ranks, R, h, stream=None):
    """h[t, j] = a[slot(t), j, ids[t]] for j < rank (zeros for ids outside [0, V))."""
    S, RR, V = a.shape
    assert RR == R and ids.dtype == torch.int64
    ad = _addr(slots, S, R)
    st = lib().lora_gather_shrink(ctypes.byref(ad), _ptr(ranks), V, _ptr(ids), _ptr(a), a.stride(0),
                                  a.stride(1), a.stride(2), _ptr(h), h.stride(0), _stream(stream))
    _check(st, "lora_gather_shrink")
    return h


def lora_device_error():
    """Reads and clears the device error word (a sync; diagnostics only)."""
    v = ctypes.c_int32(0)
    _check(lib().lora_device_error(ctypes.byref(v)), "lora_device_error")
    return v.value


def lora_kernel_launches():
    """Kernels launched by liblora.so in this process so far."""
    return int(lib().lora_kernel_launches())


def lora_version():
    return lib().lora_version().decode()
