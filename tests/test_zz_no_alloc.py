"""lora_backward_db_noalloc, the dB backward for callers that cannot allocate
device memory: code running inside another engine's memory pool, or a plugin
that is handed tensors but no allocator, or a hot path that cannot take
cudaMalloc's implicit device synchronisation.  It uses the library's own
static scratch array instead of a caller workspace.

Called through the C ABI: its dB must match both the fp64 oracle and
lora_backward_db (the same op on a caller workspace) within the fp32
tolerance of the suite, on calls in a row that reuse the array the previous
call left behind, in bf16 and fp32, including a large call, then a small one,
then a large one again (leftover counters or partial sums of a bigger call must
not leak into a smaller one).  dB is filled with NaN before every call, so a
column the call fails to write shows up.  This file is collected last on
purpose, and each test also passes when run alone in a fresh process."""
import ctypes

import pytest
import torch

from lora_rank_adapter_gb300 import _build
from lora_rank_adapter_gb300 import binding
from lora_rank_adapter_gb300 import synth
from oracle import oracle as O
from tests._util import TOL_F32, f64, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def _inputs(name, M, K, L, r, seed, mode):
    spec = synth.single_spec(name, M=M, K=K, L=L, r=r)
    w = synth.make_single(spec, seed=seed, device=DEV, prefix=f"noalloc{seed}")
    A = w["A"]
    if mode == "peft":
        A = A.t().contiguous().t()        # lora_A.weight layout: read directly
    return w["X"], A, w["dY"], spec["s"]


def _noalloc(X, A, dY, s):
    M, K = X.shape
    r = A.shape[1]
    L = dY.shape[1]
    dt = binding.LORA_BF16 if X.dtype == torch.bfloat16 else binding.LORA_F32
    dB = torch.full((r, L), float("nan"), dtype=torch.float32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = binding.lib().lora_backward_db_noalloc(dt, M, K, L, r, _p(X), X.stride(0), _p(A), A.stride(0),
                                                A.stride(1), _p(dY), dY.stride(0), ctypes.c_float(s), _p(dB),
                                                dB.stride(0), dB.stride(1), stream)
    assert st == 0, binding.STATUS.get(st)
    torch.cuda.synchronize()
    return dB


def _check(X, A, dY, s, dB):
    ref_ws = torch.empty_like(dB)
    binding.lora_backward_db(X, A, dY, s, ref_ws)          # the workspace entry point
    torch.cuda.synchronize()
    assert rel_err(f64(dB), f64(ref_ws)) <= TOL_F32
    ref = O.backward_db(f64(X), f64(A), f64(dY), s)
    assert rel_err(f64(dB), ref) <= TOL_F32
    assert binding.lora_device_error() == 0


@pytest.mark.parametrize("name,mode", [("single_c2", "peft"), ("single_c2", "rowmajor"), ("single_c1", "rowmajor")])
def test_noalloc_db_twice_in_a_row(name, mode):
    """Two calls with the same shape: the second reuses what the first left."""
    X, A, dY, s = _inputs(name, 3000, 1024, 768, 16 if name == "single_c2" else 8, 21, mode)
    for _ in range(2):
        _check(X, A, dY, s, _noalloc(X, A, dY, s))


@pytest.mark.parametrize("name", ["single_c2", "single_c1"])
def test_noalloc_db_large_small_large(name):
    """A large call, a small one, then the large one again (bf16 and fp32; in
    fp32 the intermediate h lives in the shared array too)."""
    big = (4100, 1096, 1496, 64) if name == "single_c2" else (3000, 600, 700, 32)
    small = (70, 136, 200, 9)
    for (M, K, L, r), seed in ((big, 1), (small, 2), (big, 3)):
        X, A, dY, s = _inputs(name, M, K, L, r, seed, "rowmajor")
        _check(X, A, dY, s, _noalloc(X, A, dY, s))
