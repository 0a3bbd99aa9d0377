"""lora_backward_db_noalloc, the entry point for callers that cannot allocate
device memory (it uses the library's own static scratch array instead of a
workspace).  Called through the C ABI; its dB must match lora_backward_db's
(which uses a caller workspace) within the fp32 tolerance of the suite, on two
calls in a row (the second reuses the array the first one left behind).  This
file is collected last on purpose."""
import ctypes

import pytest
import torch

from lora_rank_adapter_gb300 import _build
from lora_rank_adapter_gb300 import binding
from lora_rank_adapter_gb300 import synth
from tests._util import TOL_F32, f64, rel_err

pytestmark = pytest.mark.gpu

LORA_ERR_WORKSPACE = 4
SCRATCH_BYTES = 16 << 20


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("mode", ["peft", "rowmajor"])
def test_noalloc_db_matches_workspace_entry_point(mode):
    _build.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    L = binding.lib()
    dev = "cuda:0"
    spec = synth.single_spec("single_c2", M=3000, K=1024, L=768, r=16)
    w = synth.make_single(spec, seed=21, device=dev)
    X, A, dY = w["X"], w["A"], w["dY"]
    if mode == "peft":
        A = A.t().contiguous().t()        # lora_A.weight layout: read directly
    M, K = X.shape
    r = A.shape[1]
    Lc = dY.shape[1]
    s = spec["s"]
    ref = torch.empty((r, Lc), dtype=torch.float32, device=dev)
    binding.lora_backward_db(X, A, dY, s, ref)                  # the workspace entry point
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        dB = torch.full((r, Lc), float("nan"), dtype=torch.float32, device=dev)
        st = L.lora_backward_db_noalloc(binding.LORA_BF16, M, K, Lc, r, _p(X), X.stride(0), _p(A), A.stride(0),
                                        A.stride(1), _p(dY), dY.stride(0), ctypes.c_float(s), _p(dB), dB.stride(0),
                                        dB.stride(1), stream)
        assert st == 0, binding.STATUS.get(st)
        torch.cuda.synchronize()
        assert rel_err(f64(dB), f64(ref)) <= TOL_F32


def test_noalloc_db_rejects_sizes_beyond_the_scratch():
    _build.build()
    L = binding.lib()
    M, K, Lc, r = 16384, 14336, 4096, 64
    assert L.lora_workspace_size(binding.OP_BACKWARD_DB, binding.LORA_BF16, M, K, Lc, r, 0) > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)     # never touched: the size check comes first
    st = L.lora_backward_db_noalloc(binding.LORA_BF16, M, K, Lc, r, fake, K, fake, 1, K, fake, Lc,
                                    ctypes.c_float(0.5), fake, Lc, 1, ctypes.c_void_p(0))
    assert st == LORA_ERR_WORKSPACE
