"""Full-size parity of the wide-MLP LoRA training workloads (16384 tokens,
r = 64, scale 0.5, bf16; up 4096 -> 14336 and down 14336 -> 4096) against the
fp64 oracle, EVERY element of every output, through both training paths of
the C ABI:
  * lora_forward_h + lora_backward (h saved by the forward, one backward call),
    and lora_backward_ex with its output options;
  * lora_forward + lora_backward_dx_da + lora_backward_db.
Tolerances as in the rest of the suite: max|gpu - oracle| / max|oracle| <= 8e-3
for bf16 outputs (Y, dX, and dA / dB stored in bf16), <= 1e-4 for fp32 outputs
(h, dA, dB).  The forward is also checked on its delta alone, since the
N(0, 1) Y0 dominates Y: a second forward onto Y0 = 0.
"""
import numpy as np
import pytest
import torch

from lora_rank_adapter_gb300 import _build
from lora_rank_adapter_gb300 import binding as lora
from lora_rank_adapter_gb300 import synth
from oracle import oracle as O
from tests._util import TOL_BF16, TOL_F32, f64, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


@pytest.fixture(scope="module", params=["single_c3_up", "single_c3_down"])
def c3(request):
    """Inputs on the GPU (adapter weights in the PEFT layouts) and the oracle's
    outputs, computed once per projection."""
    name = request.param
    spec = synth.single_spec(name)
    w = synth.make_single(spec, seed=0, device=DEV, prefix=name)
    s = spec["s"]
    X, A, B, Y0, dY = w["X"], w["A"], w["B"], w["Y0"], w["dY"]
    Xf, Af, Bf, Y0f, dYf = f64(X), f64(A), f64(B), f64(Y0), f64(dY)
    M, K = Xf.shape
    r, L = Bf.shape
    ref = {"Y": O.forward(Xf, Af, Bf, Y0f, s)}
    ref["dY"] = ref["Y"] - Y0f                          # the LoRA delta s (X A) B (to ~1e-16)
    ref["dX"], ref["dA"] = O.backward_dx_da(Xf, dYf, Af, Bf, s)
    ref["dB"] = O.backward_db(Xf, Af, dYf, s)
    # h = X A: the forward with B = I (r x r), Y0 = 0 and s = 1 adds exact zeros only
    ref["h"] = O.forward(Xf, Af, np.eye(r), np.zeros((M, r)), 1.0)
    del Xf, Y0f, dYf
    yield dict(name=name, s=s, X=X, A=A.t().contiguous().t(), B=B.t().contiguous().t(), Y0=Y0, dY=dY,
               ref=ref, M=M, K=K, L=L, r=r)
    torch.cuda.empty_cache()


def _check_y(c, Y, fwd):
    """Y against the oracle, then the delta alone: a second forward onto Y0 = 0
    against s (X A) B (Y - Y0 would mostly show the rounding of Y to bf16)."""
    assert rel_err(f64(Y), c["ref"]["Y"]) <= TOL_BF16
    Z = torch.zeros_like(c["Y0"])
    fwd(Z)
    torch.cuda.synchronize()
    assert rel_err(f64(Z), c["ref"]["dY"]) <= TOL_BF16


def test_c3_forward_h_and_backward_every_element(c3):
    c = c3
    Y = c["Y0"].clone()
    h = torch.full((c["M"], c["r"]), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_forward_h(c["X"], c["A"], c["B"], Y, c["s"], h)
    dX = torch.full_like(c["X"], float("nan"))
    dA = torch.full((c["K"], c["r"]), float("nan"), dtype=torch.float32, device=DEV)
    dB = torch.full((c["r"], c["L"]), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_backward(c["X"], c["dY"], c["A"], c["B"], h, c["s"], dX, dA, dB)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    _check_y(c, Y, lambda Z: lora.lora_forward_h(c["X"], c["A"], c["B"], Z, c["s"], torch.empty_like(h)))
    assert rel_err(f64(h), c["ref"]["h"]) <= TOL_F32
    assert rel_err(f64(dX), c["ref"]["dX"]) <= TOL_BF16
    assert rel_err(f64(dA), c["ref"]["dA"]) <= TOL_F32
    assert rel_err(f64(dB), c["ref"]["dB"]) <= TOL_F32


def test_c3_two_call_backward_every_element(c3):
    c = c3
    Y = c["Y0"].clone()
    lora.lora_forward(c["X"], c["A"], c["B"], Y, c["s"])
    dX = torch.full_like(c["X"], float("nan"))
    dA = torch.full((c["K"], c["r"]), float("nan"), dtype=torch.float32, device=DEV)
    dB = torch.full((c["r"], c["L"]), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_backward_dx_da(c["X"], c["dY"], c["A"], c["B"], c["s"], dX, dA)
    lora.lora_backward_db(c["X"], c["A"], c["dY"], c["s"], dB)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    _check_y(c, Y, lambda Z: lora.lora_forward(c["X"], c["A"], c["B"], Z, c["s"]))
    assert rel_err(f64(dX), c["ref"]["dX"]) <= TOL_BF16
    assert rel_err(f64(dA), c["ref"]["dA"]) <= TOL_F32
    assert rel_err(f64(dB), c["ref"]["dB"]) <= TOL_F32


def test_c3_backward_ex_options_every_element(c3):
    """dX accumulated onto an existing gradient, dA and dB returned in bf16."""
    c = c3
    h = torch.empty((c["M"], c["r"]), dtype=torch.float32, device=DEV)
    Y = c["Y0"].clone()
    lora.lora_forward_h(c["X"], c["A"], c["B"], Y, c["s"], h)
    g = torch.Generator(device=DEV).manual_seed(5)
    dX0 = (torch.randn(c["X"].shape, generator=g, device=DEV) * 1e-3).to(torch.bfloat16)
    dX = dX0.clone()
    dA = torch.full((c["K"], c["r"]), float("nan"), dtype=torch.bfloat16, device=DEV)
    dB = torch.full((c["r"], c["L"]), float("nan"), dtype=torch.bfloat16, device=DEV)
    lora.lora_backward_ex(c["X"], c["dY"], c["A"], c["B"], h, c["s"], dX, dA, dB,
                          flags=lora.BWD_DX_ACCUMULATE | lora.BWD_GRAD_INPUT_DTYPE)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    assert rel_err(f64(dX), f64(dX0) + c["ref"]["dX"]) <= TOL_BF16
    assert rel_err(f64(dA), c["ref"]["dA"]) <= TOL_BF16
    assert rel_err(f64(dB), c["ref"]["dB"]) <= TOL_BF16
