"""torch.library registration of the ops: fake (shape) implementations run on
the CPU under FakeTensorMode; on a GPU, opcheck validates the registrations and
the autograd.Function's gradients match the fp64 oracle."""
import pytest
import torch

from lora_rank_adapter_gb300 import torch_ops
from tests._util import TOL_BF16, TOL_F32, f64, rel_err


def _fake_mode():
    from torch._subclasses.fake_tensor import FakeTensorMode
    return FakeTensorMode()


def test_fake_shapes_multi_adapter():
    with _fake_mode():
        x = torch.empty((37, 64), dtype=torch.bfloat16)
        a = torch.empty((4, 3 * 16, 64), dtype=torch.bfloat16)
        slots = torch.empty((37,), dtype=torch.int32)
        ranks = torch.empty((4,), dtype=torch.int32)
        h = torch.ops.lora_gb300.shrink(x, a, slots, ranks, 16, 3)
        assert h.shape == (37, 48) and h.dtype == torch.float32
        y = torch.empty((37, 96), dtype=torch.bfloat16)
        b = torch.empty((4, 96, 16), dtype=torch.bfloat16)
        scal = torch.empty((4,), dtype=torch.float32)
        assert torch.ops.lora_gb300.expand_(y, h, b, slots, ranks, scal, [32, 32, 32], 16) is None
        ga = torch.empty((4, 16, 500), dtype=torch.bfloat16)
        ids = torch.empty((37,), dtype=torch.int64)
        hg = torch.ops.lora_gb300.gather_shrink(ids, ga, slots, ranks, 16)
        assert hg.shape == (37, 16)


def test_fake_shapes_single_adapter():
    with _fake_mode():
        x = torch.empty((10, 24), dtype=torch.bfloat16)
        A = torch.empty((24, 8), dtype=torch.bfloat16)
        B = torch.empty((8, 40), dtype=torch.bfloat16)
        dout = torch.empty((10, 40), dtype=torch.bfloat16)
        dx, dA, dB = torch.ops.lora_gb300.backward(x, dout, A, B, 2.0)
        assert dx.shape == x.shape and dA.shape == A.shape and dB.shape == B.shape
        assert dA.dtype == torch.float32 and dB.dtype == torch.float32
        y = torch.empty((10, 40), dtype=torch.bfloat16)
        h = torch.ops.lora_gb300.forward_h_(y, x, A, B, 2.0)
        assert h.shape == (10, 8) and h.dtype == torch.float32
        dx, dA, dB = torch.ops.lora_gb300.backward_ex(x, dout, A, B, h, 2.0, True)
        assert dx.shape == x.shape and dA.dtype == torch.bfloat16 and dB.dtype == torch.bfloat16


def test_no_cpu_kernel():
    """There is no CPU fallback: calling an op on CPU tensors fails loudly."""
    x = torch.zeros((2, 8), dtype=torch.bfloat16)
    A = torch.zeros((8, 8), dtype=torch.bfloat16)
    B = torch.zeros((8, 8), dtype=torch.bfloat16)
    y = torch.zeros((2, 8), dtype=torch.bfloat16)
    with pytest.raises(Exception):
        torch.ops.lora_gb300.forward_(y, x, A, B, 1.0)


@pytest.mark.gpu
def test_opcheck_and_autograd_against_oracle():
    from lora_rank_adapter_gb300 import _build, synth
    from oracle import oracle as O
    _build.build()
    dev = "cuda:0"
    spec = synth.single_spec("single_c2", M=300, K=192, L=136, r=16)
    w = synth.make_single(spec, seed=4, device=dev)
    X, A, B, Y0, dY = w["X"], w["A"], w["B"], w["Y0"], w["dY"]
    s = spec["s"]
    torch.library.opcheck(torch.ops.lora_gb300.forward_.default, (Y0.clone(), X, A, B, s))
    torch.library.opcheck(torch.ops.lora_gb300.backward.default, (X, dY, A, B, s))
    h = torch.ops.lora_gb300.forward_h_(Y0.clone(), X, A, B, s)
    torch.library.opcheck(torch.ops.lora_gb300.forward_h_.default, (Y0.clone(), X, A, B, s))
    torch.library.opcheck(torch.ops.lora_gb300.backward_ex.default, (X, dY, A, B, h, s, True))
    Xg = X.clone().requires_grad_(True)
    Ag = A.clone().requires_grad_(True)
    Bg = B.clone().requires_grad_(True)
    Yb = Y0.clone().requires_grad_(True)
    out = torch_ops.lora_linear(Xg, Ag, Bg, Yb, s)
    out.backward(dY)
    torch.cuda.synchronize()
    ref = O.forward(f64(X), f64(A), f64(B), f64(Y0), s)
    assert rel_err(f64(out), ref) <= TOL_BF16
    rdx, rda = O.backward_dx_da(f64(X), f64(dY), f64(A), f64(B), s)
    rdb = O.backward_db(f64(X), f64(A), f64(dY), s)
    assert rel_err(f64(Xg.grad), rdx) <= TOL_BF16
    # dA / dB come back in the parameters' dtype (bf16): bf16 tolerance
    assert rel_err(f64(Ag.grad), rda) <= TOL_BF16
    assert rel_err(f64(Bg.grad), rdb) <= TOL_BF16
    assert torch.equal(Yb.grad, dY)


@pytest.mark.gpu
def test_opcheck_multi_adapter():
    """opcheck of the registrations, and the ops' results against the oracle."""
    import numpy as np
    from lora_rank_adapter_gb300 import _build, synth
    from oracle import oracle as O
    _build.build()
    spec = synth.multi_spec("multi_c4", T=200, IN=64, out_slices=[64, 32, 32], S=6, R=16,
                            rank_choices=[0, 8, 16])
    w = synth.make_multi(spec, seed=1, device="cuda:0", poison=False)
    h = torch.ops.lora_gb300.shrink(w["x"], w["a"], w["slots"], w["ranks"], 16, 3)
    y = w["y0"].clone()
    torch.ops.lora_gb300.apply_linear_(y, w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"],
                                       [64, 32, 32], 16)
    torch.cuda.synchronize()
    sl, rk = w["slots"].cpu().numpy(), w["ranks"].cpu().numpy()
    sc = w["scalings"].double().cpu().numpy()
    href = O.shrink(f64(w["x"]), f64(w["a"]), sl, rk, 16, 3)
    act = np.array([0 <= v < 6 and 1 <= rk[v] <= 16 for v in sl])
    spec_h = np.zeros(href.shape, bool)
    for t in np.nonzero(act)[0]:
        for i in range(3):
            spec_h[t, i * 16:i * 16 + rk[sl[t]]] = True
    assert rel_err(f64(h)[spec_h], href[spec_h]) <= TOL_F32
    yref = O.apply_linear(f64(w["x"]), f64(w["a"]), f64(w["b"]), sl, rk, sc, f64(w["y0"]), [64, 32, 32], 16)
    assert rel_err(f64(y)[act], yref[act]) <= TOL_BF16
    torch.library.opcheck(torch.ops.lora_gb300.shrink.default, (w["x"], w["a"], w["slots"], w["ranks"], 16, 3),
                          test_utils=("test_schema", "test_faketensor", "test_autograd_registration"))
    torch.library.opcheck(torch.ops.lora_gb300.expand_.default,
                          (w["y0"].clone(), h, w["b"], w["slots"], w["ranks"], w["scalings"], [64, 32, 32], 16),
                          test_utils=("test_schema", "test_faketensor", "test_autograd_registration"))
