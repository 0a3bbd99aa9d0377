"""GPU parity of lora_forward_h (Y and the saved h = X * A) and lora_backward
(dX, dA and dB in one call from the saved h) against the fp64 oracle, through
the C ABI.

h has no oracle function of its own: it is the multi-adapter shrink with one
slot whose adapter is A^T (a pinned oracle function).  Tolerances as for the
separate ops: 8e-3 (bf16 outputs Y, dX), 1e-4 (fp32 outputs h, dA, dB).
"""
import numpy as np
import pytest
import torch

from lora_rank_adapter_gb300 import _build
from lora_rank_adapter_gb300 import binding as lora
from lora_rank_adapter_gb300 import synth
from oracle import oracle as O
from tests._util import TOL_BF16, TOL_F32, f64, rel_err
from tests.test_parity_single import SENT, SMALL, layouts, padded, untouched

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def oracle_h(X, A):
    """h = X A through the pinned shrink oracle: one slot, adapter A^T, rank r."""
    M, K = X.shape
    r = A.shape[1]
    return O.shrink(X, A.T.reshape(1, r, K), np.zeros(M, np.int32), np.array([r], np.int32), r, 1)


def run_fused(w, s, mode="peft", pad=True):
    X, A, B, Y0, dY = w["X"], w["A"], w["B"], w["Y0"], w["dY"]
    M, K = X.shape
    L = B.shape[1]
    r = A.shape[1]
    Al, Bl = layouts(A, B, mode)
    rp, cp = (3, 5) if pad else (0, 0)
    Xv, _ = padded(X, 0, 8 if pad else 0)
    Yv, Ybuf = padded(Y0, rp, cp)
    dYv, _ = padded(dY, 0, 8 if pad else 0)
    hbuf = torch.full((M + rp, r + cp + 1), SENT, dtype=torch.float32, device=DEV)
    h = hbuf[:M, :r]
    lora.lora_forward_h(Xv, Al, Bl, Yv, s, h)
    dXv, dXbuf = padded(torch.zeros_like(X), rp, cp)
    dAbuf = torch.full((K + 2, r + 3), SENT, dtype=torch.float32, device=DEV)
    dBbuf = torch.full((r + 2, L + 3), SENT, dtype=torch.float32, device=DEV)
    dA, dB = dAbuf[:K, :r], dBbuf[:r, :L]
    lora.lora_backward(Xv, dYv, Al, Bl, h, s, dXv, dA, dB)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    return dict(Y=Yv, Ybuf=Ybuf, h=h, hbuf=hbuf, dX=dXv, dXbuf=dXbuf, dA=dA, dAbuf=dAbuf, dB=dB, dBbuf=dBbuf)


def check_fused(w, s, out, tol_lo):
    X, A, B, Y0, dY = (f64(w[k]) for k in ("X", "A", "B", "Y0", "dY"))
    M, K = X.shape
    r, L = B.shape
    ref = dict(Y=O.forward(X, A, B, Y0, s), h=oracle_h(X, A))
    ref["dX"], ref["dA"] = O.backward_dx_da(X, dY, A, B, s)
    ref["dB"] = O.backward_db(X, A, dY, s)
    tol = dict(Y=tol_lo, h=TOL_F32, dX=tol_lo, dA=TOL_F32, dB=TOL_F32)
    for k in tol:
        e = rel_err(f64(out[k]), ref[k])
        assert e <= tol[k], (k, e, tol[k])
    for k, (m, n) in dict(Ybuf=(M, L), hbuf=(M, r), dXbuf=(M, K), dAbuf=(K, r), dBbuf=(r, L)).items():
        assert untouched(out[k], m, n), k


def workload(M, K, L, r, dtype, seed):
    w = {}
    bound = 1.0 / np.sqrt(max(K, 1))
    for name, shape, dist in (("X", (M, K), ("normal", 1.0)), ("A", (K, r), ("uniform", -bound, bound)),
                              ("B", (r, L), ("normal", 0.02)), ("Y0", (M, L), ("normal", 1.0)),
                              ("dY", (M, L), ("normal", 0.01))):
        w[name] = synth.draw(dist, shape, seed, "f." + name, dtype, DEV)
    return w


@pytest.mark.parametrize("M,K,L,r", SMALL)
@pytest.mark.parametrize("mode", ["peft", "rowmajor"])
def test_fused_bf16_small(M, K, L, r, mode):
    w = workload(M, K, L, r, "bf16", M + K + L + r)
    check_fused(w, 2.0, run_fused(w, 2.0, mode), TOL_BF16)


@pytest.mark.parametrize("M,K,L,r", [(1, 4, 4, 1), (17, 33, 65, 7), (256, 512, 512, 8), (70, 130, 30, 128)])
@pytest.mark.parametrize("mode", ["peft", "strided"])
def test_fused_f32(M, K, L, r, mode):
    w = workload(M, K, L, r, "f32", M + K + L + r)
    check_fused(w, 2.0, run_fused(w, 2.0, mode), TOL_F32)


def test_fused_c2_full_bf16():
    """The q_proj workload at full size (8192 x 4096 x 4096, r = 16), every element."""
    spec = synth.single_spec("single_c2")
    w = synth.make_single(spec, seed=0, device=DEV)
    check_fused(w, spec["s"], run_fused(w, spec["s"], pad=False), TOL_BF16)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fused_matches_separate_ops(dtype):
    """lora_backward runs the dX / dA passes of lora_backward_dx_da unchanged
    (bit-identical) and its dB agrees with lora_backward_db within rounding."""
    w = workload(300, 136, 200, 24, dtype, 5)
    X, A, B, dY = w["X"], w["A"], w["B"], w["dY"]
    M, K = X.shape
    r, L = B.shape
    h = torch.empty((M, r), dtype=torch.float32, device=DEV)
    lora.lora_forward_h(X, A, B, w["Y0"].clone(), 2.0, h)
    dX1, dA1, dB1 = torch.empty_like(X), torch.empty((K, r), device=DEV), torch.empty((r, L), device=DEV)
    lora.lora_backward(X, dY, A, B, h, 2.0, dX1, dA1, dB1)
    dX2, dA2, dB2 = torch.empty_like(X), torch.empty((K, r), device=DEV), torch.empty((r, L), device=DEV)
    lora.lora_backward_dx_da(X, dY, A, B, 2.0, dX2, dA2)
    lora.lora_backward_db(X, A, dY, 2.0, dB2)
    torch.cuda.synchronize()
    assert torch.equal(dX1, dX2) and torch.equal(dA1, dA2)
    assert rel_err(f64(dB1), f64(dB2)) <= TOL_F32


def test_fused_degenerate_shapes():
    X = synth.draw(("normal", 1.0), (40, 24), 0, "g.X", "bf16", DEV)
    dY = synth.draw(("normal", 1.0), (40, 16), 0, "g.dY", "bf16", DEV)
    A = synth.draw(("normal", 1.0), (24, 4), 0, "g.A", "bf16", DEV)
    B = synth.draw(("normal", 1.0), (4, 16), 0, "g.B", "bf16", DEV)
    # L = 0: h is still X A (no Y columns); dX = 0, dA = 0, dB empty
    h = torch.full((40, 4), 3.0, device=DEV)
    Bz = torch.empty((4, 0), dtype=torch.bfloat16, device=DEV)
    lora.lora_forward_h(X, A, Bz, torch.empty((40, 0), dtype=torch.bfloat16, device=DEV), 1.0, h)
    torch.cuda.synchronize()
    assert rel_err(f64(h), oracle_h(f64(X), f64(A))) <= TOL_F32
    # K = 0: h = 0, and lora_backward gives dB = 0
    hz = torch.full((40, 4), 3.0, device=DEV)
    X0 = torch.empty((40, 0), dtype=torch.bfloat16, device=DEV)
    A0 = torch.empty((0, 4), dtype=torch.bfloat16, device=DEV)
    lora.lora_forward_h(X0, A0, B, torch.zeros((40, 16), dtype=torch.bfloat16, device=DEV), 1.0, hz)
    dB = torch.full((4, 16), 3.0, device=DEV)
    lora.lora_backward(X0, dY, A0, B, hz, 1.0, torch.empty((40, 0), dtype=torch.bfloat16, device=DEV),
                       torch.empty((0, 4), device=DEV), dB)
    # M = 0: dA = 0 and dB = 0
    dA = torch.full((24, 4), 3.0, device=DEV)
    dB2 = torch.full((4, 16), 3.0, device=DEV)
    lora.lora_backward(X[:0], dY[:0], A, B, torch.empty((0, 4), device=DEV), 1.0,
                       torch.empty((0, 24), dtype=torch.bfloat16, device=DEV), dA, dB2)
    torch.cuda.synchronize()
    assert torch.all(hz == 0) and torch.all(dB == 0) and torch.all(dA == 0) and torch.all(dB2 == 0)


# ----------------------------------------------------------------------------- output options
def _grad_bufs(K, r, L, dt):
    dAbuf = torch.full((K + 2, r + 3), SENT, dtype=dt, device=DEV)
    dBbuf = torch.full((r + 2, L + 3), SENT, dtype=dt, device=DEV)
    return dAbuf, dBbuf, dAbuf[:K, :r], dBbuf[:r, :L]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("flags", [1, 2, 3])
@pytest.mark.parametrize("M,K,L,r", [(3, 24, 40, 3), (130, 200, 72, 16), (300, 136, 200, 64), (129, 256, 192, 128)])
def test_backward_ex_options(M, K, L, r, flags, dtype):
    """lora_backward_ex: dX accumulated onto a prior dX of the update's own size
    (so the check sees the update), and dA / dB in the input dtype."""
    w = workload(M, K, L, r, dtype, 11 + M + r)
    s = 2.0
    X, A, B, dY = w["X"], w["A"], w["B"], w["dY"]
    h = torch.empty((M, r), dtype=torch.float32, device=DEV)
    lora.lora_forward_h(X, A, B, w["Y0"].clone(), s, h)
    acc = bool(flags & lora.BWD_DX_ACCUMULATE)
    upd, _ = O.backward_dx_da(f64(X), f64(dY), f64(A), f64(B), s)
    sigma = float(np.max(np.abs(upd))) / 2 or 1.0
    dX0 = synth.draw(("normal", sigma), (M, K), 7, "g.dX0", dtype, DEV)
    dXv, dXbuf = padded(dX0, 3, 5)
    gdt = X.dtype if flags & lora.BWD_GRAD_INPUT_DTYPE else torch.float32
    dAbuf, dBbuf, dA, dB = _grad_bufs(K, r, L, gdt)
    lora.lora_backward_ex(X, dY, A, B, h, s, dXv, dA, dB, flags=flags)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    rdX, rdA, rdB = O.backward_ex(f64(X), f64(dY), f64(A), f64(B), s, f64(dX0) if acc else None)
    lo = dtype == "bf16"
    tol_g = TOL_BF16 if (lo and gdt != torch.float32) else TOL_F32
    assert rel_err(f64(dXv), rdX) <= (TOL_BF16 if lo else TOL_F32)
    assert rel_err(f64(dA), rdA) <= tol_g and rel_err(f64(dB), rdB) <= tol_g
    assert untouched(dXbuf, M, K) and untouched(dAbuf, K, r) and untouched(dBbuf, r, L)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_ex_rounding_relations(dtype):
    """The bf16 gradients are the fp32 gradients rounded once (bit-exact), and an
    accumulation onto zeros is the overwriting backward (bit-exact)."""
    w = workload(257, 264, 392, 24, dtype, 3)
    X, A, B, dY = w["X"], w["A"], w["B"], w["dY"]
    M, K = X.shape
    r, L = B.shape
    h = torch.empty((M, r), dtype=torch.float32, device=DEV)
    lora.lora_forward_h(X, A, B, w["Y0"].clone(), 0.5, h)
    dX1, dA1, dB1 = torch.empty_like(X), torch.empty((K, r), device=DEV), torch.empty((r, L), device=DEV)
    lora.lora_backward(X, dY, A, B, h, 0.5, dX1, dA1, dB1)
    dX2 = torch.zeros_like(X)
    dA2 = torch.empty((K, r), dtype=X.dtype, device=DEV)
    dB2 = torch.empty((r, L), dtype=X.dtype, device=DEV)
    lora.lora_backward_ex(X, dY, A, B, h, 0.5, dX2, dA2, dB2, flags=3)
    torch.cuda.synchronize()
    assert torch.equal(dX1, dX2)
    assert torch.equal(dA1.to(X.dtype), dA2) and torch.equal(dB1.to(X.dtype), dB2)


def test_backward_ex_degenerate_shapes():
    """L = 0: the dX update is zero (an accumulated dX keeps its values), dA = 0 and
    dB is empty; M = 0: dA = 0 and dB = 0, in bf16."""
    X = synth.draw(("normal", 1.0), (40, 24), 0, "g.X", "bf16", DEV)
    A = synth.draw(("normal", 1.0), (24, 4), 0, "g.A", "bf16", DEV)
    dX0 = synth.draw(("normal", 1.0), (40, 24), 1, "g.dX0", "bf16", DEV)
    dX = dX0.clone()
    dA = torch.full((24, 4), 3.0, dtype=torch.bfloat16, device=DEV)
    h = torch.zeros((40, 4), device=DEV)
    lora.lora_backward_ex(X, torch.empty((40, 0), dtype=torch.bfloat16, device=DEV), A,
                          torch.empty((4, 0), dtype=torch.bfloat16, device=DEV), h, 1.0, dX, dA,
                          torch.empty((4, 0), dtype=torch.bfloat16, device=DEV), flags=3)
    dA2 = torch.full((24, 4), 3.0, dtype=torch.bfloat16, device=DEV)
    dB2 = torch.full((4, 16), 3.0, dtype=torch.bfloat16, device=DEV)
    B = synth.draw(("normal", 1.0), (4, 16), 0, "g.B", "bf16", DEV)
    lora.lora_backward_ex(X[:0], torch.empty((0, 16), dtype=torch.bfloat16, device=DEV), A, B,
                          torch.empty((0, 4), device=DEV), 1.0, torch.empty((0, 24), dtype=torch.bfloat16, device=DEV),
                          dA2, dB2, flags=3)
    torch.cuda.synchronize()
    assert torch.equal(dX, dX0) and torch.all(dA == 0) and torch.all(dA2 == 0) and torch.all(dB2 == 0)


def test_backward_then_dependent_launch_sees_dx():
    """The dB pass of lora_backward starts before the dX pass has finished and
    waits for it only before exiting: a launch right after the backward that
    reads dX (here, a forward with dX as its input) must see all of it.  The
    chain on one stream is compared with the same chain separated by full
    synchronizations (c3-like widths, so the dX pass is long and the dB pass
    short)."""
    M, K, L, r = 4096, 4096, 1024, 64
    spec = synth.single_spec("single_c3_down", M=M, K=K, L=L, r=r)
    w = synth.make_single(spec, seed=21, device=DEV)
    X, A, B, dY = w["X"], w["A"], w["B"], w["dY"]
    s = spec["s"]
    h = torch.empty((M, r), dtype=torch.float32, device=DEV)
    Y = w["Y0"].clone()
    lora.lora_forward_h(X, A, B, Y, s, h)
    torch.cuda.synchronize()
    A2 = (A.float() * 0.5).to(A.dtype)
    B2 = torch.randn((r, 512), device=DEV).to(B.dtype)

    def chain(sync):
        dX = torch.full_like(X, float("nan"))
        dA = torch.empty((K, r), dtype=torch.float32, device=DEV)
        dB = torch.empty((r, L), dtype=torch.float32, device=DEV)
        Y2 = torch.zeros((M, 512), dtype=X.dtype, device=DEV)
        lora.lora_backward(X, dY, A, B, h, s, dX, dA, dB)
        if sync:
            torch.cuda.synchronize()
        lora.lora_forward(dX, A2, B2, Y2, 1.0)
        torch.cuda.synchronize()
        return dX, Y2

    dx_sync, y_sync = chain(True)
    for _ in range(5):
        dx_chain, y_chain = chain(False)
        assert torch.equal(dx_chain, dx_sync)
        assert torch.equal(y_chain, y_sync)
    assert torch.isfinite(y_sync.float()).all()
