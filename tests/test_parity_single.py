"""GPU parity of the single-adapter ops against the fp64 oracle, through the C ABI.

Tolerances (max|gpu - oracle| / max|oracle|): 8e-3 for bf16 outputs (Y, dX),
1e-4 for fp32 outputs (dA, dB, and everything in the fp32 path).  Indexing is
checked bit-exactly: padding columns/rows around every output stay untouched.
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
SENT = -640.0   # sentinel in padding (exactly representable in bf16 and fp32)


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def padded(t, row_pad=0, col_pad=0):
    """Copy of t inside a larger buffer filled with SENT; returns (view, buffer)."""
    M, N = t.shape
    e = t.element_size()
    colp = col_pad
    while ((N + colp) * e) % 16:
        colp += 1
    buf = torch.full((M + row_pad, N + colp), SENT, dtype=t.dtype, device=t.device)
    v = buf[:M, :N]
    v.copy_(t)
    return v, buf


def untouched(buf, M, N):
    b = buf.float().cpu()
    ok = torch.all(b[M:, :] == SENT) and torch.all(b[:, N:] == SENT)
    return bool(ok)


def layouts(A, B, mode):
    """A [K, r] and B [r, L] in the requested memory layouts (same logical values)."""
    if mode == "peft":       # lora_A.weight (r x K) and lora_B.weight (L x r), viewed transposed
        return A.t().contiguous().t(), B.t().contiguous().t()
    if mode == "rowmajor":   # A stored K x r, B stored r x L (repacked on the device)
        return A.contiguous(), B.contiguous()
    if mode == "strided":    # both with a non-unit stride in each dimension
        Ab = torch.zeros((A.shape[0] * 2, A.shape[1] * 3), dtype=A.dtype, device=A.device)
        Ab[::2, ::3] = A
        Bb = torch.zeros((B.shape[0] * 3, B.shape[1] * 2), dtype=B.dtype, device=B.device)
        Bb[::3, ::2] = B
        return Ab[::2, ::3], Bb[::3, ::2]
    raise ValueError(mode)


def run_all(w, s, mode="peft", pad=True):
    X, A, B, Y0, dY = w["X"], w["A"], w["B"], w["Y0"], w["dY"]
    M, K = X.shape
    L = B.shape[1]
    r = A.shape[1]
    Al, Bl = layouts(A, B, mode)
    rp, cp = (3, 5) if pad else (0, 0)
    Xv, _ = padded(X, 0, 8 if pad else 0)
    Yv, Ybuf = padded(Y0, rp, cp)
    dYv, _ = padded(dY, 0, 8 if pad else 0)
    lora.lora_forward(Xv, Al, Bl, Yv, s)
    dX = torch.zeros_like(X)
    dXv, dXbuf = padded(dX, rp, cp)
    dAbuf = torch.full((K + 2, r + 3), SENT, dtype=torch.float32, device=DEV)
    dA = dAbuf[:K, :r]
    dBbuf = torch.full((r + 2, L + 3), SENT, dtype=torch.float32, device=DEV)
    dB = dBbuf[:r, :L]
    lora.lora_backward_dx_da(Xv, dYv, Al, Bl, s, dXv, dA)
    lora.lora_backward_db(Xv, Al, dYv, s, dB)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    return dict(Y=Yv, Ybuf=Ybuf, dX=dXv, dXbuf=dXbuf, dA=dA, dAbuf=dAbuf, dB=dB, dBbuf=dBbuf)


def check_all(w, s, out, tol_lo):
    X, A, B, Y0, dY = (f64(w[k]) for k in ("X", "A", "B", "Y0", "dY"))
    M, K = X.shape
    r, L = B.shape
    ref_y = O.forward(X, A, B, Y0, s)
    ref_dx, ref_da = O.backward_dx_da(X, dY, A, B, s)
    ref_db = O.backward_db(X, A, dY, s)
    errs = dict(Y=rel_err(f64(out["Y"]), ref_y), dX=rel_err(f64(out["dX"]), ref_dx),
                dA=rel_err(f64(out["dA"]), ref_da), dB=rel_err(f64(out["dB"]), ref_db))
    tol = dict(Y=tol_lo, dX=tol_lo, dA=TOL_F32, dB=TOL_F32)
    for k in errs:
        assert errs[k] <= tol[k], (k, errs[k], tol[k])
    assert untouched(out["Ybuf"], M, L)
    assert untouched(out["dXbuf"], M, K)
    assert untouched(out["dAbuf"], K, r)
    assert untouched(out["dBbuf"], r, L)
    return errs


SMALL = [  # M, K, L, r: several tiles plus ragged tails, every rank bucket
    (1, 8, 8, 1), (3, 24, 40, 3), (17, 72, 136, 7), (64, 64, 64, 8), (130, 200, 72, 16),
    (257, 264, 392, 24), (190, 128, 520, 32), (96, 520, 136, 48), (300, 136, 200, 64),
    (65, 192, 128, 100), (129, 256, 192, 128),
]


@pytest.mark.parametrize("M,K,L,r", SMALL)
@pytest.mark.parametrize("mode", ["peft", "rowmajor"])
def test_single_bf16_small(M, K, L, r, mode):
    spec = synth.single_spec("single_c2", M=M, K=K, L=L, r=r)
    w = synth.make_single(spec, seed=M * 7 + r, device=DEV)
    out = run_all(w, spec["s"], mode)
    check_all(w, spec["s"], out, TOL_BF16)


@pytest.mark.parametrize("M,K,L,r", [(8192, 64, 64, 128), (6000, 128, 72, 64), (5000, 64, 200, 16),
                                     (4096, 136, 64, 100)])
def test_single_bf16_many_tiles_per_cta(M, K, L, r):
    """Narrow K / L and tall M: each column-pass CTA walks many more row tiles than
    it has pipeline stages, so every stage is reused several times."""
    spec = synth.single_spec("single_c2", M=M, K=K, L=L, r=r)
    w = synth.make_single(spec, seed=M + r, device=DEV)
    out = run_all(w, spec["s"], "peft")
    check_all(w, spec["s"], out, TOL_BF16)


@pytest.mark.parametrize("M,K,L,r", [(12000, 256, 14200, 64), (15900, 128, 11896, 32)])
def test_forward_shared_tail_ragged(M, K, L, r):
    """Forwards large enough for the expand's shared tail (its last eighth of
    (row block, 128-column chunk) units claimed two at a time by whichever CTA
    is free first), with a ragged last row block and column chunk, chunks that
    cross row blocks, and one and two blob buffers (r = 64, 32).  y0 = 0, so a
    unit updated twice or not at all shows in full."""
    spec = synth.single_spec("single_c2", M=M, K=K, L=L, r=r)
    w = synth.make_single(spec, seed=M + L, device=DEV)
    Al, Bl = layouts(w["A"], w["B"], "peft")
    Y, Ybuf = padded(torch.zeros((M, L), dtype=w["X"].dtype, device=DEV), 3, 5)
    h = torch.empty((M, r), dtype=torch.float32, device=DEV)
    ref = O.forward(f64(w["X"]), f64(w["A"]), f64(w["B"]), np.zeros((M, L)), spec["s"])
    for _ in range(2):   # the claim counter starts from zero on every call
        Y.zero_()
        lora.lora_forward_h(w["X"], Al, Bl, Y, spec["s"], h)
        torch.cuda.synchronize()
        assert lora.lora_device_error() == 0
        assert rel_err(f64(Y), ref) <= TOL_BF16
        assert untouched(Ybuf, M, L)


@pytest.mark.parametrize("M,K,L,r", [(3, 24, 40, 3), (130, 200, 72, 16), (65, 96, 128, 33)])
def test_single_bf16_strided_small_operands(M, K, L, r):
    spec = synth.single_spec("single_c2", M=M, K=K, L=L, r=r)
    w = synth.make_single(spec, seed=11, device=DEV)
    out = run_all(w, spec["s"], "strided")
    check_all(w, spec["s"], out, TOL_BF16)


@pytest.mark.parametrize("M,K,L,r", [(1, 4, 4, 1), (17, 33, 65, 7), (256, 512, 512, 8), (70, 130, 30, 128)])
@pytest.mark.parametrize("mode", ["peft", "rowmajor", "strided"])
def test_single_f32(M, K, L, r, mode):
    spec = synth.single_spec("single_c1", M=M, K=K, L=L, r=r)
    w = synth.make_single(spec, seed=3, device=DEV)
    out = run_all(w, spec["s"], mode, pad=(K % 4 == 0))
    check_all(w, spec["s"], out, TOL_F32)


def test_forward_delta_alone_bf16():
    """With Y0 = 0 the tolerance applies to the LoRA delta itself."""
    spec = synth.single_spec("single_c2", M=300, K=520, L=264, r=16, Y0=("zeros",))
    w = synth.make_single(spec, seed=5, device=DEV)
    out = run_all(w, spec["s"])
    ref = O.forward(*(f64(w[k]) for k in ("X", "A", "B", "Y0")), spec["s"])
    assert rel_err(f64(out["Y"]), ref) <= TOL_BF16


def test_invariants_bf16():
    spec = synth.single_spec("single_c2", M=150, K=136, L=200, r=16)
    w = synth.make_single(spec, seed=6, device=DEV)
    Y = w["Y0"].clone()
    lora.lora_forward(w["X"], w["A"], torch.zeros_like(w["B"]), Y, 2.0)     # B = 0
    lora.lora_forward(w["X"], w["A"], w["B"], Y, 0.0)                       # s = 0
    torch.cuda.synchronize()
    assert torch.equal(Y, w["Y0"])


def test_degenerate_shapes():
    dev = DEV
    X = synth.draw(("normal", 1.0), (40, 24), 0, "d.X", "bf16", dev)
    dY = synth.draw(("normal", 1.0), (40, 16), 0, "d.dY", "bf16", dev)
    Y = synth.draw(("normal", 1.0), (40, 16), 0, "d.Y", "bf16", dev)
    # r = 0: Y untouched, dX zeros, dA / dB empty
    A0 = torch.empty((24, 0), dtype=torch.bfloat16, device=dev)
    B0 = torch.empty((0, 16), dtype=torch.bfloat16, device=dev)
    Yc = Y.clone()
    lora.lora_forward(X, A0, B0, Yc, 1.0)
    dX = torch.full_like(X, 3.0)
    lora.lora_backward_dx_da(X, dY, A0, B0, 1.0, dX, torch.empty((24, 0), device=dev))
    torch.cuda.synchronize()
    assert torch.equal(Yc, Y) and torch.all(dX == 0)
    # L = 0: dX = 0 and dA = 0
    A = synth.draw(("normal", 1.0), (24, 4), 0, "d.A", "bf16", dev)
    Bz = torch.empty((4, 0), dtype=torch.bfloat16, device=dev)
    dX = torch.full_like(X, 3.0)
    dA = torch.full((24, 4), 3.0, device=dev)
    lora.lora_backward_dx_da(X, torch.empty((40, 0), dtype=torch.bfloat16, device=dev), A, Bz, 1.0, dX, dA)
    # K = 0: dB = 0
    dB = torch.full((4, 16), 3.0, device=dev)
    lora.lora_backward_db(torch.empty((40, 0), dtype=torch.bfloat16, device=dev),
                          torch.empty((0, 4), dtype=torch.bfloat16, device=dev), dY, 1.0, dB)
    # M = 0: dA = 0 and dB = 0
    dA2 = torch.full((24, 4), 3.0, device=dev)
    B = synth.draw(("normal", 1.0), (4, 16), 0, "d.B", "bf16", dev)
    lora.lora_backward_dx_da(X[:0], dY[:0], A, B, 1.0, torch.empty((0, 24), dtype=torch.bfloat16, device=dev),
                             dA2)
    dB2 = torch.full((4, 16), 3.0, device=dev)
    lora.lora_backward_db(X[:0], A, dY[:0], 1.0, dB2)
    torch.cuda.synchronize()
    assert torch.all(dX == 0) and torch.all(dA == 0) and torch.all(dB == 0)
    assert torch.all(dA2 == 0) and torch.all(dB2 == 0)


def test_repeatable_bitwise():
    """No float atomics: two runs give identical bits."""
    spec = synth.single_spec("single_c2", M=1000, K=1024, L=768, r=16)
    w = synth.make_single(spec, seed=8, device=DEV)
    a = run_all(w, spec["s"], pad=False)
    b = run_all(w, spec["s"], pad=False)
    for k in ("Y", "dX", "dA", "dB"):
        assert torch.equal(a[k], b[k]), k


def test_c1_full_fp32():
    spec = synth.single_spec("single_c1")
    w = synth.make_single(spec, seed=0, device=DEV)
    out = run_all(w, spec["s"])
    check_all(w, spec["s"], out, TOL_F32)


def test_c2_full_bf16():
    """The q_proj workload at full size (8192 x 4096 x 4096, r = 16), every element."""
    spec = synth.single_spec("single_c2")
    w = synth.make_single(spec, seed=0, device=DEV)
    out = run_all(w, spec["s"], pad=False)
    check_all(w, spec["s"], out, TOL_BF16)
