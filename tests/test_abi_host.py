"""The C ABI library on the host: it loads, exports every declared entry point,
and rejects bad arguments before launching anything (no GPU needed)."""
import ctypes

import pytest

from lora_rank_adapter_gb300 import _build
from lora_rank_adapter_gb300 import binding as B
from tests._util import header_functions


@pytest.fixture(scope="module")
def L():
    _build.build()
    return B.lib()


def test_every_declared_symbol_is_exported(L):
    declared = header_functions()
    assert len(declared) == 19, declared
    assert sorted(B.EXPORTS) == declared
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.lora_version().decode().startswith("lora-gb300")
    for code, name in B.STATUS.items():
        assert L.lora_status_string(code).decode().startswith(name)


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails validation
MIS = ctypes.c_void_p(0x10002)       # not 16-byte aligned
NULL = ctypes.c_void_p(0)
S0 = ctypes.c_void_p(0)


def fwd(L, dt=1, M=64, K=64, L_=64, r=16, X=FAKE, ldx=64, A=FAKE, sak=1, sar=64, Bp=FAKE, sbr=1, sbl=16,
        Y=FAKE, ldy=64, ws=NULL, wsb=0):
    return L.lora_forward(dt, M, K, L_, r, X, ldx, A, sak, sar, Bp, sbr, sbl, Y, ldy, 1.0, ws, wsb, S0)


def test_forward_argument_errors(L):
    assert fwd(L, dt=7) == 2                       # unsupported dtype
    assert fwd(L, M=-1) == 1
    assert fwd(L, r=-1) == 1
    assert fwd(L, r=129) == 2                      # rank above LORA_MAX_RANK
    assert fwd(L, X=NULL) == 1
    assert fwd(L, Y=NULL) == 1
    assert fwd(L, A=NULL) == 1
    assert fwd(L, X=MIS) == 3                      # misaligned big operand
    assert fwd(L, ldx=60) == 1                     # ldx < K
    assert fwd(L, ldx=68) == 3                     # row stride not a 16-byte multiple (bf16)
    assert fwd(L, dt=0, ldx=66, K=66) == 3         # fp32: 264 bytes is not a multiple of 16
    assert fwd(L, K=60) == 3                       # bf16 K not a multiple of 8 (ldx 64 stays legal)
    assert fwd(L, L_=60) == 3                      # bf16 L not a multiple of 8 (ldy 64 stays legal)
    # A stored K x r (not the TMA-readable layout) needs workspace for repacking
    assert fwd(L, sak=16, sar=1) == 4
    # degenerate shapes are a no-op and touch nothing (no device needed)
    assert fwd(L, M=0, X=NULL, Y=NULL) == 0
    assert fwd(L, r=0, A=NULL, Bp=NULL) == 0
    assert fwd(L, K=0) == 0


def test_backward_argument_errors(L):
    dx = lambda **k: L.lora_backward_dx_da(k.get("dt", 1), k.get("M", 64), 64, 64, k.get("r", 16),
                                           k.get("X", FAKE), 64, k.get("dY", FAKE), 64, FAKE, 1, 64,
                                           FAKE, 1, 16, 1.0, k.get("dX", FAKE), 64, k.get("dA", FAKE), 16, 1,
                                           k.get("ws", NULL), k.get("wsb", 0), S0)
    assert dx(dt=3) == 2
    assert dx(r=1000) == 2
    assert dx(dX=NULL) == 1
    assert dx(dA=NULL) == 1
    assert dx(dY=MIS) == 3
    assert dx() == 4                               # the backward always needs workspace
    need = L.lora_workspace_size(B.OP_BACKWARD_DX_DA, 1, 64, 64, 64, 16, 0)
    assert need > 0
    assert dx(ws=ctypes.c_void_p(0x10080), wsb=need) == 4     # not 256-byte aligned
    assert dx(ws=ctypes.c_void_p(0x10000), wsb=need - 1) == 4  # too small
    db = lambda **k: L.lora_backward_db(1, 64, 64, 64, 16, k.get("X", FAKE), 64, FAKE, 1, 64, FAKE, 64, 1.0,
                                        k.get("dB", FAKE), 64, 1, NULL, 0, S0)
    assert db(dB=NULL) == 1
    assert db(X=MIS) == 3
    assert db() == 4


def test_bf16_extents_multiple_of_8(L):
    """bf16 single-adapter calls with K or L off a multiple of 8 return
    LORA_ERR_ALIGNMENT before anything else is looked at (rows of Y and dX are
    stored in 16-byte pieces); fp32 keeps any extent."""
    for K, Lc in ((60, 64), (64, 60)):
        assert L.lora_backward_dx_da(1, 64, K, Lc, 16, FAKE, 64, FAKE, 64, FAKE, 1, 64, FAKE, 1, 16, 1.0,
                                     FAKE, 64, FAKE, 16, 1, NULL, 0, S0) == 3
        assert L.lora_backward_db(1, 64, K, Lc, 16, FAKE, 64, FAKE, 1, 64, FAKE, 64, 1.0, FAKE, 64, 1,
                                  NULL, 0, S0) == 3
        assert L.lora_forward_h(1, 64, K, Lc, 16, FAKE, 64, FAKE, 1, 64, FAKE, 1, 16, FAKE, 64, 1.0, FAKE, 16,
                                NULL, 0, S0) == 3
        assert L.lora_backward(1, 64, K, Lc, 16, FAKE, 64, FAKE, 64, FAKE, 1, 64, FAKE, 1, 16, FAKE, 16, 1.0,
                               FAKE, 64, FAKE, 16, 1, FAKE, 64, 1, NULL, 0, S0) == 3
        assert L.lora_backward_ex(1, 64, K, Lc, 16, FAKE, 64, FAKE, 64, FAKE, 1, 64, FAKE, 1, 16, FAKE, 16, 1.0,
                                  FAKE, 64, FAKE, 16, 1, FAKE, 64, 1, 0, NULL, 0, S0) == 3
        assert L.lora_backward_db_noalloc(1, 64, K, Lc, 16, FAKE, 64, FAKE, 1, 64, FAKE, 64, 1.0, FAKE, 64, 1,
                                          S0) == 3
    # fp32: the same extents pass the checks (and then want their workspace)
    assert L.lora_backward_dx_da(0, 64, 60, 60, 16, FAKE, 64, FAKE, 64, FAKE, 1, 64, FAKE, 1, 16, 1.0,
                                 FAKE, 64, FAKE, 16, 1, NULL, 0, S0) == 4


def test_fused_argument_errors(L):
    fh = lambda **k: L.lora_forward_h(1, k.get("M", 64), 64, 64, 16, FAKE, 64, FAKE, 1, 64, FAKE, 1, 16, FAKE, 64,
                                      1.0, k.get("h", FAKE), k.get("ldh", 16), NULL, 0, S0)
    assert fh(h=NULL) == 1                         # h is required
    assert fh(ldh=8) == 1                          # ldh < r
    assert fh(M=0, h=NULL) == 0                    # nothing to write
    bw = lambda **k: L.lora_backward(1, 64, 64, 64, 16, FAKE, 64, FAKE, 64, FAKE, 1, 64, FAKE, 1, 16,
                                     k.get("h", FAKE), k.get("ldh", 16), 1.0, FAKE, 64, FAKE, 16, 1,
                                     k.get("dB", FAKE), 64, 1, k.get("ws", NULL), k.get("wsb", 0), S0)
    assert bw(h=NULL) == 1
    assert bw(ldh=4) == 1
    assert bw(dB=NULL) == 1
    assert bw() == 4                               # needs workspace
    need = L.lora_workspace_size(B.OP_BACKWARD, 1, 64, 64, 64, 16, 0)
    assert need >= L.lora_workspace_size(B.OP_BACKWARD_DX_DA, 1, 64, 64, 64, 16, 0)
    bx = lambda **k: L.lora_backward_ex(k.get("dt", 1), k.get("M", 64), 64, 64, 16, FAKE, 64, FAKE, 64, FAKE, 1, 64,
                                        FAKE, 1, 16, FAKE, 16, 1.0, FAKE, 64, k.get("dA", FAKE), 16, 1, FAKE, 64,
                                        1, k.get("flags", 0), k.get("ws", NULL), k.get("wsb", 0), S0)
    assert bx(flags=4) == 1                        # unknown flag
    assert bx(flags=3, dA=NULL) == 1               # dA still required
    assert bx(flags=3) == 4                        # needs the lora_backward workspace
    assert bx(flags=1) == 4


def test_workspace_sizes_monotone(L):
    for op in (B.OP_FORWARD, B.OP_BACKWARD_DX_DA, B.OP_BACKWARD_DB, B.OP_BACKWARD):
        small = L.lora_workspace_size(op, 1, 256, 512, 512, 8, 0)
        big = L.lora_workspace_size(op, 1, 8192, 4096, 4096, 16, 0)
        assert big >= small >= 0
        assert L.lora_workspace_size(op, 1, 256, 512, 512, 500, 0) == 0   # invalid rank
    assert L.lora_workspace_size(B.OP_BACKWARD_DX_DA, 0, 256, 512, 512, 8, 0) == 256 * 8 * 4


def test_multi_argument_errors(L):
    slots = ctypes.c_void_p(0x20000)
    ad = B.LoraAddressing(slots.value, 16, 4, 8)
    P = ctypes.byref
    osl = (ctypes.c_int32 * 1)(32)
    assert L.lora_shrink(None, FAKE, 64, 1, FAKE, 64, FAKE, 512, 64, FAKE, 8, NULL, 0, S0) == 1
    bad = B.LoraAddressing(slots.value, 16, 0, 8)
    assert L.lora_shrink(P(bad), FAKE, 64, 1, FAKE, 64, FAKE, 512, 64, FAKE, 8, NULL, 0, S0) == 1
    bad = B.LoraAddressing(slots.value, 16, 5000, 8)
    assert L.lora_shrink(P(bad), FAKE, 64, 1, FAKE, 64, FAKE, 512, 64, FAKE, 8, NULL, 0, S0) == 2
    assert L.lora_shrink(P(ad), FAKE, 64, 9, FAKE, 64, FAKE, 512, 64, FAKE, 72, NULL, 0, S0) == 2
    assert L.lora_shrink(P(ad), FAKE, 64, 1, MIS, 64, FAKE, 512, 64, FAKE, 8, NULL, 0, S0) == 3
    assert L.lora_expand(P(ad), FAKE, FAKE, None, 1, FAKE, 8, FAKE, 256, 8, 1, FAKE, 32, NULL, 0, S0) == 1
    assert L.lora_expand(P(ad), FAKE, NULL, osl, 1, FAKE, 8, FAKE, 256, 8, 1, FAKE, 32, NULL, 0, S0) == 1
    assert L.lora_gather_shrink(P(ad), FAKE, 100, NULL, FAKE, 800, 100, 1, FAKE, 8, S0) == 1
    empty = B.LoraAddressing(0, 0, 4, 8)
    assert L.lora_gather_shrink(P(empty), NULL, 100, NULL, NULL, 800, 100, 1, NULL, 8, S0) == 0


def test_noalloc_argument_errors_come_before_the_size_check(L):
    """lora_backward_db_noalloc reports a bad dtype, size or rank as such (the
    errors of lora_backward_db), and only then compares the workspace the call
    would need with its fixed scratch array; nothing is launched either way."""
    M, K, Lc, r = 16384, 14336, 4096, 64
    scratch = 16 << 20
    assert L.lora_workspace_size(B.OP_BACKWARD_DB, B.LORA_BF16, M, K, Lc, r, 0) > scratch
    nb = lambda dt=B.LORA_BF16, m=M, rr=r: L.lora_backward_db_noalloc(
        dt, m, K, Lc, rr, FAKE, K, FAKE, 1, K, FAKE, Lc, 0.5, FAKE, Lc, 1, S0)
    assert nb(dt=7) == 2                  # unsupported dtype, not a scratch overflow
    assert nb(m=-1) == 1                  # negative size
    assert nb(rr=500) == 2                # rank above LORA_MAX_RANK
    assert nb() == 4                      # valid but larger than the scratch array


def test_schedule_argument_errors(L):
    """lora_build_schedule checks its buffer; a prebuilt schedule in the
    addressing must be 256-byte aligned (checked before any launch)."""
    slots = ctypes.c_void_p(0x20000)
    assert L.lora_schedule_size(4096, 32) > 4096 * 4
    assert L.lora_schedule_size(0, 32) == 0 and L.lora_schedule_size(10, 0) == 0
    ad = B.LoraAddressing(slots.value, 4096, 32, 64, 0)
    P = ctypes.byref
    assert L.lora_build_schedule(P(ad), FAKE, NULL, 0, S0) == 4
    assert L.lora_build_schedule(P(ad), FAKE, MIS, 1 << 20, S0) == 4
    assert L.lora_build_schedule(None, FAKE, FAKE, 1 << 20, S0) == 1
    bad = B.LoraAddressing(slots.value, 4096, 32, 64, 0x10010)   # not 256-byte aligned
    assert L.lora_shrink(P(bad), FAKE, 64, 1, FAKE, 64, FAKE, 512, 64, FAKE, 64, NULL, 0, S0) == 3
