"""GPU parity of the multi-adapter ops against the fp64 oracle, through the C ABI.

group_by_slot and gather_shrink are integer / copy work: bit-exact.  shrink
produces fp32 h (tolerance 1e-4 of max|oracle| over the specified entries:
active tokens, columns below the slot's rank); expand / apply_linear produce
bf16 y (8e-3), and every row of an inactive token, every padding column and
every padding row around y must stay bit-identical.  The adapter stacks carry
NaN in their padding and the scalings of rank-0 slots are NaN, so any read of
unspecified data shows up.
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
SENT = -640.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def workload(T, IN, osl, S, R, choices, layout="uniform", seed=0, bad_slots=0.0, V=0, zero_y=False):
    spec = synth.multi_spec("multi_c4" if layout == "segments" else "multi_c5", T=T, IN=IN, out_slices=osl,
                            S=S, R=R, rank_choices=choices, V=V)
    w = synth.make_multi(spec, seed=seed, device=DEV)
    if bad_slots:
        g = torch.Generator().manual_seed(seed + 99)
        pick = torch.rand(T, generator=g) < bad_slots
        bad = torch.where(torch.rand(T, generator=g) < 0.5, torch.full((T,), -1), torch.full((T,), S + 3))
        w["slots"] = torch.where(pick.to(DEV), bad.to(DEV, torch.int32), w["slots"])
    if zero_y:
        w["y0"].zero_()
    return w


def active_mask(w):
    slots = w["slots"].cpu().numpy()
    ranks = w["ranks"].cpu().numpy()
    S, R = ranks.shape[0], w["R"]
    return np.array([0 <= s < S and 1 <= ranks[s] <= R for s in slots])


def padded_y(y0, row_pad=2, col_pad=8):
    T, O_ = y0.shape
    buf = torch.full((T + row_pad, O_ + col_pad), SENT, dtype=y0.dtype, device=y0.device)
    buf[:T, :O_] = y0
    return buf[:T, :O_], buf


def check_y(w, y, buf, ref):
    T, O_ = y.shape
    act = active_mask(w)
    got = f64(y)
    assert rel_err(got[act], ref[act]) <= TOL_BF16
    # inactive rows, padding rows and columns: untouched, bit for bit
    y0 = f64(w["y0"])
    assert np.array_equal(got[~act], y0[~act])
    b = buf.float().cpu()
    assert torch.all(b[T:, :] == SENT) and torch.all(b[:, O_:] == SENT)


def spec_mask(w, n):
    """[T, n*R] mask of the entries of h that the page specifies."""
    act = active_mask(w)
    slots = w["slots"].cpu().numpy()
    ranks = w["ranks"].cpu().numpy()
    R = w["R"]
    m = np.zeros((len(slots), n * R), bool)
    for t in np.nonzero(act)[0]:
        for i in range(n):
            m[t, i * R:i * R + ranks[slots[t]]] = True
    return m


def run_group(w):
    T = w["slots"].numel()
    S = w["ranks"].numel()
    counts = torch.full((S,), -5, dtype=torch.int32, device=DEV)
    perm = torch.full((max(T, 1),), -5, dtype=torch.int32, device=DEV)
    na = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    lora.lora_group_by_slot(w["slots"], w["ranks"], w["R"], counts, perm, na)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), perm.cpu().numpy(), int(na.item())


CASES = [  # T, IN, out_slices, S, R, rank choices, layout
    (1, 64, [64], 1, 8, [8], "uniform"),
    (5, 72, [24], 3, 16, [0, 8, 16], "uniform"),
    (37, 200, [40, 16], 4, 16, [0, 8, 16], "uniform"),
    (130, 128, [128, 32, 32], 6, 32, [0, 8, 16, 32], "segments"),
    (300, 520, [136], 9, 64, [8, 16, 32, 64], "uniform"),
    (257, 96, [64, 64], 5, 64, [0, 16, 64], "segments"),
    (200, 64, [72], 3, 128, [0, 40, 128], "uniform"),
    (90, 136, [64], 4, 24, [0, 8, 24], "uniform"),
    # decode-shaped batches (at most four tokens per slot on average)
    (64, 256, [128, 64], 32, 64, [8, 16, 32, 64], "uniform"),
    (200, 520, [136], 64, 32, [0, 8, 16, 24, 32], "uniform"),
    (100, 72, [24, 40], 40, 16, [0, 8, 16], "uniform"),
    (9, 1000, [256], 9, 128, [0, 40, 128], "uniform"),
    # decode-shaped, `in` a multiple of 64: a ragged last 256-column chunk, two and
    # four 64-row blocks of adapter rows, one token over many slots
    (200, 576, [136], 64, 32, [0, 8, 16, 24, 32], "uniform"),
    (9, 1024, [256], 9, 128, [0, 40, 128], "uniform"),
    (60, 320, [64, 64, 64, 64], 20, 64, [0, 8, 64], "uniform"),
    (1, 8192, [64], 40, 64, [64], "uniform"),
]


@pytest.mark.parametrize("T,IN,osl,S,R,ch,layout", CASES)
def test_group_by_slot_bit_exact(T, IN, osl, S, R, ch, layout):
    w = workload(T, IN, osl, S, R, ch, layout, seed=T, bad_slots=0.1)
    counts, perm, na = run_group(w)
    rc, rp = O.group_by_slot(w["slots"].cpu().numpy(), w["ranks"].cpu().numpy(), R)
    assert counts.tolist() == rc.tolist()
    assert na == len(rp) and perm[:na].tolist() == rp.tolist()


@pytest.mark.parametrize("T,S", [(4096, 32), (8192, 128), (70000, 7), (3000, 4096), (1, 1)])
def test_group_by_slot_large(T, S):
    g = torch.Generator().manual_seed(T + S)
    slots = torch.randint(-2, S + 2, (T,), generator=g, dtype=torch.int32)
    ranks = torch.randint(0, 66, (S,), generator=g, dtype=torch.int32)
    w = dict(slots=slots.to(DEV), ranks=ranks.to(DEV), R=64)
    counts, perm, na = run_group(w)
    rc, rp = O.group_by_slot(slots.numpy(), ranks.numpy(), 64)
    assert counts.tolist() == rc.tolist()
    assert na == len(rp) and perm[:na].tolist() == rp.tolist()


def oracle_inputs(w):
    return dict(x=f64(w["x"]), a=f64(w["a"]), b=f64(w["b"]), y0=f64(w["y0"]),
                slots=w["slots"].cpu().numpy(), ranks=w["ranks"].cpu().numpy(),
                scal=w["scalings"].double().cpu().numpy())


@pytest.mark.parametrize("T,IN,osl,S,R,ch,layout", CASES)
def test_shrink(T, IN, osl, S, R, ch, layout):
    w = workload(T, IN, osl, S, R, ch, layout, seed=T + 1, bad_slots=0.05)
    n = len(osl)
    h = torch.full((T, n * R), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_shrink(w["x"], w["a"], w["slots"], w["ranks"], R, h, num_slices=n)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    o = oracle_inputs(w)
    ref = O.shrink(o["x"], o["a"], o["slots"], o["ranks"], R, n)
    m = spec_mask(w, n)
    got = f64(h)
    assert np.all(np.isfinite(got[m]))
    assert rel_err(got[m], ref[m]) <= TOL_F32


@pytest.mark.parametrize("T,IN,osl,S,R,ch,layout", CASES)
def test_expand(T, IN, osl, S, R, ch, layout):
    w = workload(T, IN, osl, S, R, ch, layout, seed=T + 2, bad_slots=0.05)
    n = len(osl)
    o = oracle_inputs(w)
    href = O.shrink(o["x"], o["a"], o["slots"], o["ranks"], R, n)
    # h given to the GPU: NaN wherever the page leaves it unspecified
    hin = np.where(spec_mask(w, n), href, np.nan).astype(np.float32)
    h = torch.from_numpy(hin).to(DEV)
    y, buf = padded_y(w["y0"])
    lora.lora_expand(h, w["b"], w["slots"], w["ranks"], w["scalings"], y, osl, R)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    ref = O.expand(hin.astype(np.float64), o["b"], o["slots"], o["ranks"], o["scal"], o["y0"], osl, R)
    check_y(w, y, buf, ref)


@pytest.mark.parametrize("T,IN,osl,S,R,ch,layout", CASES)
def test_apply_linear(T, IN, osl, S, R, ch, layout):
    w = workload(T, IN, osl, S, R, ch, layout, seed=T + 3, bad_slots=0.05)
    o = oracle_inputs(w)
    y, buf = padded_y(w["y0"])
    lora.lora_apply_linear(w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"], y, osl, R)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    ref = O.apply_linear(o["x"], o["a"], o["b"], o["slots"], o["ranks"], o["scal"], o["y0"], osl, R)
    check_y(w, y, buf, ref)


def test_apply_linear_delta_alone():
    """y0 = 0: the tolerance applies to the LoRA delta itself."""
    w = workload(300, 256, [128, 64, 64], 8, 64, [0, 8, 16, 32, 64], "segments", seed=7, zero_y=True)
    o = oracle_inputs(w)
    y = w["y0"].clone()
    lora.lora_apply_linear(w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"], y, [128, 64, 64], 64)
    torch.cuda.synchronize()
    ref = O.apply_linear(o["x"], o["a"], o["b"], o["slots"], o["ranks"], o["scal"], o["y0"], [128, 64, 64], 64)
    act = active_mask(w)
    assert rel_err(f64(y)[act], ref[act]) <= TOL_BF16


@pytest.mark.parametrize("T,V,S,R", [(1, 10, 1, 8), (64, 300, 5, 16), (257, 1000, 9, 64), (100, 77, 3, 128)])
def test_gather_shrink_bit_exact(T, V, S, R):
    w = workload(T, 64, [64], S, R, sorted({8, R // 2, R} - {0}), "uniform", seed=V, V=V, bad_slots=0.1)
    h = torch.full((T, R), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_gather_shrink(w["ids"], w["ga"], w["slots"], w["ranks"], R, h)
    torch.cuda.synchronize()
    ref = O.gather_shrink(w["ids"].cpu().numpy(), f64(w["ga"]), w["slots"].cpu().numpy(),
                          w["ranks"].cpu().numpy(), R)
    m = spec_mask(w, 1)
    got = f64(h)
    assert np.array_equal(got[m], ref[m])


def test_shrink_expand_equals_apply():
    """apply_linear and shrink followed by expand give the same y within the bf16
    tolerance (h is fp32 in both)."""
    w = workload(500, 128, [64, 32], 6, 32, [0, 8, 16, 32], "segments", seed=11)
    h = torch.zeros((500, 64), dtype=torch.float32, device=DEV)
    lora.lora_shrink(w["x"], w["a"], w["slots"], w["ranks"], 32, h, num_slices=2)
    y1 = w["y0"].clone()
    lora.lora_expand(h, w["b"], w["slots"], w["ranks"], w["scalings"], y1, [64, 32], 32)
    y2 = w["y0"].clone()
    lora.lora_apply_linear(w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"], y2, [64, 32], 32)
    torch.cuda.synchronize()
    assert rel_err(f64(y1), f64(y2)) <= TOL_BF16


def test_repeatable_bitwise_multi():
    w = workload(700, 256, [128, 64], 12, 64, [0, 8, 16, 32, 64], "segments", seed=12)
    outs = []
    for _ in range(2):
        y = w["y0"].clone()
        lora.lora_apply_linear(w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"], y, [128, 64], 64)
        outs.append(y)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("T,S,R,osl", [(1, 1, 8, [64]), (2, 2, 16, [24]), (5, 3, 16, [256, 40]), (9, 9, 64, [512])])
def test_expand_tiny_batches_each_unit_once(T, S, R, osl):
    """Decode batches whose split cost is below the grid size: with y0 = 0 a unit
    that two CTAs both add into shows as a doubled delta.  Whether two such
    read-modify-writes interleave depends on timing, so the expand runs many
    times; every run must give the oracle's y, bit-identical to the first."""
    w = workload(T, 64, osl, S, R, [R], "uniform", seed=T + 40, zero_y=True)
    n = len(osl)
    o = oracle_inputs(w)
    href = O.shrink(o["x"], o["a"], o["slots"], o["ranks"], R, n)
    h = torch.from_numpy(href.astype(np.float32)).to(DEV)
    ref = O.expand(href.astype(np.float32).astype(np.float64), o["b"], o["slots"], o["ranks"], o["scal"],
                   o["y0"], osl, R)
    outs = []
    for _ in range(40):
        y = torch.zeros_like(w["y0"])
        lora.lora_expand(h, w["b"], w["slots"], w["ranks"], w["scalings"], y, osl, R)
        outs.append(y)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    assert rel_err(f64(outs[0]), ref) <= TOL_BF16
    for y in outs[1:]:
        assert torch.equal(y, outs[0])


def test_c4_prefill_full():
    """The prefill workload at full size: T = 4096, fused QKV [4096, 1024, 1024]."""
    spec = synth.multi_spec("multi_c4")
    w = synth.make_multi(spec, seed=0, device=DEV)
    R, osl = spec["R"], spec["out_slices"]
    o = oracle_inputs(w)
    h = torch.full((spec["T"], 3 * R), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_shrink(w["x"], w["a"], w["slots"], w["ranks"], R, h, num_slices=3)
    y, buf = padded_y(w["y0"])
    lora.lora_apply_linear(w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"], y, osl, R)
    y2 = w["y0"].clone()
    lora.lora_expand(h, w["b"], w["slots"], w["ranks"], w["scalings"], y2, osl, R)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    href = O.shrink(o["x"], o["a"], o["slots"], o["ranks"], R, 3)
    m = spec_mask(w, 3)
    assert rel_err(f64(h)[m], href[m]) <= TOL_F32
    ref = O.apply_linear(o["x"], o["a"], o["b"], o["slots"], o["ranks"], o["scal"], o["y0"], osl, R)
    check_y(w, y, buf, ref)
    act = active_mask(w)
    assert rel_err(f64(y2)[act], ref[act]) <= TOL_BF16


def test_c5_decode_full():
    """The decode workload at full size (T = 256 over 128 slots, in = out = 8192,
    R = 64): lora_shrink, lora_expand and lora_apply_linear each against the
    oracle, every element; the expand is fed the oracle's h with NaN wherever the
    page leaves h unspecified, and also checked on its delta alone (y0 = 0)."""
    spec = synth.multi_spec("multi_c5", V=0)
    w = synth.make_multi(spec, seed=0, device=DEV)
    R, osl, T = spec["R"], spec["out_slices"], spec["T"]
    o = oracle_inputs(w)
    h = torch.full((T, R), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_shrink(w["x"], w["a"], w["slots"], w["ranks"], R, h, num_slices=1)
    y, buf = padded_y(w["y0"])
    lora.lora_apply_linear(w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"], y, osl, R)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    href = O.shrink(o["x"], o["a"], o["slots"], o["ranks"], R, 1)
    m = spec_mask(w, 1)
    got = f64(h)
    assert np.all(np.isfinite(got[m])) and rel_err(got[m], href[m]) <= TOL_F32
    ref = O.apply_linear(o["x"], o["a"], o["b"], o["slots"], o["ranks"], o["scal"], o["y0"], osl, R)
    check_y(w, y, buf, ref)
    hin = np.where(m, href, np.nan).astype(np.float32)
    for zero in (False, True):
        y0 = torch.zeros_like(w["y0"]) if zero else w["y0"]
        y2, buf2 = padded_y(y0)
        lora.lora_expand(torch.from_numpy(hin).to(DEV), w["b"], w["slots"], w["ranks"], w["scalings"], y2, osl, R)
        torch.cuda.synchronize()
        assert lora.lora_device_error() == 0
        ref2 = O.expand(hin.astype(np.float64), o["b"], o["slots"], o["ranks"], o["scal"], f64(y0), osl, R)
        check_y(dict(w, y0=y0), y2, buf2, ref2)


def test_c5_gather_every_token():
    """The decode gather at full size: a [128, 64, 128256] bf16, ids uniform in
    [0, 128256) with 5% = -1; every token's row is compared bit for bit with the
    oracle (run slot by slot on that slot's table)."""
    spec = synth.multi_spec("multi_c5")
    w = synth.make_multi(spec, seed=0, device=DEV)
    R, T = spec["R"], spec["T"]
    hg = torch.full((T, R), float("nan"), dtype=torch.float32, device=DEV)
    lora.lora_gather_shrink(w["ids"], w["ga"], w["slots"], w["ranks"], R, hg)
    torch.cuda.synchronize()
    assert lora.lora_device_error() == 0
    slots = w["slots"].cpu().numpy()
    ranks = w["ranks"].cpu().numpy()
    ids = w["ids"].cpu().numpy()
    got = f64(hg)
    m = spec_mask(w, 1)
    assert (ids < 0).any() and m.any()
    checked = 0
    for s in np.unique(slots):
        toks = np.nonzero(slots == s)[0]
        one = O.gather_shrink(ids[toks], f64(w["ga"][s:s + 1]), np.zeros(len(toks), np.int32),
                              ranks[s:s + 1], R)
        assert np.array_equal(got[toks][m[toks]], one[m[toks]])
        checked += len(toks)
    assert checked == T


@pytest.mark.parametrize("T,IN,osl,S,R,ch,layout", [CASES[3], CASES[4], CASES[8], CASES[10], CASES[11], CASES[12],
                                                     CASES[14]])
def test_prebuilt_schedule_same_bits(T, IN, osl, S, R, ch, layout):
    """A schedule built once (lora_build_schedule) and passed in the addressing
    gives bit-for-bit the results of the ops that group the tokens themselves,
    and the same y as the oracle."""
    w = workload(T, IN, osl, S, R, ch, layout, seed=T + 5, bad_slots=0.05)
    n = len(osl)
    sched = lora.lora_build_schedule(w["slots"], w["ranks"], R)
    outs = {}
    for tag, sc in (("own", None), ("pre", sched)):
        h = torch.full((T, n * R), float("nan"), dtype=torch.float32, device=DEV)
        lora.lora_shrink(w["x"], w["a"], w["slots"], w["ranks"], R, h, num_slices=n, schedule=sc)
        y1 = w["y0"].clone()
        lora.lora_expand(h, w["b"], w["slots"], w["ranks"], w["scalings"], y1, osl, R, schedule=sc)
        y2 = w["y0"].clone()
        lora.lora_apply_linear(w["x"], w["a"], w["b"], w["slots"], w["ranks"], w["scalings"], y2, osl, R,
                               schedule=sc)
        torch.cuda.synchronize()
        outs[tag] = (h, y1, y2)
    assert lora.lora_device_error() == 0
    m = torch.from_numpy(spec_mask(w, n)).to(DEV)
    assert torch.equal(outs["own"][0][m], outs["pre"][0][m])
    assert torch.equal(outs["own"][1], outs["pre"][1]) and torch.equal(outs["own"][2], outs["pre"][2])
    o = oracle_inputs(w)
    ref = O.apply_linear(o["x"], o["a"], o["b"], o["slots"], o["ranks"], o["scal"], o["y0"], osl, R)
    act = active_mask(w)
    assert rel_err(f64(outs["pre"][2])[act], ref[act]) <= TOL_BF16


def test_prebuilt_schedule_holds_the_grouping():
    """The schedule's permutation and counts are lora_group_by_slot's (the oracle's stable sort)."""
    w = workload(3000, 64, [64], 40, 64, [0, 8, 16, 64], "segments", seed=3, bad_slots=0.1)
    sched = lora.lora_build_schedule(w["slots"], w["ranks"], 64)
    torch.cuda.synchronize()
    raw = sched.cpu().numpy()
    S, T = 40, 3000
    rc, rp = O.group_by_slot(w["slots"].cpu().numpy(), w["ranks"].cpu().numpy(), 64)
    # layout: header (256 B), counts [S] (256-byte rounded), perm [T]
    header = raw[:256].view(np.int32)
    counts = raw[256:256 + 4 * S].view(np.int32)
    off = 256 + ((4 * S + 255) // 256) * 256
    perm = raw[off:off + 4 * T].view(np.int32)
    assert header[0] == len(rp)
    assert counts.tolist() == rc.tolist() and perm[:len(rp)].tolist() == rp.tolist()
