"""Seeded synthetic inputs for the LoRA adapter-product workloads.

This module only draws random numbers and lays out inputs; it contains none of
the adapter arithmetic.  The same tensors feed both the CUDA library and the
fp64 oracle used by the tests, so both sides always see identical values.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser as published by Vigna),
used counter-style: draw i of a stream with base state g is mix(g + (i+1)*gamma),
which is exactly the i-th output of a SplitMix64 seeded with g.  Uniforms take
the top 53 bits; normals use the Box-Muller transform on two uniforms.  Every
named tensor gets its own stream, derived from (seed, name), so a tensor's
values do not depend on which other tensors were drawn.  The integer part runs
in torch int64 (wrapping arithmetic, logical shifts by masking) on any device,
so large inputs are generated on the GPU; values are then rounded to the
storage dtype (bf16 or fp32) by torch's round-to-nearest-even conversion.

Workloads (the five synthetic configurations of the LoRA benchmark):
  single_c1  fp32  M=256   K=512   L=512   r=8   s=2
  single_c2  bf16  M=8192  K=4096  L=4096  r=16  s=2      (q_proj, batch 4 x seq 2048)
  single_c3_up / single_c3_down  bf16  M=16384, r=64, s=0.5, 4096<->14336
  multi_c4   prefill: T=4096, in=4096, out_slices [4096,1024,1024], 32 slots
  multi_c5   decode:  T=256, 128 slots, in=out=8192, plus a 128256-wide gather
Normal parameters are standard deviations.  Padding of the adapter stacks
(rows/columns past a slot's rank, whole rank-0 slots) and the scalings of
rank-0 slots are filled with NaN so that any read of them shows up.
"""
import hashlib
import math

import torch

_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def _s64(c):
    """Signed int64 value with the same bits as the unsigned constant c."""
    c &= _MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def _lsr(z, k):
    """Logical right shift of an int64 tensor."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix_t(z):
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def mix64(z):
    """The SplitMix64 finaliser on a Python int (reference for tests)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def splitmix64_sequence(seed, n):
    """The first n outputs of a plain SplitMix64 seeded with `seed` (Python ints)."""
    out, state = [], seed & _MASK64
    for _ in range(n):
        state = (state + _GAMMA) & _MASK64
        out.append(mix64(state))
    return out


def stream_base(seed, name):
    """Base state of the stream for tensor `name` under `seed`."""
    h = int.from_bytes(hashlib.blake2b(name.encode(), digest_size=8).digest(), "little")
    return mix64((seed * _GAMMA) ^ h)


def bits(base, start, n, device="cpu"):
    """Draws start .. start+n-1 of the stream with base state `base` (int64 tensor)."""
    idx = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    return _mix_t(idx * _s64(_GAMMA) + _s64(base))


def _uniform01(base, start, n, device):
    return _lsr(bits(base, start, n, device), 11).to(torch.float64) * (2.0 ** -53)


_CHUNK = 1 << 24


def _fill(shape, device, fn):
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.float64, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = fn(s, e - s)
    return out.view(*shape)


def uniform64(shape, lo, hi, seed, name, device="cpu"):
    base = stream_base(seed, name)
    return _fill(shape, device, lambda s, n: lo + (hi - lo) * _uniform01(base, s, n, device))


def normal64(shape, std, seed, name, device="cpu", mean=0.0):
    base = stream_base(seed, name)

    def chunk(s, n):
        u1 = 1.0 - _uniform01(base, 2 * s, n, device)           # (0, 1]
        u2 = _uniform01(base, 2 * s + n, n, device)
        return mean + std * torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)

    # each chunk uses its own block of 2n draws starting at 2s
    return _fill(shape, device, chunk)


def uniform_int(n, low, high, seed, name, device="cpu"):
    """n integers uniform in [low, high)."""
    base = stream_base(seed, name)
    u = _uniform01(base, 0, n, device)
    return (low + torch.floor(u * (high - low))).to(torch.int64).clamp_(low, high - 1)


_TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def draw(spec, shape, seed, name, dtype, device="cpu"):
    """A tensor of `dtype` ('bf16' or 'f32') drawn from spec = ('normal', std) or
    ('uniform', lo, hi)."""
    if spec[0] == "normal":
        v = normal64(shape, spec[1], seed, name, device)
    elif spec[0] == "uniform":
        v = uniform64(shape, spec[1], spec[2], seed, name, device)
    elif spec[0] == "zeros":
        v = torch.zeros(shape, dtype=torch.float64, device=device)
    else:
        raise ValueError(spec)
    return v.to(_TORCH_DT[dtype])


# --------------------------------------------------------------------------- single adapter
SINGLE = {
    "single_c1": dict(dtype="f32", M=256, K=512, L=512, r=8, s=2.0,
                      X=("normal", 1.0), A=("uniform", -1 / math.sqrt(512), 1 / math.sqrt(512)),
                      B=("normal", 0.02), Y0=("normal", 1.0), dY=("normal", 1.0)),
    "single_c2": dict(dtype="bf16", M=8192, K=4096, L=4096, r=16, s=2.0,
                      X=("normal", 1.0), A=("uniform", -1 / 64, 1 / 64),
                      B=("normal", 0.02), Y0=("normal", 1.0), dY=("normal", 1e-2)),
    "single_c3_up": dict(dtype="bf16", M=16384, K=4096, L=14336, r=64, s=0.5,
                         X=("normal", 1.0), A=("uniform", -1 / 64, 1 / 64),
                         B=("normal", 0.02), Y0=("normal", 1.0), dY=("normal", 1e-2)),
    "single_c3_down": dict(dtype="bf16", M=16384, K=14336, L=4096, r=64, s=0.5,
                           X=("normal", 1.0),
                           A=("uniform", -1 / math.sqrt(14336), 1 / math.sqrt(14336)),
                           B=("normal", 0.02), Y0=("normal", 1.0), dY=("normal", 1e-2)),
}


def single_spec(name, **over):
    """The named single-adapter workload, with any field overridden."""
    spec = dict(SINGLE[name])
    spec.update(over)
    return spec


def make_single(spec, seed=0, device="cpu", prefix=None):
    """Inputs of one single-adapter workload in their logical shapes:
    X [M,K], A [K,r], B [r,L], Y0 [M,L], dY [M,L] (storage dtype)."""
    p = prefix or "single"
    M, K, L, r, dt = spec["M"], spec["K"], spec["L"], spec["r"], spec["dtype"]
    return dict(
        X=draw(spec["X"], (M, K), seed, p + ".X", dt, device),
        A=draw(spec["A"], (K, r), seed, p + ".A", dt, device),
        B=draw(spec["B"], (r, L), seed, p + ".B", dt, device),
        Y0=draw(spec["Y0"], (M, L), seed, p + ".Y0", dt, device),
        dY=draw(spec["dY"], (M, L), seed, p + ".dY", dt, device),
    )


# --------------------------------------------------------------------------- multi adapter
MULTI = {
    # prefill: contiguous segments of Geometric(1/128) length, 10% on the zero adapter
    "multi_c4": dict(T=4096, IN=4096, out_slices=[4096, 1024, 1024], S=32, R=64,
                     rank_choices=[0, 8, 16, 32, 64], zero_slot_frac=0.1, seg_p=1 / 128,
                     layout="segments"),
    # decode: each token on a uniform random slot among 128
    "multi_c5": dict(T=256, IN=8192, out_slices=[8192], S=128, R=64,
                     rank_choices=[8, 16, 32, 64], layout="uniform", V=128256, ids_invalid=0.05),
}


def multi_spec(name, **over):
    spec = dict(MULTI[name])
    spec.update(over)
    return spec


def _slots_segments(spec, seed):
    T, S = spec["T"], spec["S"]
    p = spec["seg_p"]
    base_len = stream_base(seed, "multi.seglen")
    base_slot = stream_base(seed, "multi.segslot")
    slots, i, t = [], 0, 0
    while t < T:
        u = float(_uniform01(base_len, i, 1, "cpu")[0])
        length = max(1, int(math.ceil(math.log1p(-u) / math.log1p(-p)))) if u > 0 else 1
        v = _uniform01(base_slot, 2 * i, 2, "cpu")
        if float(v[0]) < spec["zero_slot_frac"] or S == 1:
            s = 0
        else:
            s = 1 + min(S - 2, int(float(v[1]) * (S - 1)))
        length = min(length, T - t)
        slots += [s] * length
        t += length
        i += 1
    return torch.tensor(slots, dtype=torch.int32)


def make_multi(spec, seed=0, device="cpu", poison=True):
    """Inputs of one multi-adapter workload:
    slots [T] i32, ranks [S] i32, scalings [S] f32, x [T,IN] bf16, a [S,n*R,IN] bf16,
    b [S,O,R] bf16, y0 [T,O] bf16; for the decode workload also the gather table
    ga [S,R,V] bf16 and ids [T] i64 (spec["V"] > 0)."""
    T, IN, S, R = spec["T"], spec["IN"], spec["S"], spec["R"]
    osl = list(spec["out_slices"])
    n, O = len(osl), sum(osl)
    choices = spec["rank_choices"]
    ri = uniform_int(S, 0, len(choices), seed, "multi.rank")
    ranks = torch.tensor([choices[int(k)] for k in ri], dtype=torch.int32)
    if spec["layout"] == "segments":
        ranks[0] = 0                                  # slot 0 is the zero adapter
        slots = _slots_segments(spec, seed)
    else:
        slots = uniform_int(T, 0, S, seed, "multi.slot").to(torch.int32)
    scal = torch.full((S,), float("nan"), dtype=torch.float32)
    for s in range(S):
        if ranks[s] > 0:
            scal[s] = 16.0 / float(ranks[s])
    x = draw(("normal", 1.0), (T, IN), seed, "multi.x", "bf16", device)
    y0 = draw(("normal", 1.0), (T, O), seed, "multi.y0", "bf16", device)
    a = draw(("normal", 0.02), (S, n * R, IN), seed, "multi.a", "bf16", device)
    b = draw(("normal", 0.02), (S, O, R), seed, "multi.b", "bf16", device)
    if poison:
        rk = ranks.to(device)
        jj = torch.arange(R, device=device)
        pad = jj[None, :] >= rk[:, None]                          # [S, R]
        a.view(S, n, R, IN).masked_fill_(pad[:, None, :, None], float("nan"))
        b.masked_fill_(pad[:, None, :], float("nan"))
    out = dict(slots=slots.to(device), ranks=ranks.to(device), scalings=scal.to(device),
               x=x, a=a, b=b, y0=y0, out_slices=osl, R=R, IN=IN, T=T, S=S)
    V = spec.get("V", 0)
    if V:
        ga = torch.empty((S, R, V), dtype=torch.bfloat16, device=device)
        flat = ga.view(-1)
        base = stream_base(seed, "multi.ga")
        for st in range(0, flat.numel(), _CHUNK):
            e = min(flat.numel(), st + _CHUNK)
            nn = e - st
            u1 = 1.0 - _uniform01(base, 2 * st, nn, device)
            u2 = _uniform01(base, 2 * st + nn, nn, device)
            flat[st:e] = (0.02 * torch.sqrt(-2.0 * torch.log(u1))
                          * torch.cos((2.0 * math.pi) * u2)).to(torch.bfloat16)
        if poison:
            rk = ranks.to(device)
            pad = torch.arange(R, device=device)[None, :] >= rk[:, None]
            ga.masked_fill_(pad[:, :, None], float("nan"))
        ids = uniform_int(T, 0, V, seed, "multi.ids", device)
        bad = _uniform01(stream_base(seed, "multi.ids_bad"), 0, T, device) < spec["ids_invalid"]
        ids = torch.where(bad, torch.full_like(ids, -1), ids)
        out.update(ga=ga, ids=ids, V=V)
    return out
