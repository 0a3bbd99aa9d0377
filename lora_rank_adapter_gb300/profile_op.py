"""Runs one library op a few times on seeded inputs, for profilers (ncu).

  python -m lora_rank_adapter_gb300.profile_op --config c3_down --op lora_backward --M 4096 --reps 3

--config names a single-adapter workload (c1, c2, c3_up, c3_down) or a
multi-adapter one (c4, c5); --M (single) / --T (multi) shrinks the token count
so that a capture stays small.  Every launch goes through the C ABI like any
user call; the op's results are not checked here (the tests do that).
"""
import argparse

import torch

from lora_rank_adapter_gb300 import _build
from lora_rank_adapter_gb300 import binding
from lora_rank_adapter_gb300 import synth

SINGLE = {"c1": "single_c1", "c2": "single_c2", "c3_up": "single_c3_up", "c3_down": "single_c3_down"}
MULTI = {"c4": "multi_c4", "c5": "multi_c5"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", required=True, choices=sorted(SINGLE) + sorted(MULTI))
    ap.add_argument("--op", required=True)
    ap.add_argument("--M", type=int, default=0, help="tokens of a single-adapter workload (0: full)")
    ap.add_argument("--T", type=int, default=0, help="tokens of a multi-adapter workload (0: full)")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    _build.build()
    dev = "cuda:0"
    torch.cuda.set_device(0)
    L = binding
    if args.config in SINGLE:
        over = {"M": args.M} if args.M else {}
        spec = synth.single_spec(SINGLE[args.config], **over)
        w = synth.make_single(spec, seed=0, device=dev)
        X, A, B, Y, dY = w["X"], w["A"].t().contiguous().t(), w["B"].t().contiguous().t(), w["Y0"], w["dY"]
        M, K = X.shape
        r, Lc = B.shape
        s = spec["s"]
        h = torch.empty((M, r), dtype=torch.float32, device=dev)
        dX = torch.empty_like(X)
        dA = torch.empty((K, r), dtype=torch.float32, device=dev)
        dB = torch.empty((r, Lc), dtype=torch.float32, device=dev)
        L.lora_forward_h(X, A, B, Y, s, h)
        fns = {
            "lora_forward": lambda: L.lora_forward(X, A, B, Y, s),
            "lora_forward_h": lambda: L.lora_forward_h(X, A, B, Y, s, h),
            "lora_backward": lambda: L.lora_backward(X, dY, A, B, h, s, dX, dA, dB),
            "lora_backward_dx_da": lambda: L.lora_backward_dx_da(X, dY, A, B, s, dX, dA),
            "lora_backward_db": lambda: L.lora_backward_db(X, A, dY, s, dB),
        }
    else:
        over = {"T": args.T} if args.T else {}
        spec = synth.multi_spec(MULTI[args.config], **over)
        m = synth.make_multi(spec, seed=0, device=dev)
        R, osl, T = spec["R"], spec["out_slices"], spec["T"]
        h = torch.zeros((T, len(osl) * R), dtype=torch.float32, device=dev)
        y = m["y0"]
        fns = {
            "lora_shrink": lambda: L.lora_shrink(m["x"], m["a"], m["slots"], m["ranks"], R, h, num_slices=len(osl)),
            "lora_expand": lambda: L.lora_expand(h, m["b"], m["slots"], m["ranks"], m["scalings"], y, osl, R),
            "lora_apply_linear": lambda: L.lora_apply_linear(m["x"], m["a"], m["b"], m["slots"], m["ranks"],
                                                             m["scalings"], y, osl, R),
        }
        if "ga" in m:
            hg = torch.zeros((T, R), dtype=torch.float32, device=dev)
            fns["lora_gather_shrink"] = lambda: L.lora_gather_shrink(m["ids"], m["ga"], m["slots"], m["ranks"], R, hg)
    if args.op not in fns:
        raise SystemExit(f"unknown op {args.op}; known: {sorted(fns)}")
    torch.cuda.synchronize()
    for _ in range(args.reps):
        fns[args.op]()
    torch.cuda.synchronize()
    assert L.lora_device_error() == 0
    print(f"ran {args.op} on {args.config} x{args.reps}")


if __name__ == "__main__":
    main()
