"""Helpers shared by the tests (no method arithmetic here)."""
import re
import os

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TOL_BF16 = 8e-3   # max|gpu - oracle| / max|oracle| for bf16 outputs
TOL_F32 = 1e-4    # ... for fp32 outputs


def f64(t):
    """Exact fp64 copy of a tensor (bf16/fp32 widen without rounding)."""
    return t.detach().to("cpu").double().numpy()


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    m = float(np.max(np.abs(ref)))
    d = float(np.max(np.abs(got - ref)))
    return d / m if m > 0 else d


def header_functions():
    """Names of the functions declared in include/lora.h."""
    with open(os.path.join(ROOT, "include", "lora.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"^LORA_API\s+[\w\s\*]+?\b(lora_\w+)\s*\(", src, re.M)))


def cuda_ok():
    return torch.cuda.is_available()
