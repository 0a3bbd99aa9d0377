"""PyTorch integration of liblora.so: custom ops and autograd.

The multi-adapter ops are registered as torch.library custom ops so that
torch.compile sees each as one opaque node, as the mstar page
"mstar.engine.resources.lora.ops" describes for its own ops: `expand_`,
`apply_linear_` and `forward_` add into their output in place and declare it
(mutates_args), so functionalization keeps every read of it ordered around the
add.  Each op has a fake (shape-only) implementation that runs without a GPU and
a CUDA implementation that calls the C ABI; there is no CPU kernel.

`LoraLinearFn` / `lora_linear` is an autograd.Function over the single-adapter
ops (NeMo AutoModel page "nemo_automodel.components._peft.lora_kernel":
lora_forward_wrapper, lora_da_dx_update_wrapper, lora_db_update_wrapper), on
the fused pair forward_h_ / backward_ex:
    out = base + scale * (x @ A) @ B
with gradients dx = scale * dout @ B^T @ A^T, dA = scale * x^T @ (dout @ B^T),
dB = scale * (x @ A)^T @ dout and dbase = dout.
"""
from typing import List, Sequence

import torch

from . import binding

NS = "lora_gb300"


def _slots_list(out_slices: Sequence[int]) -> List[int]:
    return [int(v) for v in out_slices]


# ----------------------------------------------------------------------------- multi adapter
@torch.library.custom_op(f"{NS}::shrink", mutates_args=(), device_types="cuda")
def shrink(x: torch.Tensor, a: torch.Tensor, slots: torch.Tensor, ranks: torch.Tensor,
           max_rank: int, num_slices: int) -> torch.Tensor:
    """h[t, i*R + j] = x[t] . a[slot(t), i*R + j] (fp32; unspecified past the rank)."""
    h = torch.zeros((x.shape[0], num_slices * max_rank), dtype=torch.float32, device=x.device)
    binding.lora_shrink(x, a, slots, ranks, max_rank, h, num_slices=num_slices)
    return h


@shrink.register_fake
def _(x, a, slots, ranks, max_rank, num_slices):
    return x.new_empty((x.shape[0], num_slices * max_rank), dtype=torch.float32)


@torch.library.custom_op(f"{NS}::expand_", mutates_args=("y",), device_types="cuda")
def expand_(y: torch.Tensor, h: torch.Tensor, b: torch.Tensor, slots: torch.Tensor, ranks: torch.Tensor,
            scalings: torch.Tensor, out_slices: List[int], max_rank: int) -> None:
    """y[t, slice i] += scalings[slot] * h[t, slice i] @ b[slot, slice i]^T, in place."""
    binding.lora_expand(h, b, slots, ranks, scalings, y, _slots_list(out_slices), max_rank)


@expand_.register_fake
def _(y, h, b, slots, ranks, scalings, out_slices, max_rank):
    return None


@torch.library.custom_op(f"{NS}::apply_linear_", mutates_args=("y",), device_types="cuda")
def apply_linear_(y: torch.Tensor, x: torch.Tensor, a: torch.Tensor, b: torch.Tensor, slots: torch.Tensor,
                  ranks: torch.Tensor, scalings: torch.Tensor, out_slices: List[int], max_rank: int) -> None:
    """Shrink then expand into y, in place."""
    binding.lora_apply_linear(x, a, b, slots, ranks, scalings, y, _slots_list(out_slices), max_rank)


@apply_linear_.register_fake
def _(y, x, a, b, slots, ranks, scalings, out_slices, max_rank):
    return None


@torch.library.custom_op(f"{NS}::gather_shrink", mutates_args=(), device_types="cuda")
def gather_shrink(ids: torch.Tensor, a: torch.Tensor, slots: torch.Tensor, ranks: torch.Tensor,
                  max_rank: int) -> torch.Tensor:
    """h[t, j] = a[slot(t), j, ids[t]] for j < rank; zeros for ids outside [0, V)."""
    h = torch.zeros((ids.shape[0], max_rank), dtype=torch.float32, device=ids.device)
    binding.lora_gather_shrink(ids, a, slots, ranks, max_rank, h)
    return h


@gather_shrink.register_fake
def _(ids, a, slots, ranks, max_rank):
    return a.new_empty((ids.shape[0], max_rank), dtype=torch.float32)


# ----------------------------------------------------------------------------- single adapter
@torch.library.custom_op(f"{NS}::forward_", mutates_args=("y",), device_types="cuda")
def forward_(y: torch.Tensor, x: torch.Tensor, A: torch.Tensor, B: torch.Tensor, scale: float) -> None:
    """y += scale * (x @ A) @ B, in place."""
    binding.lora_forward(x, A, B, y, scale)


@forward_.register_fake
def _(y, x, A, B, scale):
    return None


@torch.library.custom_op(f"{NS}::backward", mutates_args=(), device_types="cuda")
def backward(x: torch.Tensor, dout: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
             scale: float) -> List[torch.Tensor]:
    """(dx, dA, dB) of out = base + scale * (x @ A) @ B; dA and dB in fp32."""
    dx = torch.empty_like(x)
    dA = torch.empty(A.shape, dtype=torch.float32, device=x.device)
    dB = torch.empty(B.shape, dtype=torch.float32, device=x.device)
    binding.lora_backward_dx_da(x, dout, A, B, scale, dx, dA)
    binding.lora_backward_db(x, A, dout, scale, dB)
    return [dx, dA, dB]


@backward.register_fake
def _(x, dout, A, B, scale):
    return [torch.empty_like(x), A.new_empty(A.shape, dtype=torch.float32),
            B.new_empty(B.shape, dtype=torch.float32)]


@torch.library.custom_op(f"{NS}::forward_h_", mutates_args=("y",), device_types="cuda")
def forward_h_(y: torch.Tensor, x: torch.Tensor, A: torch.Tensor, B: torch.Tensor, scale: float) -> torch.Tensor:
    """y += scale * (x @ A) @ B in place; returns h = x @ A (fp32) for backward_ex."""
    h = torch.empty((x.shape[0], A.shape[1]), dtype=torch.float32, device=x.device)
    binding.lora_forward_h(x, A, B, y, scale, h)
    return h


@forward_h_.register_fake
def _(y, x, A, B, scale):
    return x.new_empty((x.shape[0], A.shape[1]), dtype=torch.float32)


@torch.library.custom_op(f"{NS}::backward_ex", mutates_args=(), device_types="cuda")
def backward_ex(x: torch.Tensor, dout: torch.Tensor, A: torch.Tensor, B: torch.Tensor, h: torch.Tensor,
                scale: float, grads_in_input_dtype: bool) -> List[torch.Tensor]:
    """(dx, dA, dB) in one call from the h that forward_h_ saved (x is read
    once); dA and dB in x's dtype when grads_in_input_dtype, else fp32."""
    gdt = x.dtype if grads_in_input_dtype else torch.float32
    dx = torch.empty_like(x)
    dA = torch.empty(A.shape, dtype=gdt, device=x.device)
    dB = torch.empty(B.shape, dtype=gdt, device=x.device)
    flags = binding.BWD_GRAD_INPUT_DTYPE if grads_in_input_dtype else 0
    binding.lora_backward_ex(x, dout, A, B, h, scale, dx, dA, dB, flags=flags)
    return [dx, dA, dB]


@backward_ex.register_fake
def _(x, dout, A, B, h, scale, grads_in_input_dtype):
    gdt = x.dtype if grads_in_input_dtype else torch.float32
    return [torch.empty_like(x), A.new_empty(A.shape, dtype=gdt), B.new_empty(B.shape, dtype=gdt)]


class LoraLinearFn(torch.autograd.Function):
    """out = base + scale * (x @ A) @ B on the GPU kernels: the forward saves
    h = x @ A, and the backward computes dx, dA and dB in one call from it (x is
    read once), returning dA and dB in the parameters' dtype (rounded once from
    the fp32 sums)."""

    @staticmethod
    def forward(ctx, x, A, B, base, scale):
        out = base.clone()
        h = forward_h_(out, x, A, B, float(scale))
        ctx.save_for_backward(x, A, B, h)
        ctx.scale = float(scale)
        return out

    @staticmethod
    def backward(ctx, dout):
        x, A, B, h = ctx.saved_tensors
        in_dtype = A.dtype == x.dtype and B.dtype == x.dtype
        dx, dA, dB = backward_ex(x, dout.contiguous(), A, B, h, ctx.scale, in_dtype)
        return dx, dA.to(A.dtype), dB.to(B.dtype), dout, None


def lora_linear(x: torch.Tensor, A: torch.Tensor, B: torch.Tensor, base: torch.Tensor, scale: float):
    """Differentiable out = base + scale * (x @ A) @ B (x [M,K], A [K,r], B [r,L], base [M,L])."""
    return LoraLinearFn.apply(x, A, B, base, scale)
