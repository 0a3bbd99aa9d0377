"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle/lora_oracle.c, plants one plausible slip (a transposed
operand, a sign, a dropped scale, a wrong index, a missed mask), builds it on
the CPU and runs the pins of tests/test_oracle_pins.py against it: at least one
pin has to fail.  The committed oracle itself is never modified.
"""
import os

import pytest

from oracle import oracle as O
from tests import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "lora_oracle.c")

MUTATIONS = [
    ("fwd_transposed_A", ") h[j] += xk * A[k * r + j];", ") h[j] += xk * A[j * K + k];"),
    ("fwd_sign", "Y[m * L + l] = Y0[m * L + l] + s * acc[l];", "Y[m * L + l] = Y0[m * L + l] - s * acc[l];"),
    ("fwd_index_B", "acc[l] += hj * B[j * L + l];", "acc[l] += hj * B[j * L + 0];"),
    ("dx_dropped_scale", "dX[m * K + k] = s * acc;", "dX[m * K + k] = acc;"),
    ("dx_transposed_B", "acc += dY[m * L + l] * B[j * L + l];", "acc += dY[m * L + l] * B[l * r + j];"),
    ("da_index", "dA[k * r + j] += xk * dyb[m * r + j];", "dA[k * r + j] += xk * dyb[m * r + 0];"),
    ("db_index", "dB[j * L + l] += hj * dY[m * L + l];", "dB[j * L + l] += hj * dY[m * L + 0];"),
    ("shrink_past_rank", "for (int32_t j = 0; j < rank; ++j) {\n                const double *arow",
     "for (int32_t j = 0; j < R; ++j) {\n                const double *arow"),
    ("expand_slice_offset", "bs[(off + c) * R + j]", "bs[(c) * R + j]"),
    ("rank0_active", "return ranks[slot] >= 1 && ranks[slot] <= R;",
     "return ranks[slot] >= 0 && ranks[slot] <= R;"),
    ("gather_wrong_column", "h[t * R + j] = a[((int64_t)slot * R + j) * V + id];",
     "h[t * R + j] = a[((int64_t)slot * R + j) * V + 0];"),
    ("group_counts_unmasked", "if (slot_active(slots[t], S, R, ranks)) counts[slots[t]] += 1;",
     "if (slots[t] >= 0 && slots[t] < S) counts[slots[t]] += 1;"),
]


def _pins():
    yield P.test_golden_single_adapter, ()
    yield P.test_golden_multi_adapter, ()
    for shp in P.SHAPES:
        yield P.test_forward_dense_association, shp
        yield P.test_backward_dense_association, shp
    yield P.test_rank1_closed_form, ()
    yield P.test_finite_differences_exact, ()
    yield P.test_invariants_single, ()
    yield P.test_multi_equals_per_token_single_adapter, ()
    yield P.test_multi_inactive_rows_untouched_and_h_zero, ()
    yield P.test_multi_token_permutation, ()
    yield P.test_multi_slices_equal_separate_calls, ()
    yield P.test_apply_equals_expand_of_shrink, ()
    yield P.test_multi_scale_linearity_and_zero_b, ()
    yield P.test_gather_is_shrink_of_one_hot_bit_exact, ()
    for s in (0, 1, 2):
        yield P.test_group_by_slot_is_stable_sort, (s,)


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name, old, new):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, name
    c = tmp_path / "mutant.c"
    c.write_text(src.replace(old, new))
    so = O.build(force=True, src=str(c), out=str(tmp_path / "libmutant.so"))
    monkeypatch.setattr(O, "_lib", O.load(so))
    failed = []
    for fn, args in _pins():
        try:
            fn(*args)
        except AssertionError:
            failed.append(fn.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
