"""Pins of the fp64 oracle to facts other than itself (no GPU needed).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a missed mask) fails at least one:
  * hand-worked integer fixtures (tests/golden/*.json, each citing its page)
  * brute force through a different association (dense W = s*A*B)
  * the rank-1 closed form, written as explicit Python loops
  * exact central differences of the linear functional sum(dY * y)
  * invariants: B = 0 / s = 0 / rank 0 / inactive slot leave y bit-identical,
    linearity in s, per-token single-adapter equivalence, token permutation,
    slice splitting, apply = expand(shrink), gather = shrink of a one-hot
  * grouping by slot = numpy's stable argsort on the active tokens
"""
import json
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _nan(a):
    return np.array([[np.nan if v is None else v for v in row] for row in a], dtype=np.float64) \
        if np.ndim(a) == 2 else np.array(
            [[[np.nan if v is None else v for v in row] for row in m] for m in a], dtype=np.float64)


def _rel(a, b):
    d = np.max(np.abs(np.asarray(a) - np.asarray(b))) if np.size(a) else 0.0
    m = np.max(np.abs(b)) if np.size(b) else 0.0
    return d / (m if m > 0 else 1.0)


# ----------------------------------------------------------------------------- fixtures
def test_golden_single_adapter():
    g = _load("single_adapter_hand.json")
    X, A, B, Y0, dY = (np.array(g[k], float) for k in ("X", "A", "B", "Y0", "dY"))
    s = g["s"]
    assert np.array_equal(O.forward(X, A, B, Y0, s), np.array(g["Y"], float))
    dX, dA = O.backward_dx_da(X, dY, A, B, s)
    assert np.array_equal(dX, np.array(g["dX"], float))
    assert np.array_equal(dA, np.array(g["dA"], float))
    assert np.array_equal(O.backward_db(X, A, dY, s), np.array(g["dB"], float))


def test_golden_multi_adapter():
    g = _load("multi_adapter_hand.json")
    R = g["R"]
    ranks = np.array(g["ranks"], np.int32)
    slots = np.array(g["slots"], np.int32)
    scal = np.array([np.nan if v is None else v for v in g["scalings"]])
    x = np.array(g["x"], float)
    a = _nan(g["a"])
    b = _nan(g["b"])
    y0 = np.array(g["y0"], float)
    h = O.shrink(x, a, slots, ranks, R, 1)
    assert np.array_equal(h, np.array(g["h"], float))
    y = O.expand(h, b, slots, ranks, scal, y0, g["out_slices"], R)
    assert np.array_equal(y, np.array(g["y"], float))
    y2 = O.apply_linear(x, a, b, slots, ranks, scal, y0, g["out_slices"], R)
    assert np.array_equal(y2, np.array(g["y"], float))
    hg = O.gather_shrink(np.array(g["ids"], np.int64), a, slots, ranks, R)
    assert np.array_equal(hg, np.array(g["h_gather"], float))
    counts, perm = O.group_by_slot(slots, ranks, R)
    assert counts.tolist() == g["counts"] and perm.tolist() == g["perm"]


# ----------------------------------------------------------------------------- single adapter
def _rand_single(rng, M, K, L, r):
    return (rng.standard_normal((M, K)), rng.standard_normal((K, r)), rng.standard_normal((r, L)),
            rng.standard_normal((M, L)), rng.standard_normal((M, L)))


SHAPES = [(1, 1, 1, 1), (2, 3, 5, 1), (3, 7, 4, 2), (9, 8, 9, 3), (5, 9, 2, 3), (4, 6, 7, 2)]


@pytest.mark.parametrize("M,K,L,r", SHAPES)
def test_forward_dense_association(M, K, L, r):
    rng = np.random.default_rng(100 + M * 31 + K * 7 + L * 3 + r)
    X, A, B, Y0, _ = _rand_single(rng, M, K, L, r)
    s = 0.75
    W = s * (A @ B)                      # K x L, formed first: a different association
    ref = Y0 + X @ W
    assert _rel(O.forward(X, A, B, Y0, s), ref) < 1e-12


@pytest.mark.parametrize("M,K,L,r", SHAPES)
def test_backward_dense_association(M, K, L, r):
    rng = np.random.default_rng(200 + M * 31 + K * 7 + L * 3 + r)
    X, A, B, _, dY = _rand_single(rng, M, K, L, r)
    s = -1.25
    dW = X.T @ dY                        # gradient of the dense K x L weight
    W = s * (A @ B)
    dX, dA = O.backward_dx_da(X, dY, A, B, s)
    assert _rel(dX, dY @ W.T) < 1e-12
    assert _rel(dA, s * dW @ B.T) < 1e-12
    assert _rel(O.backward_db(X, A, dY, s), s * A.T @ dW) < 1e-12


@pytest.mark.parametrize("M,K,L,r", SHAPES)
def test_backward_ex_accumulates_dense_gradient(M, K, L, r):
    # the accumulating dX is dX0 plus dY W^T of the dense weight; dA, dB as the backward
    rng = np.random.default_rng(300 + M * 31 + K * 7 + L * 3 + r)
    X, A, B, _, dY = _rand_single(rng, M, K, L, r)
    dX0 = rng.standard_normal((M, K))
    s = 0.5
    W = s * (A @ B)
    dW = X.T @ dY
    dX, dA, dB = O.backward_ex(X, dY, A, B, s, dX0)
    assert _rel(dX, dX0 + dY @ W.T) < 1e-12
    assert _rel(dA, s * dW @ B.T) < 1e-12
    assert _rel(dB, s * A.T @ dW) < 1e-12
    dXo, _, _ = O.backward_ex(X, dY, A, B, s)
    assert _rel(dXo, dY @ W.T) < 1e-12


def test_rank1_closed_form():
    rng = np.random.default_rng(7)
    M, K, L = 4, 5, 6
    X = rng.standard_normal((M, K))
    av = rng.standard_normal(K)
    bv = rng.standard_normal(L)
    Y0 = rng.standard_normal((M, L))
    s = 3.0
    Y = O.forward(X, av[:, None], bv[None, :], Y0, s)
    for m in range(M):
        xa = 0.0
        for k in range(K):
            xa += X[m, k] * av[k]
        for l in range(L):
            assert abs(Y[m, l] - (Y0[m, l] + s * xa * bv[l])) <= 1e-12 * (1 + abs(Y[m, l]))


def test_single_adapter_sums_run_in_ascending_order():
    """Each element of the oracle's single-adapter outputs is one sum over its
    contraction index in ascending order (no reassociation, no fused
    multiply-add): bit-for-bit what plain Python float loops give.  This guards
    the loop nesting of the oracle, which is arranged for cache locality; it is
    a regression check of the summation order, not a pin of the definition."""
    rng = np.random.default_rng(11)
    M, K, L, r, s = 5, 7, 6, 3, 0.75
    X, A, B = rng.standard_normal((M, K)), rng.standard_normal((K, r)), rng.standard_normal((r, L))
    Y0, dY = rng.standard_normal((M, L)), rng.standard_normal((M, L))

    def dot(n, f):
        acc = 0.0
        for i in range(n):
            acc += f(i)
        return acc

    h = [[dot(K, lambda k: X[m, k] * A[k, j]) for j in range(r)] for m in range(M)]
    Y = [[Y0[m, l] + s * dot(r, lambda j: h[m][j] * B[j, l]) for l in range(L)] for m in range(M)]
    dyb = [[dot(L, lambda l: dY[m, l] * B[j, l]) for j in range(r)] for m in range(M)]
    dX = [[s * dot(r, lambda j: dyb[m][j] * A[k, j]) for k in range(K)] for m in range(M)]
    dA = [[s * dot(M, lambda m: X[m, k] * dyb[m][j]) for j in range(r)] for k in range(K)]
    dB = [[s * dot(M, lambda m: h[m][j] * dY[m, l]) for l in range(L)] for j in range(r)]
    gdX, gdA = O.backward_dx_da(X, dY, A, B, s)
    assert np.array_equal(O.forward(X, A, B, Y0, s), np.array(Y))
    assert np.array_equal(gdX, np.array(dX)) and np.array_equal(gdA, np.array(dA))
    assert np.array_equal(O.backward_db(X, A, dY, s), np.array(dB))


def test_finite_differences_exact():
    """L(X, A, B) = sum(dY * forward(X, A, B, 0)) is linear in each of X, A, B,
    so a central difference is exact up to fp64 rounding for any step."""
    rng = np.random.default_rng(11)
    M, K, L, r = 3, 5, 4, 2
    X, A, B, _, dY = _rand_single(rng, M, K, L, r)
    s = 0.6
    Z = np.zeros((M, L))

    def loss(X_, A_, B_):
        return float(np.sum(dY * O.forward(X_, A_, B_, Z, s)))

    dX, dA = O.backward_dx_da(X, dY, A, B, s)
    dB = O.backward_db(X, A, dY, s)
    eps = 0.37
    for (arr, grad, which) in ((X, dX, 0), (A, dA, 1), (B, dB, 2)):
        for idx in np.ndindex(arr.shape):
            p = [X.copy(), A.copy(), B.copy()]
            m = [X.copy(), A.copy(), B.copy()]
            p[which][idx] += eps
            m[which][idx] -= eps
            fd = (loss(*p) - loss(*m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-9 * (1 + abs(grad[idx])), (which, idx)


def test_invariants_single():
    rng = np.random.default_rng(5)
    M, K, L, r = 6, 7, 5, 3
    X, A, B, Y0, dY = _rand_single(rng, M, K, L, r)
    assert np.array_equal(O.forward(X, A, np.zeros_like(B), Y0, 1.5), Y0)
    assert np.array_equal(O.forward(X, A, B, Y0, 0.0), Y0)
    d1 = O.forward(X, A, B, Y0, 1.0) - Y0
    d3 = O.forward(X, A, B, Y0, 3.0) - Y0
    assert _rel(d3, 3.0 * d1) < 1e-12
    # rank 0: nothing added, zero gradients, empty dA/dB
    Y = O.forward(X, np.zeros((K, 0)), np.zeros((0, L)), Y0, 2.0)
    assert np.array_equal(Y, Y0)
    dX, dA = O.backward_dx_da(X, dY, np.zeros((K, 0)), np.zeros((0, L)), 2.0)
    assert np.array_equal(dX, np.zeros((M, K))) and dA.shape == (K, 0)
    # K = 0: h = 0 so dB = 0; L = 0: dyb = 0 so dX = 0 and dA = 0
    assert np.array_equal(O.backward_db(np.zeros((M, 0)), np.zeros((0, r)), dY, 1.0),
                          np.zeros((r, L)))
    dX, dA = O.backward_dx_da(X, np.zeros((M, 0)), A, np.zeros((r, 0)), 1.0)
    assert np.array_equal(dX, np.zeros((M, K))) and np.array_equal(dA, np.zeros((K, r)))


# ----------------------------------------------------------------------------- multi adapter
def _rand_multi(rng, T, IN, S, R, osl, rank_choices=(0, 1, 2, 3, 4)):
    n = len(osl)
    O_ = sum(osl)
    ranks = rng.choice(rank_choices, size=S).astype(np.int32)
    ranks[0] = 0
    slots = rng.integers(-1, S + 1, size=T).astype(np.int32)   # includes out-of-range
    scal = rng.uniform(0.5, 2.0, size=S)
    scal[ranks == 0] = np.nan
    x = rng.standard_normal((T, IN))
    a = rng.standard_normal((S, n * R, IN))
    b = rng.standard_normal((S, O_, R))
    for s in range(S):
        a.reshape(S, n, R, IN)[s, :, ranks[s]:, :] = np.nan
        b[s, :, ranks[s]:] = np.nan
    y0 = rng.standard_normal((T, O_))
    return ranks, slots, scal, x, a, b, y0


def _active(slot, S, R, ranks):
    return 0 <= slot < S and 1 <= ranks[slot] <= R


def test_multi_equals_per_token_single_adapter():
    rng = np.random.default_rng(21)
    T, IN, S, R, osl = 17, 6, 5, 4, [3, 2, 4]
    ranks, slots, scal, x, a, b, y0 = _rand_multi(rng, T, IN, S, R, osl)
    y = O.apply_linear(x, a, b, slots, ranks, scal, y0, osl, R)
    off = np.concatenate([[0], np.cumsum(osl)])
    for t in range(T):
        s = slots[t]
        if not _active(s, S, R, ranks):
            assert np.array_equal(y[t], y0[t])
            continue
        k = ranks[s]
        for i, o in enumerate(osl):
            A = a[s, i * R:i * R + k, :].T                  # IN x k
            B = b[s, off[i]:off[i] + o, :k].T               # k x o
            ref = O.forward(x[t:t + 1], A, B, y0[t:t + 1, off[i]:off[i] + o], scal[s])
            assert _rel(y[t:t + 1, off[i]:off[i] + o], ref) < 1e-12


def test_multi_inactive_rows_untouched_and_h_zero():
    rng = np.random.default_rng(22)
    T, IN, S, R, osl = 23, 5, 6, 3, [4]
    ranks, slots, scal, x, a, b, y0 = _rand_multi(rng, T, IN, S, R, osl, (0, 1, 3, 4))
    ranks[2] = R + 1                                          # rank past R: inactive too
    h = O.shrink(x, a, slots, ranks, R, 1)
    y = O.expand(h, b, slots, ranks, scal, y0, osl, R)
    for t in range(T):
        if not _active(slots[t], S, R, ranks):
            assert np.array_equal(y[t], y0[t]) and not np.any(h[t])
        else:
            assert np.all(h[t, ranks[slots[t]]:] == 0)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(h))


def test_multi_token_permutation():
    rng = np.random.default_rng(23)
    T, IN, S, R, osl = 19, 7, 5, 4, [2, 3]
    ranks, slots, scal, x, a, b, y0 = _rand_multi(rng, T, IN, S, R, osl)
    p = rng.permutation(T)
    y = O.apply_linear(x, a, b, slots, ranks, scal, y0, osl, R)
    yp = O.apply_linear(x[p], a, b, slots[p], ranks, scal, y0[p], osl, R)
    assert np.array_equal(yp, y[p])
    h = O.shrink(x, a, slots, ranks, R, 2)
    hp = O.shrink(x[p], a, slots[p], ranks, R, 2)
    assert np.array_equal(hp, h[p])


def test_multi_slices_equal_separate_calls():
    rng = np.random.default_rng(24)
    T, IN, S, R, osl = 11, 5, 4, 3, [2, 4, 3]
    ranks, slots, scal, x, a, b, y0 = _rand_multi(rng, T, IN, S, R, osl, (0, 1, 2, 3))
    y = O.apply_linear(x, a, b, slots, ranks, scal, y0, osl, R)
    off = np.concatenate([[0], np.cumsum(osl)])
    for i, o in enumerate(osl):
        ai = a[:, i * R:(i + 1) * R, :]
        bi = b[:, off[i]:off[i] + o, :]
        yi = O.apply_linear(x, ai, bi, slots, ranks, scal, y0[:, off[i]:off[i] + o], [o], R)
        assert np.array_equal(yi, y[:, off[i]:off[i] + o])


def test_apply_equals_expand_of_shrink():
    rng = np.random.default_rng(25)
    T, IN, S, R, osl = 13, 6, 4, 4, [5, 2]
    ranks, slots, scal, x, a, b, y0 = _rand_multi(rng, T, IN, S, R, osl)
    h = O.shrink(x, a, slots, ranks, R, 2)
    assert np.array_equal(O.expand(h, b, slots, ranks, scal, y0, osl, R),
                          O.apply_linear(x, a, b, slots, ranks, scal, y0, osl, R))


def test_multi_scale_linearity_and_zero_b():
    rng = np.random.default_rng(26)
    T, IN, S, R, osl = 9, 4, 3, 2, [3]
    ranks, slots, scal, x, a, b, y0 = _rand_multi(rng, T, IN, S, R, osl, (1, 2))
    y1 = O.apply_linear(x, a, b, slots, ranks, scal, y0, osl, R)
    y2 = O.apply_linear(x, a, b, slots, ranks, 2 * scal, y0, osl, R)
    assert _rel(y2 - y0, 2 * (y1 - y0)) < 1e-12
    bz = np.where(np.isnan(b), np.nan, 0.0)
    assert np.array_equal(O.apply_linear(x, a, bz, slots, ranks, scal, y0, osl, R), y0)


def test_gather_is_shrink_of_one_hot_bit_exact():
    rng = np.random.default_rng(27)
    T, V, S, R = 15, 9, 4, 3
    ranks, slots, scal, _, a, _, _ = _rand_multi(rng, T, V, S, R, [1], (0, 1, 2, 3))
    ids = rng.integers(-2, V + 2, size=T)
    hg = O.gather_shrink(ids, a, slots, ranks, R)
    onehot = np.zeros((T, V))
    for t in range(T):
        if 0 <= ids[t] < V:
            onehot[t, ids[t]] = 1.0
    hs = O.shrink(onehot, a, slots, ranks, R, 1)
    assert np.array_equal(hg, hs)
    for t in range(T):
        if not (0 <= ids[t] < V) or not _active(slots[t], S, R, ranks):
            assert not np.any(hg[t])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_group_by_slot_is_stable_sort(seed):
    rng = np.random.default_rng(300 + seed)
    T, S, R = 200, 9, 4
    ranks = rng.integers(0, R + 2, size=S).astype(np.int32)
    slots = rng.integers(-2, S + 2, size=T).astype(np.int32)
    counts, perm = O.group_by_slot(slots, ranks, R)
    act = np.array([_active(s, S, R, ranks) for s in slots])
    idx = np.nonzero(act)[0]
    ref = idx[np.argsort(slots[idx], kind="stable")]
    assert perm.tolist() == ref.tolist()
    assert counts.tolist() == [int(np.sum(slots[idx] == s)) for s in range(S)]
