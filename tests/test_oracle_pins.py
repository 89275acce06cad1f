"""Pins of the CPU oracle against things other than itself.

Each pin is a function ``pin_*(O)`` taking an oracle module and returning
(ok, message).  The real oracle must pass all of them; every planted mistake in
``test_planted_mistakes_are_caught`` (a textual edit of the oracle's own source,
run on the CPU) must fail at least one.
"""
import importlib.util
import json
import os
import types

import numpy as np
import pytest

import oracle.lora_oracle as ORACLE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------------------
# independent helpers (pure Python / numpy library calls, no oracle code)
# ------------------------------------------------------------------------------------------

def brute_force(x, W, adapters, idx, r_max):
    """Pure-Python loops straight from the formula, true-rank adapters, no padding."""
    n, h_in = len(x), len(x[0])
    h_out = len(W)
    y = [[0.0] * h_out for _ in range(n)]
    for t in range(n):
        s = idx[t]
        for o in range(h_out):
            acc = 0.0
            for k in range(h_in):
                acc += x[t][k] * W[o][k]
            if s >= 0:
                A, B, r, alpha = adapters[s]
                lora = 0.0
                for j in range(r):
                    u = 0.0
                    for k in range(h_in):
                        u += A[j][k] * x[t][k]
                    lora += B[o][j] * u
                acc += (alpha / r) * lora
            y[t][o] = acc
    return y


def tiny_problem(seed, n=7, h_in=5, h_out=6, ranks=(1, 3, 2), r_max=4, p_base=0.3):
    rng = np.random.default_rng(seed)
    S = len(ranks)
    idx = np.where(rng.random(n) < p_base, -1, rng.integers(0, S, n)).astype(np.int32)
    x = rng.standard_normal((n, h_in))
    W = rng.standard_normal((h_out, h_in))
    adapters = []
    for r in ranks:
        A = rng.standard_normal((r, h_in))
        B = rng.standard_normal((h_out, r))
        alpha = float(rng.integers(1, 33))
        adapters.append((A, B, r, alpha))
    return x, W, adapters, idx, r_max


def make_pool(O, adapters, r_max, h_in, h_out, n_slots=None):
    return O.pad_pool([a[0] for a in adapters], [a[1] for a in adapters], [a[2] for a in adapters],
                      [a[3] for a in adapters], r_max, h_in, h_out, n_slots=n_slots)


# ------------------------------------------------------------------------------------------
# pins
# ------------------------------------------------------------------------------------------

def pin_golden(O):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_small.json")))
    ads = sorted(g["adapters"], key=lambda a: a["slot"])
    pool = O.pad_pool([np.array(a["A"], float) for a in ads], [np.array(a["B"], float) for a in ads],
                      [a["rank"] for a in ads], [a["alpha"] for a in ads], g["r_max"], g["h_in"],
                      g["h_out"], n_slots=g["n_slots"], slots=[a["slot"] for a in ads])
    x = np.array(g["x"], float)
    idx = np.array(g["idx"], np.int32)
    y = O.lora_linear(x, np.array(g["W"], float), pool, idx)
    if not np.array_equal(y, np.array(g["y"], float)):
        return False, f"golden y mismatch {y.tolist()}"
    perm, ss, sl, nseg = O.segments(idx, pool)
    if perm.tolist() != g["perm"] or ss.tolist() != g["seg_start"] or sl.tolist() != g["seg_slot"] \
            or nseg != g["nseg"]:
        return False, "golden segments mismatch"
    return True, ""


def pin_brute_force(O):
    for seed in range(6):
        x, W, adapters, idx, r_max = tiny_problem(seed)
        pool = make_pool(O, adapters, r_max, x.shape[1], W.shape[0])
        y = O.lora_linear(x, W, pool, idx)
        yb = np.array(brute_force(x.tolist(), W.tolist(), adapters, idx.tolist(), r_max))
        if not np.allclose(y, yb, rtol=1e-12, atol=1e-12):
            return False, f"seed {seed}: max err {np.abs(y - yb).max()}"
    return True, ""


def pin_segments_argsort(O):
    rng = np.random.default_rng(123)
    cases = [np.full(9, -1), np.zeros(9), np.array([3]), np.arange(5)[::-1], np.array([], np.int32)]
    for _ in range(40):
        S = int(rng.integers(1, 12))
        n = int(rng.integers(1, 200))
        cases.append(rng.integers(-1, S, n))
    for idx in cases:
        idx = np.asarray(idx, np.int32)
        S = int(idx.max()) + 1 if idx.size and idx.max() >= 0 else 1
        perm, ss, sl, nseg = O.segments(idx, S)
        if perm.tolist() != np.argsort(idx, kind="stable").tolist():
            return False, f"perm differs from stable argsort for {idx.tolist()}"
        # runs by brute force over the sorted keys
        keys = idx[np.argsort(idx, kind="stable")].tolist()
        runs_start, runs_key = [], []
        for j, k in enumerate(keys):
            if j == 0 or keys[j - 1] != k:
                runs_start.append(j)
                runs_key.append(k)
        if ss.tolist() != runs_start + [len(keys)] or sl.tolist() != runs_key or nseg != len(runs_key):
            return False, f"runs differ for {idx.tolist()}"
    return True, ""


def pin_base_only(O):
    x, W, adapters, idx, r_max = tiny_problem(7, n=9)
    pool = make_pool(O, adapters, r_max, x.shape[1], W.shape[0])
    y = O.lora_linear(x, W, pool, np.full(9, -1, np.int32))
    if not np.allclose(y, np.matmul(x, W.T), rtol=1e-13, atol=1e-13):
        return False, "idx=-1 differs from x W^T"
    return True, ""


def pin_merged_weight(O):
    x, W, adapters, idx, r_max = tiny_problem(8, n=6)
    pool = make_pool(O, adapters, r_max, x.shape[1], W.shape[0])
    for s, (A, B, r, alpha) in enumerate(adapters):
        y = O.lora_linear(x, W, pool, np.full(6, s, np.int32))
        merged = W + (alpha / r) * (B @ A)
        if not np.allclose(y, x @ merged.T, rtol=1e-12, atol=1e-12):
            return False, f"slot {s}: merged-weight identity fails"
    return True, ""


def pin_zero_pad(O):
    x, W, adapters, idx, r_max = tiny_problem(9, n=8)
    y_tight = O.lora_linear(x, W, make_pool(O, adapters, max(a[2] for a in adapters), x.shape[1], W.shape[0]),
                            idx)
    y_pad = O.lora_linear(x, W, make_pool(O, adapters, 16, x.shape[1], W.shape[0]), idx)
    # padded terms are exact zeros; only the summation order of the dot products may move
    if not np.allclose(y_tight, y_pad, rtol=1e-13, atol=1e-13):
        return False, "padding to r_max changed the result"
    return True, ""


def pin_permutation(O):
    x, W, adapters, idx, r_max = tiny_problem(10, n=11)
    pool = make_pool(O, adapters, r_max, x.shape[1], W.shape[0])
    y = O.lora_linear(x, W, pool, idx)
    p = np.random.default_rng(3).permutation(11)
    yp = O.lora_linear(x[p], W, pool, idx[p])
    if not np.allclose(yp, y[p], rtol=1e-13, atol=1e-13):
        return False, "permuting tokens does not permute outputs"
    return True, ""


def pin_selector(O):
    # W = 0, A = e_j (one row), B = e_i (one column): y[t, i] = scale * x[t, j], else 0
    h_in, h_out, r_max = 5, 4, 3
    x = np.arange(1.0, 1.0 + 3 * h_in).reshape(3, h_in)
    A0 = np.zeros((1, h_in)); A0[0, 3] = 1.0
    B0 = np.zeros((h_out, 1)); B0[1, 0] = 1.0
    A1 = np.zeros((2, h_in)); A1[1, 0] = 1.0
    B1 = np.zeros((h_out, 2)); B1[2, 1] = 1.0
    pool = O.pad_pool([A0, A1], [B0, B1], [1, 2], [3.0, 8.0], r_max, h_in, h_out)
    y = O.lora_linear(x, np.zeros((h_out, h_in)), pool, np.array([0, 1, -1], np.int32))
    want = np.zeros((3, h_out))
    want[0, 1] = 3.0 * x[0, 3]
    want[1, 2] = 4.0 * x[1, 0]
    if not np.array_equal(y, want):
        return False, f"selector closed form fails {y.tolist()}"
    return True, ""


def pin_rank1(O):
    rng = np.random.default_rng(11)
    h_in, h_out = 6, 5
    a, b = rng.standard_normal(h_in), rng.standard_normal(h_out)
    x = rng.standard_normal((4, h_in))
    pool = O.pad_pool([a[None, :]], [b[:, None]], [1], [2.5], 4, h_in, h_out)
    y = O.lora_linear(x, np.zeros((h_out, h_in)), pool, np.zeros(4, np.int32))
    want = 2.5 * np.outer(x @ a, b)
    if not np.allclose(y, want, rtol=1e-13, atol=1e-13):
        return False, "rank-1 outer product fails"
    return True, ""


def pin_errors(O):
    x, W, adapters, idx, r_max = tiny_problem(12, n=4)
    pool = make_pool(O, adapters, r_max, x.shape[1], W.shape[0], n_slots=5)  # slots 3,4 empty
    for bad in ([0, 1, 3, -1], [0, 5, 1, 1], [-2, 0, 0, 0]):
        try:
            O.lora_linear(x, W, pool, np.array(bad, np.int32))
        except O.OracleError as e:
            if e.code != O.EIDX:
                return False, "wrong error code"
            continue
        return False, f"idx {bad} accepted"
    return True, ""


def tiny_group(seed, n=6, h_in=5, h_outs=(3, 4, 2), ranks=((1, 2), (2, 2), (3, 1)), r_max=3):
    """Slices sharing x and idx; ranks[q][s] is slice q's rank for slot s."""
    rng = np.random.default_rng(seed)
    S = len(ranks[0])
    idx = np.where(rng.random(n) < 0.25, -1, rng.integers(0, S, n)).astype(np.int32)
    x = rng.standard_normal((n, h_in))
    Ws, slices = [], []
    for h_out, rq in zip(h_outs, ranks):
        Ws.append(rng.standard_normal((h_out, h_in)))
        slices.append([(rng.standard_normal((r, h_in)), rng.standard_normal((h_out, r)), r,
                        float(rng.integers(1, 33))) for r in rq])
    return x, Ws, slices, idx, r_max


def pin_group_block_diagonal(O):
    """The group equals one linear over the stacked weight whose LoRA term, per token, is a
    block-diagonal B (every slice's B_s on the diagonal) applied to the stacked, scaled A_s x."""
    from scipy.linalg import block_diag

    for seed in range(4):
        x, Ws, slices, idx, r_max = tiny_group(20 + seed)
        pools = [make_pool(O, ads, r_max, x.shape[1], W.shape[0]) for W, ads in zip(Ws, slices)]
        y = O.lora_linear_group(x, Ws, pools, idx)
        want = x @ np.vstack(Ws).T
        for t, s in enumerate(idx.tolist()):
            if s < 0:
                continue
            A_stack = np.vstack([(ads[s][3] / ads[s][2]) * ads[s][0] for ads in slices])
            B_blk = block_diag(*[ads[s][1] for ads in slices])
            want[t] += B_blk @ (A_stack @ x[t])
        if y.shape != want.shape or not np.allclose(y, want, rtol=1e-12, atol=1e-12):
            return False, f"seed {seed}: block-diagonal form differs"
    return True, ""


def pin_group_brute_force(O):
    x, Ws, slices, idx, r_max = tiny_group(30, n=5)
    pools = [make_pool(O, ads, r_max, x.shape[1], W.shape[0]) for W, ads in zip(Ws, slices)]
    y = O.lora_linear_group(x, Ws, pools, idx)
    cols = [brute_force(x.tolist(), W.tolist(), ads, idx.tolist(), r_max) for W, ads in zip(Ws, slices)]
    want = np.array([sum((c[t] for c in cols), []) for t in range(len(idx))])
    if y.shape != want.shape or not np.allclose(y, want, rtol=1e-12, atol=1e-12):
        return False, "group differs from per-slice brute force side by side"
    return True, ""


def pin_group_errors(O):
    x, Ws, slices, idx, r_max = tiny_group(31)
    pools = [make_pool(O, ads, r_max, x.shape[1], W.shape[0]) for W, ads in zip(Ws, slices)]
    # slice 1 holds slot 0 only (slot 1 of the same identity is missing there)
    pools[1] = make_pool(O, slices[1][:1], r_max, x.shape[1], Ws[1].shape[0], n_slots=2)
    try:
        O.lora_linear_group(x, Ws, pools, np.array([0, 1, -1, 0, 0, 1], np.int32))
    except O.OracleError as e:
        return (e.code == O.EIDX), "wrong error code"
    return False, "slot missing from one slice accepted"


def pin_rows_subset(O):
    """lora_linear(..., rows=r) against brute force on the requested rows, in the order given:
    permuted, repeated and unsorted subsets, with x as a numpy array and as a torch tensor."""
    import torch

    for seed in range(3):
        x, W, adapters, idx, r_max = tiny_problem(40 + seed, n=9, p_base=0.2)
        pool = make_pool(O, adapters, r_max, x.shape[1], W.shape[0])
        full = np.array(brute_force(x.tolist(), W.tolist(), adapters, idx.tolist(), r_max))
        subsets = [[8, 0, 3], [2, 2, 7, 2], list(np.random.default_rng(seed).permutation(9)), [5]]
        for rows in subsets:
            for xin in (x, torch.from_numpy(x)):
                y = O.lora_linear(xin, W, pool, idx, rows=rows)
                if y.shape != (len(rows), W.shape[0]) or not np.allclose(y, full[rows], rtol=1e-12, atol=1e-12):
                    return False, f"seed {seed}: rows={rows} ({type(xin).__name__} x) differ from brute force"
    return True, ""


def pin_tolerance(O):
    """within_tolerance is the stated bar |y - y_ref| <= 1e-2 + 1e-2 |y_ref|, elementwise.
    Hand-computed pairs just inside and just outside the bound (positive, negative and zero
    references) and 16-bit outputs whose exact values are known."""
    import torch

    # (y, y_ref, expected): bound = 0.01 + 0.01 |y_ref|
    pairs = [
        (2.0299, 2.0, True), (2.0301, 2.0, False), (1.9701, 2.0, True), (1.9699, 2.0, False),  # bound 0.03
        (-3.0399, -3.0, True), (-3.0401, -3.0, False), (-2.9601, -3.0, True), (-2.9599, -3.0, False),  # 0.04
        (0.0099, 0.0, True), (-0.0101, 0.0, False),  # bound 0.01 at a zero reference
        (100.0, 101.0, True), (98.97, 101.0, False),  # bound 1.02
    ]
    y = np.array([p[0] for p in pairs])
    ref = np.array([p[1] for p in pairs])
    got = O.within_tolerance(y, ref)
    want = np.array([p[2] for p in pairs])
    if got.shape != want.shape or not np.array_equal(got, want):
        return False, f"float64 pairs: got {got.tolist()}"
    # 16-bit inputs are upcast exactly: fp16 1 + 2^-7 vs 1.0 (diff 0.0078125 <= 0.02: inside);
    # bf16 1 + 2^-6 vs 0.99 (diff 0.025625 > 0.0199: outside); bf16 -2^-7 vs 0 (0.0078125: inside)
    y16 = torch.tensor([[1.0078125, 0.0]], dtype=torch.float16)
    yb = torch.tensor([[1.015625, -0.0078125]], dtype=torch.bfloat16)
    g16 = O.within_tolerance(y16, np.array([[1.0, 0.0]]))
    gb = O.within_tolerance(yb, np.array([[0.99, 0.0]]))
    if g16.tolist() != [[True, True]] or gb.tolist() != [[False, True]]:
        return False, f"16-bit inputs: {g16.tolist()} {gb.tolist()}"
    return True, ""


PINS = [pin_golden, pin_brute_force, pin_segments_argsort, pin_base_only, pin_merged_weight,
        pin_zero_pad, pin_permutation, pin_selector, pin_rank1, pin_errors, pin_group_block_diagonal,
        pin_group_brute_force, pin_group_errors, pin_rows_subset, pin_tolerance]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    ok, msg = pin(ORACLE)
    assert ok, msg


def test_empty_batch_segments():
    perm, ss, sl, nseg = ORACLE.segments(np.zeros(0, np.int32), 4)
    assert perm.size == 0 and ss.tolist() == [0] and sl.size == 0 and nseg == 0


# ------------------------------------------------------------------------------------------
# planted mistakes: each is a textual edit of the oracle's source, run on the CPU
# ------------------------------------------------------------------------------------------

MUTANTS = {
    "scale_by_r_max": ("scale[s] = float(alpha) / float(r)", "scale[s] = float(alpha) / float(r_max)"),
    "minus_one_wraps_to_last_slot": ("if s < 0:\n            continue", "if s < -1:\n            continue"),
    "wrong_slot_for_B": ("(pool.B[s] @ u)", "(pool.B[(s + 1) % pool.n_slots] @ u)"),
    "dropped_base_term": ("y = xs @ W64.T", "y = 0.0 * (xs @ W64.T)"),
    "W_not_transposed": ("y = xs @ W64.T", "y = xs @ W64.T.T.T.T"),
    "A_transposed_pad": ("A[s, :r, :] = a", "A[s, :r, :] = a[::-1]"),
    "unstable_placement": ("for t, k in enumerate(idx.tolist()):\n        perm[nxt[k + 1]] = t",
                           "for t, k in reversed(list(enumerate(idx.tolist()))):\n        perm[nxt[k + 1]] = t"),
    "base_only_sorted_last": ("count[k + 1] += 1", "count[(k + 1) if k >= 0 else S] += 1"),
    "scale_missing": ("y[i] += pool.scale[s] * (pool.B[s] @ u)", "y[i] += (pool.B[s] @ u)"),
    "no_validation": ("if k < -1 or k >= S:", "if False:"),
    "group_slices_in_reverse": ("[lora_linear(x, W, p, idx, rows=rows) for W, p in zip(Ws, pools)]",
                                "[lora_linear(x, W, p, idx, rows=rows) for W, p in zip(Ws, pools)][::-1]"),
    "group_one_pool_for_all": ("[lora_linear(x, W, p, idx, rows=rows) for W, p in zip(Ws, pools)]",
                               "[lora_linear(x, W, pools[0], idx, rows=rows) for W, p in zip(Ws, pools)]"),
    "rows_slot_of_output_position": ("s = int(idx[t])", "s = int(idx[i])"),
    "rows_ignored_for_x": ("xs = _f64(x)[rows]", "xs = _f64(x)[np.sort(rows)]"),
    "tolerance_atol_times_10": ("<= atol + rtol * np.abs(y_ref)", "<= 10 * atol + rtol * np.abs(y_ref)"),
    "tolerance_signed_reference": ("<= atol + rtol * np.abs(y_ref)", "<= atol + rtol * y_ref"),
    "tolerance_one_sided": ("return np.abs(y - y_ref) <=", "return (y - y_ref) <="),
}


def _load_mutant(old, new):
    src = open(ORACLE.__file__).read()
    assert old in src, f"mutation anchor vanished from the oracle: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = ORACLE.__file__
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    mod = _load_mutant(*MUTANTS[name])
    caught = []
    for pin in PINS:
        try:
            ok, _ = pin(mod)
        except Exception:
            ok = False
        if not ok:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passes every pin"
