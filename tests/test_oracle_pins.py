"""Pins of the FP64 oracle against facts fixed outside the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a missing max shift, a double rounding, a miscounted
comparison) fails at least one of them:

* closed forms from tests/golden/closed_forms.txt (uniform rows, V = 1, V = 2,
  masked tails, inactive rows, closed-form gradients);
* brute-force nearest-BF16 search for the rounding routine;
* Richardson-extrapolated central differences of the oracle's own forward
  (gradient sign, the one-hot term, the g scaling);
* central differences of a library routine (torch float64 log_softmax);
* a library cross-check of the forward (torch float64 log_softmax + gather);
* 50-digit decimal brute force for a few tiny rows;
* invariants: shift and permutation invariance, rows summing to zero, the
  sharded merge equalling the unsharded log-sum-exp;
* for the fused LM head: numpy float64 matmul + torch float64 log_softmax,
  one-hot weight rows reducing to the logits oracle, equal rows giving
  -log V, a hand-worked two-column example; its backward against torch
  float64 autograd, Richardson central differences of the forward, and the
  BF16-rounded dZ times the operands by numpy matmul.
"""

import math
import struct
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
import workloads
from golden import closed_forms, to_bf16_bits_exact

IGN = -100


def _bits(vals):
    return to_bf16_bits_exact(vals)


def _rand_bf16(rng, n, v, sigma=2.0):
    f = (rng.standard_normal((n, v)) * sigma).astype(np.float32)
    return workloads.bf16_bits(torch.from_numpy(f).to(torch.bfloat16))


# ---------------------------------------------------------------- rounding


def _bf16_value(b):
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


def _brute_nearest_bf16(d):
    """Nearest BF16 by search over all patterns near d's binary32 truncation;
    ties go to the even pattern."""
    if math.isnan(d):
        return None
    f32 = struct.unpack("<I", struct.pack("<f", np.float32(d)))[0] if abs(d) < 3.4e38 else None
    if f32 is None:
        return 0x7F80 | (0x8000 if d < 0 else 0)
    top = f32 >> 16
    cands = []
    for k in range(-3, 4):
        b = (top + k) & 0xFFFF
        if (b & 0x7F80) == 0x7F80 and (b & 0x7F):
            continue  # NaN patterns
        val = _bf16_value(b)
        if math.isinf(val) and not math.isinf(d):
            # inf is the result only when |d| reaches max + half ulp
            if abs(d) < (2 - 2 ** -8) * 2.0 ** 127:
                continue
        cands.append((abs(val - d) if not math.isinf(val) else 0.0, b))
    best = min(c[0] for c in cands)
    ties = [b for dist, b in cands if dist == best]
    # ties: prefer even significand, and among equal values prefer the
    # pattern whose sign matches d (so -0 rounds to -0)
    ties.sort(key=lambda b: (b & 1, (b >> 15) != (1 if math.copysign(1, d) < 0 else 0)))
    return ties[0]


def test_round_bf16_known_values():
    cases = {
        1.0: 0x3F80,
        -1.0: 0xBF80,
        1.0 + 2 ** -8: 0x3F80,          # tie, even stays
        1.0 + 3 * 2 ** -8: 0x3F82,      # tie, rounds up to even
        1.0 + 2 ** -8 + 2 ** -30: 0x3F81,  # just above the tie
        2.0 ** -133: 0x0001,            # smallest subnormal
        2.0 ** -134: 0x0000,            # tie with zero, even
        3 * 2.0 ** -134: 0x0002,        # tie, even
        255 * 2.0 ** 120: 0x7F7F,       # largest finite
        255.5 * 2.0 ** 120: 0x7F80,     # overflow at max + half ulp
        -0.0: 0x8000,
        float("inf"): 0x7F80,
        float("-inf"): 0xFF80,
    }
    for d, want in cases.items():
        assert int(oracle.round_bf16(d)) == want, (d, hex(int(oracle.round_bf16(d))))
    assert int(oracle.round_bf16(float("nan"))) & 0x7FFF > 0x7F80


def test_round_bf16_matches_brute_force():
    rng = np.random.default_rng(1)
    d = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000),
        rng.standard_normal(500) * 2.0 ** -128,     # subnormal range
        (1 + (2 * rng.integers(0, 128, 200) + 1) * 2.0 ** -8) * 2.0 ** rng.integers(-20, 20, 200),  # ties
    ])
    got = oracle.round_bf16(d)
    for di, gi in zip(d, got):
        assert int(gi) == _brute_nearest_bf16(float(di)), (di, hex(int(gi)))


def test_round_bf16_is_not_double_rounding():
    # d sits just above a BF16 tie, but its binary32 rounding lands exactly on
    # the tie; rounding via binary32 would then go to even (down).
    d = 1.0 + 2 ** -8 + 2 ** -40
    assert int(oracle.round_bf16(d)) == 0x3F81


def test_bf16_widening_exact():
    b = np.arange(0, 65536, dtype=np.uint16)
    got = oracle.bf16_to_f64(b)
    want = np.array([_bf16_value(i) for i in range(65536)], dtype=np.float64)
    finite = ~np.isnan(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.all(np.isnan(got[~finite]))


# ---------------------------------------------------------------- closed forms


@pytest.mark.parametrize("case", closed_forms(), ids=lambda c: c["name"])
def test_closed_forms(case):
    x = _bits(case["logits"])[None, :]
    y = np.array([case["target"]], dtype=np.int64)
    logp, lse = oracle.forward(x, y, IGN)
    assert abs(logp[0] - case["logp"]) <= 1e-13 * max(1.0, abs(case["logp"]))
    assert abs(lse[0] - case["lse"]) <= 1e-13 * max(1.0, abs(case["lse"]))
    if case["dlogits"] is not None:
        g = np.array([case["grad"]], dtype=np.float32)
        d = oracle.backward(x, y, g, IGN)
        np.testing.assert_allclose(d[0], case["dlogits"], rtol=0, atol=1e-14)


def test_inactive_rows_are_exact_zero():
    rng = np.random.default_rng(2)
    x = _rand_bf16(rng, 6, 37)
    y = np.array([-100, 37, 40, -1, 5, 36], dtype=np.int64)
    g = np.ones(6, dtype=np.float32)
    logp, _ = oracle.forward(x, y, IGN)
    d = oracle.backward(x, y, g, IGN)
    for t in range(4):
        assert logp[t] == 0.0 and np.all(d[t] == 0.0)
    assert logp[4] < 0 and np.any(d[4] != 0)
    # an ignore index inside [0, V) also deactivates its rows
    logp2, _ = oracle.forward(x, y, 5)
    assert logp2[4] == 0.0


# ---------------------------------------------------------------- library and brute force


def test_forward_matches_torch_float64_log_softmax():
    rng = np.random.default_rng(3)
    for n, v in [(16, 1), (16, 7), (32, 1031), (4, workloads.QWEN3_VOCAB)]:
        x = _rand_bf16(rng, n, v, sigma=3.0)
        y = rng.integers(0, v, n).astype(np.int64)
        logp, lse = oracle.forward(x, y, IGN)
        xt = torch.from_numpy(oracle.bf16_to_f64(x))
        ref_lsm = torch.log_softmax(xt, dim=1)
        ref_logp = ref_lsm.gather(1, torch.from_numpy(y)[:, None])[:, 0].numpy()
        ref_lse = torch.logsumexp(xt, dim=1).numpy()
        np.testing.assert_allclose(logp, ref_logp, rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-12)


def test_forward_decimal_brute_force():
    getcontext().prec = 50
    rng = np.random.default_rng(4)
    x = _rand_bf16(rng, 5, 9, sigma=4.0)
    y = np.array([0, 3, 8, 4, 1], dtype=np.int64)
    logp, lse = oracle.forward(x, y, IGN)
    xv = oracle.bf16_to_f64(x)
    for t in range(5):
        s = sum(Decimal(float(v)).exp() for v in xv[t])
        want_lse = s.ln()
        want_logp = Decimal(float(xv[t, y[t]])) - want_lse
        assert abs(Decimal(lse[t]) - want_lse) < Decimal("1e-14")
        assert abs(Decimal(logp[t]) - want_logp) < Decimal("1e-14")


def test_gradient_against_decimal_softmax():
    getcontext().prec = 50
    rng = np.random.default_rng(5)
    x = _rand_bf16(rng, 3, 6, sigma=2.0)
    y = np.array([0, 5, 2], dtype=np.int64)
    g = np.array([1.5, -0.25, 3.0], dtype=np.float32)
    d = oracle.backward(x, y, g, IGN)
    xv = oracle.bf16_to_f64(x)
    for t in range(3):
        e = [Decimal(float(v)).exp() for v in xv[t]]
        s = sum(e)
        for c in range(6):
            want = Decimal(float(g[t])) * ((1 if c == y[t] else 0) - e[c] / s)
            assert abs(Decimal(d[t, c]) - want) < Decimal("1e-15")


# ---------------------------------------------------------------- finite differences


def test_gradient_by_richardson_central_differences_of_oracle_forward():
    """d logp / d x_v of the oracle's own forward, with perturbations that keep
    every logit an exact BF16 value: logits are small integers in [2, 4), where
    x +- 2^-5 and x +- 2^-6 are BF16 numbers."""
    rng = np.random.default_rng(6)
    v = 12
    base = rng.integers(2, 4, v).astype(np.float64) + rng.integers(0, 8, v) * 2.0 ** -3
    y = np.array([4], dtype=np.int64)
    g = np.array([1.0], dtype=np.float32)
    d = oracle.backward(_bits(base)[None, :], y, g, IGN)[0]

    def logp_at(xs):
        return oracle.forward(_bits(xs)[None, :], y, IGN)[0][0]

    for c in range(v):
        est = []
        for h in (2.0 ** -5, 2.0 ** -6):
            xp, xm = base.copy(), base.copy()
            xp[c] += h
            xm[c] -= h
            est.append((logp_at(xp) - logp_at(xm)) / (2 * h))
        rich = (4 * est[1] - est[0]) / 3
        assert abs(rich - d[c]) < 2e-7, (c, rich, d[c])


def test_gradient_by_central_differences_of_torch_log_softmax():
    rng = np.random.default_rng(7)
    v = 20
    x = _rand_bf16(rng, 1, v, sigma=1.5)
    y = np.array([13], dtype=np.int64)
    g = np.array([-2.5], dtype=np.float32)
    d = oracle.backward(x, y, g, IGN)[0]
    xv = torch.from_numpy(oracle.bf16_to_f64(x)[0])
    h = 1e-6
    for c in range(v):
        xp, xm = xv.clone(), xv.clone()
        xp[c] += h
        xm[c] -= h
        fd = (torch.log_softmax(xp, 0)[13] - torch.log_softmax(xm, 0)[13]).item() / (2 * h)
        assert abs(float(g[0]) * fd - d[c]) < 1e-8


# ---------------------------------------------------------------- invariants


def test_rows_sum_to_zero_and_uniform_gradient():
    rng = np.random.default_rng(8)
    x = _rand_bf16(rng, 8, 1031, sigma=3.0)
    y = rng.integers(0, 1031, 8).astype(np.int64)
    g = rng.standard_normal(8).astype(np.float32)
    d = oracle.backward(x, y, g, IGN)
    for t in range(8):
        assert abs(d[t].sum()) <= 1e-12 * max(1.0, abs(float(g[t])))
        assert np.sign(d[t, y[t]]) == np.sign(g[t]) or g[t] == 0
        off = np.delete(d[t], y[t])
        assert np.all(np.sign(off) * np.sign(g[t]) <= 0)


def test_shift_invariance():
    rng = np.random.default_rng(9)
    # integer-valued logits stay exact BF16 numbers after adding an integer
    xi = rng.integers(-40, 40, (4, 200)).astype(np.float64)
    y = rng.integers(0, 200, 4).astype(np.int64)
    a_logp, a_lse = oracle.forward(_bits(xi), y, IGN)
    b_logp, b_lse = oracle.forward(_bits(xi + 64.0), y, IGN)
    np.testing.assert_allclose(a_logp, b_logp, rtol=0, atol=1e-12)
    np.testing.assert_allclose(b_lse - a_lse, 64.0, rtol=0, atol=1e-12)


def test_large_logits_do_not_overflow():
    # exp(1024) overflows a double: a missing max shift would give inf/nan
    xi = np.array([[1024.0, 1016.0, 1008.0, 1024.0]])
    logp, lse = oracle.forward(_bits(xi), np.array([1], dtype=np.int64), IGN)
    want = -8.0 - math.log(2 + math.exp(-8) + math.exp(-16))
    assert abs(logp[0] - want) < 1e-13 and math.isfinite(lse[0])


def test_permutation_invariance():
    rng = np.random.default_rng(10)
    x = _rand_bf16(rng, 3, 300)
    y = np.array([7, 150, 299], dtype=np.int64)
    logp, lse = oracle.forward(x, y, IGN)
    perm = rng.permutation(300)
    inv = np.argsort(perm)
    logp2, lse2 = oracle.forward(np.ascontiguousarray(x[:, perm]), inv[y], IGN)
    np.testing.assert_allclose(logp, logp2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=1e-14)


def test_masked_tail_equals_truncated_row():
    rng = np.random.default_rng(11)
    x = _rand_bf16(rng, 2, 100)
    xm = x.copy()
    xm[:, 60:] = 0xFF80  # -inf
    y = np.array([3, 59], dtype=np.int64)
    g = np.array([1.0, -1.0], dtype=np.float32)
    logp_m, lse_m = oracle.forward(xm, y, IGN)
    logp_t, lse_t = oracle.forward(np.ascontiguousarray(x[:, :60]), y, IGN)
    np.testing.assert_allclose(logp_m, logp_t, rtol=0, atol=1e-13)
    d = oracle.backward(xm, y, g, IGN)
    assert np.all(d[:, 60:] == 0.0) and np.all(np.isfinite(d))


def test_strided_rows_ignore_padding_columns():
    rng = np.random.default_rng(12)
    x = _rand_bf16(rng, 3, 64)
    y = np.array([1, 2, 3], dtype=np.int64)
    logp, lse = oracle.forward(np.ascontiguousarray(x[:, :50]), y, IGN)
    logp2, lse2 = oracle.forward(x, y, IGN, v=50)
    assert np.array_equal(logp, logp2) and np.array_equal(lse, lse2)


# ---------------------------------------------------------------- partials and merge


@pytest.mark.parametrize("v,w,k", [(1031, 72, 16), (151936, 9496, 16), (151936, 75968, 2),
                                   (151936, 37984, 4), (255, 16, 16), (9, 8, 16)])
def test_merge_of_partials_equals_unsharded_lse(v, w, k):
    rng = np.random.default_rng(13)
    n = 3 if v > 10000 else 16
    x = _rand_bf16(rng, n, v, sigma=2.5)
    pm, ps = oracle.range_partials(x, w, k)
    lse = oracle.merge_partials(pm, ps)
    _, lse_ref = oracle.forward(x, np.zeros(n, dtype=np.int64), IGN)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=0)
    xv = oracle.bf16_to_f64(x)
    for j in range(k):
        c0, c1 = min(j * w, v), min((j + 1) * w, v)
        if c0 == c1:
            assert np.all(pm[:, j] == -np.inf) and np.all(ps[:, j] == 0.0)
        else:
            assert np.array_equal(pm[:, j], xv[:, c0:c1].max(axis=1))


def test_identity_partials_change_nothing():
    rng = np.random.default_rng(14)
    x = _rand_bf16(rng, 4, 500)
    pm, ps = oracle.range_partials(x, 125, 4)
    lse = oracle.merge_partials(pm, ps)
    pm2 = np.concatenate([pm, np.full((4, 3), -np.inf)], axis=1)
    ps2 = np.concatenate([ps, np.zeros((4, 3))], axis=1)
    assert np.array_equal(oracle.merge_partials(pm2, ps2), lse)
    assert np.all(oracle.merge_partials(np.full((2, 3), -np.inf), np.zeros((2, 3))) == -np.inf)


def test_single_partial_merge_is_m_plus_log_s():
    pm = np.array([[3.0], [-2.0]])
    ps = np.array([[5.0], [1.0]])
    np.testing.assert_allclose(oracle.merge_partials(pm, ps), [3 + math.log(5.0), -2.0],
                               rtol=1e-15)


# ---------------------------------------------------------------- the comparison routine


def test_backward_compare_counts_planted_mistakes():
    rng = np.random.default_rng(15)
    n, v = 12, 333
    x = _rand_bf16(rng, n, v)
    y = rng.integers(0, v, n).astype(np.int64)
    y[3] = IGN
    g = rng.standard_normal(n).astype(np.float32)
    d = oracle.backward(x, y, g, IGN)
    cr = oracle.round_bf16(d)
    st = oracle.backward_compare(x, y, g, cr, IGN)
    assert st["n_compared"] == n * v
    assert st["n_not_correctly_rounded"] == 0
    assert st["max_abs_diff"] == st["max_rounding_gap"]
    assert st["max_abs_d"] == np.abs(d).max()
    bad = cr.copy()
    bad[5, 17] ^= 1          # one ulp off
    bad[3, 0] = 0x3F80       # an inactive row that is not zero
    st2 = oracle.backward_compare(x, y, g, bad, IGN)
    assert st2["n_not_correctly_rounded"] == 2
    assert st2["max_abs_diff"] >= 1.0
    # strided output with padding columns
    wide = np.zeros((n, v + 5), dtype=np.uint16)
    wide[:, :v] = cr
    assert oracle.backward_compare(x, y, g, wide, IGN)["n_not_correctly_rounded"] == 0


def test_workload_recipe_shapes():
    x, y, g = workloads.make("tiny")
    assert x.shape == (64, 1024) and x.dtype == torch.bfloat16
    assert int((y == IGN).sum()) == 6 and g.dtype == torch.float32
    x2, y2, g2 = workloads.make("tiny")
    assert torch.equal(x.view(torch.int16), x2.view(torch.int16)) and torch.equal(y, y2)
    lw = workloads.WORKLOADS["long"]
    gl = workloads.grads(64, lw.grad, 0)
    assert torch.all(gl.abs() == 1.0 / 64)


# ---------------------------------------------------------------- variants: FP16 / FP32 logits,
# temperature, explicit active mask


def test_f16_widening_matches_numpy():
    b = np.arange(0, 65536, dtype=np.uint16)
    got = oracle.f16_to_f64(b)
    want = b.view(np.float16).astype(np.float64)
    finite = ~np.isnan(want)
    assert np.array_equal(got[finite], want[finite]) and np.all(np.isnan(got[~finite]))


def test_round_f16_matches_numpy_and_known_values():
    rng = np.random.default_rng(20)
    d = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
                        (1 + (2 * rng.integers(0, 1024, 500) + 1) * 2.0 ** -11)
                        * 2.0 ** rng.integers(-14, 15, 500),          # ties
                        rng.integers(1, 2048, 200) * 2.0 ** -25])      # subnormal ties
    got = oracle.round_f16(d)
    with np.errstate(over="ignore"):
        want = d.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    for val, bits in [(65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00), (2.0 ** -24, 0x0001),
                      (2.0 ** -25, 0x0000), (3 * 2.0 ** -25, 0x0002), (-1.0, 0xBC00),
                      (1.0 + 2.0 ** -11, 0x3C00), (1.0 + 3 * 2.0 ** -11, 0x3C02)]:
        assert int(oracle.round_f16(val)) == bits, (val, hex(int(oracle.round_f16(val))))


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_forward_other_dtypes_match_torch(dtype):
    rng = np.random.default_rng(21)
    n, v = 12, 1031
    f = (rng.standard_normal((n, v)) * 3.0).astype(np.float32)
    x = f.astype(np.float16).view(np.uint16) if dtype == "f16" else f
    xv = (x.view(np.float16).astype(np.float64) if dtype == "f16" else f.astype(np.float64))
    y = rng.integers(0, v, n).astype(np.int64)
    for scale in (1.0, float(np.float32(1 / 0.7))):
        logp, lse = oracle.forward(x, y, dtype=dtype, scale=scale)
        t = torch.from_numpy(xv) * scale
        ref = torch.log_softmax(t, 1).gather(1, torch.from_numpy(y)[:, None])[:, 0].numpy()
        np.testing.assert_allclose(logp, ref, rtol=0, atol=1e-11)
        np.testing.assert_allclose(lse, torch.logsumexp(t, 1).numpy(), rtol=1e-13)


@pytest.mark.parametrize("case", __import__("golden").temperature_forms(), ids=lambda c: c["name"])
def test_temperature_closed_forms(case):
    x = _bits(case["logits"])[None, :]
    y = np.array([case["target"]], dtype=np.int64)
    logp, lse = oracle.forward(x, y, IGN, scale=case["scale"])
    assert abs(logp[0] - case["logp"]) <= 1e-13 * max(1.0, abs(case["logp"]))
    assert abs(lse[0] - case["lse"]) <= 1e-13 * max(1.0, abs(case["lse"]))
    if case["dlogits"] is not None:
        d = oracle.backward(x, y, np.array([case["grad"]], np.float32), IGN, scale=case["scale"])
        np.testing.assert_allclose(d[0], case["dlogits"], rtol=0, atol=1e-14)


def test_temperature_gradient_by_richardson_central_differences():
    """With a temperature the gradient with respect to the unscaled logits
    carries the factor s (chain rule); central differences of the oracle's own
    forward see it."""
    rng = np.random.default_rng(22)
    v = 10
    base = rng.integers(2, 4, v).astype(np.float64) + rng.integers(0, 8, v) * 2.0 ** -3
    y = np.array([3], dtype=np.int64)
    g = np.array([1.5], dtype=np.float32)
    for scale in (0.5, float(np.float32(1 / 0.7)), 3.0):
        d = oracle.backward(_bits(base)[None, :], y, g, IGN, scale=scale)[0]
        for c in range(v):
            est = []
            for h in (2.0 ** -5, 2.0 ** -6):
                xp, xm = base.copy(), base.copy()
                xp[c] += h
                xm[c] -= h
                lp = oracle.forward(_bits(xp)[None, :], y, IGN, scale=scale)[0][0]
                lm = oracle.forward(_bits(xm)[None, :], y, IGN, scale=scale)[0][0]
                est.append((lp - lm) / (2 * h))
            rich = (4 * est[1] - est[0]) / 3
            assert abs(1.5 * rich - d[c]) < 2e-6 * scale ** 3, (scale, c, rich, d[c])


def test_active_mask():
    rng = np.random.default_rng(23)
    x = _rand_bf16(rng, 6, 50)
    y = rng.integers(0, 50, 6).astype(np.int64)
    y[4] = IGN
    g = np.ones(6, dtype=np.float32)
    mask = np.array([1, 0, 1, 0, 1, 1], dtype=np.uint8)
    logp0, lse0 = oracle.forward(x, y, IGN)
    logp, lse = oracle.forward(x, y, IGN, mask=mask)
    d0 = oracle.backward(x, y, g, IGN)
    d = oracle.backward(x, y, g, IGN, mask=mask)
    for t in range(6):
        if mask[t] and y[t] != IGN:
            assert logp[t] == logp0[t] and np.array_equal(d[t], d0[t])
        else:
            assert logp[t] == 0.0 and np.all(d[t] == 0.0)
    assert np.array_equal(lse, lse0)  # the LSE is computed for every row


@pytest.mark.parametrize("out_dtype", ["f16", "f32"])
def test_backward_compare_other_out_dtypes(out_dtype):
    rng = np.random.default_rng(24)
    n, v = 6, 200
    f = (rng.standard_normal((n, v)) * 2).astype(np.float32)
    x = f.astype(np.float16).view(np.uint16) if out_dtype == "f16" else f
    y = rng.integers(0, v, n).astype(np.int64)
    g = rng.standard_normal(n).astype(np.float32)
    d = oracle.backward(x, y, g, dtype=out_dtype)
    cr = oracle.round_f16(d) if out_dtype == "f16" else d.astype(np.float32)
    st = oracle.backward_compare(x, y, g, cr, dtype=out_dtype)
    assert st["n_not_correctly_rounded"] == 0 and st["n_compared"] == n * v
    bad = cr.copy()
    if out_dtype == "f16":
        bad[2, 5] ^= 1
    else:
        bad[2, 5] = np.nextafter(bad[2, 5], np.float32(np.inf))
    assert oracle.backward_compare(x, y, g, bad, dtype=out_dtype)["n_not_correctly_rounded"] == 1


def test_scaled_range_partials_merge_to_scaled_lse():
    rng = np.random.default_rng(25)
    x = _rand_bf16(rng, 4, 1031, sigma=3.0)
    s = float(np.float32(1 / 0.7))
    pm, ps = oracle.range_partials(x, 72, 16, scale=s)
    _, lse = oracle.forward(x, np.zeros(4, np.int64), scale=s)
    np.testing.assert_allclose(oracle.merge_partials(pm, ps), lse, rtol=1e-13)
    xv = oracle.bf16_to_f64(x)
    assert np.array_equal(pm[:, 0], (s * xv[:, :72]).max(axis=1))


# ---------------------------------------------------------------- GRPO loss on the logp path


def _grpo_case(rng, n=12):
    lp = -rng.uniform(0.5, 6.0, n)
    old = lp + rng.uniform(-0.6, 0.6, n)
    ref = lp + rng.uniform(-0.5, 0.5, n)
    adv = rng.standard_normal(n)
    return lp, old, ref, adv


def test_grpo_kl_zero_identity():
    """logp == old_logp: every ratio is exactly 1, the clipped and unclipped
    terms agree, pg = -A exactly and the gradient is -A times the weight."""
    rng = np.random.default_rng(30)
    lp, _, _, adv = _grpo_case(rng)
    cu = np.array([0, 5, 12])
    for mode, w in [("token_mean", np.full(12, 1 / 12)),
                    ("seq_mean_token_mean", np.r_[np.full(5, 1 / 10), np.full(7, 1 / 14)]),
                    ("seq_mean_token_sum", np.full(12, 1 / 2))]:
        loss, g = oracle.grpo_loss(lp, lp, adv, cu_seqlens=cu, mode=mode)
        assert np.array_equal(g, -adv * w)
        assert abs(loss - np.sum(-adv * w)) < 1e-15


def test_grpo_clip_branches_closed_forms():
    eps = 0.2
    cases = [  # (ratio, A, loss, dloss/dlogp)
        (1.5, 2.0, -2.0 * 1.2, 0.0),          # clipped above: constant
        (1.5, -2.0, 2.0 * 1.5, 2.0 * 1.5),    # negative advantage: unclipped term is the max
        (0.5, 2.0, -2.0 * 0.5, -2.0 * 0.5),   # below 1 - eps with A > 0: unclipped is the max
        (0.5, -2.0, 2.0 * 0.8, 0.0),          # below 1 - eps with A < 0: clipped, constant
        (1.1, 3.0, -3.0 * 1.1, -3.0 * 1.1),   # inside the trust region
    ]
    for r, a, want_l, want_g in cases:
        old = np.array([-2.0])
        lp = old + math.log(r)
        loss, g = oracle.grpo_loss(lp, old, np.array([a]), eps_lo=eps, eps_hi=eps)
        assert abs(loss - want_l) < 1e-12 and abs(g[0] - want_g) < 1e-12, (r, a, loss, g)


def test_grpo_kl_closed_form():
    lp = np.array([-1.0, -2.0, -3.0])
    d = np.array([0.0, 0.3, -0.4])
    loss, g = oracle.grpo_loss(lp, lp, np.zeros(3), ref_logp=lp + d, beta=0.5)
    kl = np.exp(d) - d - 1
    assert abs(loss - 0.5 * kl.mean()) < 1e-15
    np.testing.assert_allclose(g, 0.5 * (1 - np.exp(d)) / 3, rtol=0, atol=1e-15)


@pytest.mark.parametrize("mode", ["token_mean", "seq_mean_token_mean", "seq_mean_token_sum"])
def test_grpo_gradient_by_richardson_central_differences(mode):
    rng = np.random.default_rng(31)
    lp, old, ref, adv = _grpo_case(rng)
    cu = np.array([0, 4, 4, 12])              # includes an empty sequence
    mask = np.ones(12, np.uint8)
    mask[[2, 9]] = 0
    kw = dict(ref_logp=ref, mask=mask, cu_seqlens=cu, mode=mode, eps_lo=0.2, eps_hi=0.28,
              beta=0.05)
    _, g = oracle.grpo_loss(lp, old, adv, **kw)
    r = np.exp(lp - old)
    for t in range(12):
        if min(abs(r[t] - 0.8), abs(r[t] - 1.28)) < 1e-3:
            continue   # at a clip kink the derivative is one-sided
        est = []
        for h in (1e-4, 5e-5):
            p, m = lp.copy(), lp.copy()
            p[t] += h
            m[t] -= h
            est.append((oracle.grpo_loss(p, old, adv, **kw)[0] - oracle.grpo_loss(m, old, adv, **kw)[0])
                       / (2 * h))
        rich = (4 * est[1] - est[0]) / 3
        assert abs(rich - g[t]) < 1e-9, (mode, t, rich, g[t])
    assert g[2] == 0 and g[9] == 0


def test_grpo_reduction_invariants():
    rng = np.random.default_rng(32)
    lp, old, ref, adv = _grpo_case(rng, n=12)
    cu = np.array([0, 4, 8, 12])              # equal lengths
    l0, g0 = oracle.grpo_loss(lp, old, adv, ref_logp=ref, beta=0.1, cu_seqlens=cu)
    l1, g1 = oracle.grpo_loss(lp, old, adv, ref_logp=ref, beta=0.1, cu_seqlens=cu,
                              mode="seq_mean_token_mean")
    l2, g2 = oracle.grpo_loss(lp, old, adv, ref_logp=ref, beta=0.1, cu_seqlens=cu,
                              mode="seq_mean_token_sum")
    assert abs(l0 - l1) < 1e-14 and np.allclose(g0, g1, rtol=1e-14, atol=0)
    assert abs(l2 - 4 * l0) < 1e-13 and np.allclose(g2, 4 * g0, rtol=1e-14, atol=0)
    # a masked token is the same as a removed one
    mask = np.ones(12, np.uint8)
    mask[5] = 0
    lm, gm = oracle.grpo_loss(lp, old, adv, mask=mask)
    keep = np.arange(12) != 5
    lr, gr = oracle.grpo_loss(lp[keep], old[keep], adv[keep])
    assert abs(lm - lr) < 1e-15 and np.allclose(gm[keep], gr, rtol=1e-14, atol=0) and gm[5] == 0
    # a global normaliser rescales
    ln, gn = oracle.grpo_loss(lp, old, adv, normalizer=48.0)
    la, ga = oracle.grpo_loss(lp, old, adv)
    assert abs(ln - la / 4) < 1e-15 and np.allclose(gn, ga / 4, rtol=1e-14, atol=0)


def test_grpo_tokens_outside_sequences_are_inactive():
    """Sequences covering [3, 9) of 12 tokens: the loss equals the loss of the
    covered slice alone, the uncovered tokens' gradients are exactly 0 (the
    same as masking them out)."""
    rng = np.random.default_rng(33)
    lp, old, ref, adv = _grpo_case(rng, n=12)
    for mode in ("token_mean", "seq_mean_token_mean", "seq_mean_token_sum"):
        kw = dict(ref_logp=ref, beta=0.1, mode=mode)
        lo_, g = oracle.grpo_loss(lp, old, adv, cu_seqlens=np.array([3, 5, 9]), **kw)
        kw_s = dict(kw, ref_logp=ref[3:9])
        ls, gs = oracle.grpo_loss(lp[3:9], old[3:9], adv[3:9], cu_seqlens=np.array([0, 2, 6]), **kw_s)
        assert abs(lo_ - ls) < 1e-15 and np.array_equal(g[3:9], gs)
        assert np.all(g[:3] == 0) and np.all(g[9:] == 0)
        mask = np.zeros(12, np.uint8)
        mask[3:9] = 1
        # masking [0, 3) and [9, 12) inside sequences [0, 5), [5, 12) leaves the
        # same active tokens per sequence: the same loss and gradient
        lm, gm = oracle.grpo_loss(lp, old, adv, mask=mask, cu_seqlens=np.array([0, 5, 12]), **kw)
        assert abs(lm - lo_) < 1e-15 and np.array_equal(gm, g)


# ---- fused LM head + logp (linear_logp) -------------------------------------

def _bf16_of(a):
    return workloads.bf16_bits(torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16))


def test_linear_logp_matches_numpy_matmul_and_torch_log_softmax():
    """A library chain: numpy float64 matmul of the widened BF16 operands, then
    torch float64 log_softmax / logsumexp of s z; non-square shapes (a
    transposed operand fails), ragged d, padded row strides, temperature, mask,
    ignore and out-of-range targets."""
    rng = np.random.default_rng(11)
    n, d, v = 7, 72, 333
    h = _bf16_of(rng.standard_normal((n, d + 8)))
    w = _bf16_of(rng.standard_normal((v, d + 24)) * 0.1)
    h[:, d:] = 0x7F7F   # padding columns hold huge values: must be ignored
    w[:, d:] = 0xFF7F
    y = np.array([0, 5, IGN, v - 1, 17, v, 200], dtype=np.int64)
    mask = np.array([1, 1, 1, 1, 0, 1, 1], dtype=np.uint8)
    s = float(np.float32(1 / 0.7))
    lp, lse, bound = oracle.linear_logp(h, w, y, d=d, scale=s, mask=mask, with_bound=True)
    hd = oracle.bf16_to_f64(h)[:, :d]
    wd = oracle.bf16_to_f64(w)[:, :d]
    z = torch.from_numpy(hd @ wd.T) * s
    ref_lse = torch.logsumexp(z, dim=1).numpy()
    ls = torch.log_softmax(z, dim=1).numpy()
    act = (mask != 0) & (y >= 0) & (y < v)
    ref_lp = np.where(act, ls[np.arange(n), np.clip(y, 0, v - 1)], 0.0)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lp, ref_lp, rtol=0, atol=1e-12)
    assert np.all(lp[~act] == 0.0)
    np.testing.assert_allclose(bound, np.max(np.abs(hd) @ np.abs(wd).T, axis=1), rtol=1e-13)


def test_linear_logp_one_hot_weights_select_hidden_columns():
    """Weight rows e_{p(j)}: the logits are the hidden columns p(j) exactly, so
    the result equals the (separately pinned) logits oracle on those columns."""
    rng = np.random.default_rng(12)
    n, d, v = 9, 64, 48
    h = _bf16_of(rng.standard_normal((n, d)) * 2)
    p = rng.permutation(d)[:v]
    w = np.zeros((v, d), dtype=np.uint16)
    w[np.arange(v), p] = 0x3F80          # BF16 1.0
    y = rng.integers(0, v, n)
    y[3] = IGN
    for s in (1.0, float(np.float32(1 / 0.7))):
        lp, lse = oracle.linear_logp(h, w, y, scale=s)
        cols = np.ascontiguousarray(h[:, p])
        want_lp, want_lse = oracle.forward(cols, y, scale=s)
        np.testing.assert_allclose(lp, want_lp, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-15)


def test_linear_logp_equal_weight_rows_give_minus_log_v():
    """All weight rows equal: every logit of a row is the same, logp = -log V
    and LSE = z + log V (closed form)."""
    rng = np.random.default_rng(13)
    n, d, v = 5, 40, 1000
    h = _bf16_of(rng.standard_normal((n, d)))
    row = _bf16_of(rng.standard_normal((1, d)) * 0.3)
    w = np.repeat(row, v, axis=0)
    y = rng.integers(0, v, n)
    lp, lse = oracle.linear_logp(h, w, y)
    z = oracle.bf16_to_f64(h) @ oracle.bf16_to_f64(row)[0]
    np.testing.assert_allclose(lp, -math.log(v), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, z + math.log(v), rtol=0, atol=1e-12)


def test_linear_logp_hand_example():
    """h = (1, -2); weight rows (3, 4) and (0.5, 0.25): z = (-5, 0), so
    logp(y=0) = -log(1 + e^5), logp(y=1) = -log(1 + e^-5), LSE = log(1 + e^-5),
    and the bound is max(3 + 8, 0.5 + 0.5) = 11."""
    h = _bits([[1.0, -2.0], [1.0, -2.0]])
    w = _bits([[3.0, 4.0], [0.5, 0.25]])
    lp, lse, b = oracle.linear_logp(h, w, np.array([0, 1]), with_bound=True)
    assert lp[0] == pytest.approx(-math.log1p(math.exp(5.0)), abs=1e-14)
    assert lp[1] == pytest.approx(-math.log1p(math.exp(-5.0)), abs=1e-14)
    assert lse[0] == pytest.approx(math.log1p(math.exp(-5.0)), abs=1e-14)
    assert b[0] == 11.0 and b[1] == 11.0


def _torch_linear_grads(h, w, y, g, s, mask=None):
    """torch float64 autograd of sum_t g_t logp_t through z = H W^T."""
    H = torch.from_numpy(oracle.bf16_to_f64(h)).requires_grad_(True)
    W = torch.from_numpy(oracle.bf16_to_f64(w)).requires_grad_(True)
    ls = torch.log_softmax(s * (H @ W.T), dim=1)
    v = w.shape[0]
    act = (y >= 0) & (y < v)
    if mask is not None:
        act &= mask != 0
    sel = ls[torch.arange(len(y)), torch.from_numpy(np.clip(y, 0, v - 1))]
    F = (sel * torch.from_numpy(g.astype(np.float64)) * torch.from_numpy(act.astype(np.float64))).sum()
    F.backward()
    return H.grad.numpy(), W.grad.numpy()


def test_linear_backward_matches_torch_autograd():
    """The unrounded oracle gradient equals torch float64 autograd of
    sum g logp through H W^T (non-square shapes, temperature, mask, ignore)."""
    rng = np.random.default_rng(31)
    n, d, v = 6, 40, 97
    h = _bf16_of(rng.standard_normal((n, d)))
    w = _bf16_of(rng.standard_normal((v, d)) * 0.3)
    y = np.array([0, 96, IGN, 5, 50, 200], dtype=np.int64)
    g = rng.standard_normal(n).astype(np.float32)
    mask = np.array([1, 1, 1, 0, 1, 1], dtype=np.uint8)
    s = float(np.float32(1 / 0.7))
    dh, dw = oracle.linear_backward(h, w, y, g, scale=s, mask=mask, round_dz=False)
    th, tw = _torch_linear_grads(h, w, y, g, s, mask)
    np.testing.assert_allclose(dh, th, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dw, tw, rtol=0, atol=1e-12)
    assert np.all(dh[[2, 3, 5]] == 0)


def test_linear_backward_by_central_differences():
    """d/dH and d/dW of sum g logp (the oracle's forward) by Richardson-
    extrapolated central differences on BF16-exact perturbations."""
    rng = np.random.default_rng(32)
    n, d, v = 3, 16, 11
    h = _bf16_of(rng.uniform(0.5, 1.0, (n, d)))
    w = _bf16_of(rng.uniform(0.5, 1.0, (v, d)))
    y = np.array([1, 7, 10], dtype=np.int64)
    g = np.array([0.5, -1.5, 2.0], dtype=np.float32)
    dh, dw = oracle.linear_backward(h, w, y, g, round_dz=False)

    def F(hh, ww):
        lp, _ = oracle.linear_logp(hh, ww, y)
        return float(np.dot(lp, g.astype(np.float64)))

    def bump(a, idx, k):       # add k BF16 units in the last place (values in [0.5, 1): 2^-8)
        b = a.copy()
        b[idx] = _bf16_of(np.array([oracle.bf16_to_f64(a[idx]) + k * 2.0 ** -8]))[0]
        return b

    for arr, which, idx, ref in ((h, 0, (1, 3), dh[1, 3]), (w, 1, (7, 5), dw[7, 5]), (w, 1, (2, 0), dw[2, 0])):
        def Fk(k):
            hh, ww = (bump(h, idx, k), w) if which == 0 else (h, bump(w, idx, k))
            return F(hh, ww)
        e = 2.0 ** -8
        c1 = (Fk(1) - Fk(-1)) / (2 * e)
        c2 = (Fk(2) - Fk(-2)) / (4 * e)
        rich = (4 * c1 - c2) / 3
        assert rich == pytest.approx(ref, rel=1e-5, abs=1e-8), (which, idx, rich, ref)


def test_linear_backward_rounded_dz_equals_bf16_dz_times_weights():
    """round_dz: dH and dW are the BF16-rounded dZ times W and H exactly (numpy
    float64 matmul), and dZ rows sum to ~0 for active rows."""
    rng = np.random.default_rng(33)
    n, d, v = 5, 24, 300
    h = _bf16_of(rng.standard_normal((n, d)))
    w = _bf16_of(rng.standard_normal((v, d)) * 0.2)
    y = rng.integers(0, v, n)
    g = rng.standard_normal(n).astype(np.float32)
    dh, dw, dz = oracle.linear_backward(h, w, y, g, with_dz=True)
    _, _, dz0 = oracle.linear_backward(h, w, y, g, round_dz=False, with_dz=True)
    assert np.array_equal(dz, oracle.bf16_to_f64(oracle.round_bf16(dz0)))
    np.testing.assert_allclose(dh, dz @ oracle.bf16_to_f64(w), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, dz.T @ oracle.bf16_to_f64(h), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dz0.sum(axis=1), 0.0, atol=1e-12)
