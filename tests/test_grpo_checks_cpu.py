"""The GRPO test helpers pinned on the CPU: the per-token weights from the
normalisers' definitions equal the FP64 oracle's gradient weights (with
logp == old_logp the gradient is exactly -A times the weight), and the
branch-tolerant comparison rejects a wrong gradient away from the bounds."""

import numpy as np
import pytest

import oracle
from grpo_checks import _assert_grad, _token_weights

MODES = ["token_mean", "seq_mean_token_mean", "seq_mean_token_sum"]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("cu", [None, [0, 100, 100, 2500, 4000], [37, 900, 4100]])
@pytest.mark.parametrize("norm", [0.0, 321.0])
def test_token_weights_match_the_oracle(mode, cu, norm):
    rng = np.random.default_rng(5)
    n = 5000
    lp = -rng.uniform(0.1, 3, n)
    adv = rng.standard_normal(n)
    mask = (rng.random(n) > 0.2).astype(np.uint8)
    cu = None if cu is None else np.array(cu)
    _, g = oracle.grpo_loss(lp, lp, adv, mask=mask, cu_seqlens=cu, mode=mode, normalizer=norm)
    w = _token_weights(n, mask, cu, mode, norm)
    np.testing.assert_allclose(g, -adv * w, rtol=1e-14, atol=0)


def test_branch_tolerant_comparison():
    rng = np.random.default_rng(6)
    n = 2000
    lp = -rng.uniform(0.5, 3, n)
    old = lp + rng.uniform(-0.5, 0.5, n)
    adv = rng.standard_normal(n)
    old[7] = lp[7] - np.log1p(0.28)          # ratio exactly at 1 + eps_hi
    kw = dict(eps_lo=0.2, eps_hi=0.28)
    _, g = oracle.grpo_loss(lp, old, adv, **kw)
    w = _token_weights(n, None, None, "token_mean")
    _assert_grad(g.copy(), g, lp, old, adv, None, 0.0, 0.2, 0.28, w)
    flipped = g.copy()                        # the other branch at the bound: accepted
    flipped[7] = 0.0 if g[7] != 0 else w[7] * (-adv[7] * np.exp(lp[7] - old[7]))
    _assert_grad(flipped, g, lp, old, adv, None, 0.0, 0.2, 0.28, w)
    wrong = g.copy()                          # a wrong value away from the bounds: rejected
    far = int(np.argmax(np.abs(np.exp(lp - old) - 1.0) < 0.05))
    wrong[far] += 1e-3 * np.max(np.abs(g))
    with pytest.raises(AssertionError):
        _assert_grad(wrong, g, lp, old, adv, None, 0.0, 0.2, 0.28, w)
