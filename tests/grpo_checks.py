"""Comparison helpers for the GRPO loss tests (test infrastructure): each
token's normaliser weight from the definitions, and the gradient comparison
that accepts either branch at a clip bound."""

import numpy as np


def _token_weights(n, mask, cu, mode, normalizer=0.0):
    """Each token's normaliser weight by the definitions (token mean 1/D,
    sequence mean of token means 1/(S_active n_s), of token sums
    1/S_active); 0 for inactive tokens and tokens in no sequence."""
    act = np.ones(n, bool) if mask is None else mask.astype(bool)
    if cu is None:
        seg = np.zeros(n, np.int64)
        nseq = 1
    else:
        seg = np.searchsorted(cu, np.arange(n), side="right") - 1
        nseq = len(cu) - 1
        act &= (seg >= 0) & (seg < nseq)
    cnt = np.bincount(seg[act], minlength=nseq)
    den = float(act.sum()) if mode == "token_mean" else float((cnt > 0).sum())
    if normalizer > 0:
        den = normalizer
    w = np.zeros(n)
    if den > 0:
        if mode == "seq_mean_token_mean":
            w[act] = 1.0 / (den * cnt[seg[act]])
        else:
            w[act] = 1.0 / den
    return w


def _assert_grad(got, want, lp, old, adv, ref, beta, eps_lo, eps_hi, w, rtol=1e-5):
    """max |got - want| <= rtol max |want|, except at tokens whose ratio lies
    within 1e-6 of a clip bound: there the kernel's FP32 ratio and the
    oracle's FP64 one may take different branches (both correct to the
    precision), so either branch's gradient is accepted."""
    r = np.exp(lp - old)
    near = (np.abs(r - (1 - eps_lo)) <= 1e-6 * r) | (np.abs(r - (1 + eps_hi)) <= 1e-6 * r)
    tol = rtol * np.max(np.abs(want))
    far = ~near
    assert np.max(np.abs(got[far] - want[far]), initial=0.0) <= tol, np.max(np.abs(got[far] - want[far]))
    if near.any():
        kl = beta * (1 - np.exp(ref[near] - lp[near])) if ref is not None else 0.0
        unclipped = w[near] * (-adv[near] * r[near] + kl)
        clipped = w[near] * kl
        d = np.minimum(np.abs(got[near] - unclipped), np.abs(got[near] - clipped))
        assert np.max(d) <= tol, (np.max(d), int(near.sum()))
