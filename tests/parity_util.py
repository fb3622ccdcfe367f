"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare it with the FP64 oracle.

Tolerances (the stated targets of this path):
  logp     |GPU - FP64| <= 1e-4 absolute
  dlogits  max |GPU - FP64| <= max(2e-3 * max|d|, max |round_bf16(d) - d|),
           i.e. no worse than 2e-3 of the largest gradient or than the
           correctly rounded result itself; and at least 99.99% of the
           elements are exactly the correctly rounded BF16 of the FP64 value.
  lse      |GPU - FP64| <= 1e-4 + one binary32 ulp of the LSE (an FP32 LSE
           cannot be closer than half an ulp, which exceeds 1e-4 once
           |LSE| >= 1024).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import selected_token_logprob_gb300 as flp
import workloads

LOGP_ATOL = 1e-4
LSE_ATOL = 1e-4
GRAD_REL = 2e-3
MIN_CORRECTLY_ROUNDED = 0.9999


def run(x, y, g, ignore_index=-100, use_lse_lo=True):
    """Forward + backward through the C ABI; by default the backward gets the
    LSE's FP32 rounding residual (the path the autograd wrapper takes)."""
    if use_lse_lo:
        logp, lse, lse_lo = flp.fused_logp_forward(x, y, ignore_index, with_lse_lo=True)
    else:
        (logp, lse), lse_lo = flp.fused_logp_forward(x, y, ignore_index), None
    dl = flp.fused_logp_backward(x, y, lse, g, ignore_index, lse_lo=lse_lo)
    return logp, lse, dl


def bits(t: torch.Tensor) -> np.ndarray:
    return workloads.bf16_bits(t)


def check_forward(xb, y_np, logp, lse, ignore_index=-100, v=None):
    ref_logp, ref_lse = oracle.forward(xb, y_np, ignore_index, v=v)
    got_logp = logp.detach().cpu().numpy().astype(np.float64)
    got_lse = lse.detach().cpu().numpy().astype(np.float64)
    e_logp = float(np.max(np.abs(got_logp - ref_logp))) if len(ref_logp) else 0.0
    e_lse = float(np.max(np.abs(got_lse - ref_lse))) if len(ref_lse) else 0.0
    assert e_logp <= LOGP_ATOL, f"logp error {e_logp}"
    # an FP32 LSE cannot be closer than half its ulp: the bound is 1e-4 plus
    # one ulp of the reference value (matters only for |LSE| >= 1024)
    lse_tol = LSE_ATOL + np.spacing(np.abs(ref_lse).astype(np.float32)).astype(np.float64)
    finite = np.isfinite(ref_lse)
    assert np.all(np.abs(got_lse - ref_lse)[finite] <= lse_tol[finite]), f"lse error {e_lse}"
    inactive = ~((y_np >= 0) & (y_np < (xb.shape[1] if v is None else v)) & (y_np != ignore_index))
    assert np.all(got_logp[inactive] == 0.0)
    return {"max_abs_logp_err": e_logp, "max_abs_lse_err": e_lse}


def check_backward(xb, y_np, g_np, dl, ignore_index=-100, v=None, min_cr=MIN_CORRECTLY_ROUNDED):
    dlb = bits(dl) if isinstance(dl, torch.Tensor) else dl
    st = oracle.backward_compare(xb, y_np, g_np, dlb, ignore_index, v=v)
    bound = max(GRAD_REL * st["max_abs_d"], st["max_rounding_gap"])
    cr = 1.0 - st["n_not_correctly_rounded"] / max(1, st["n_compared"])
    st["bound"] = bound
    st["correctly_rounded"] = cr
    assert st["n_nonfinite"] == 0, st
    assert st["max_abs_diff"] <= bound, st
    assert cr >= min_cr, st
    return st
