"""Size extremes of the logits path on the GPU.

* Very wide rows: V = 2^24 + 37 (ragged), three rows of random logits, the
  whole forward and backward against the FP64 oracle.  Tiles are 2^20 wide,
  every lane walks thousands of groups.
* A row wider than 2^31 elements (V = 2^31 + 24, 4.3 GB of BF16): the plain
  forward (the bulk-copy forward is for rows below 2^31) and the backward's
  64-bit column arithmetic, against closed forms.  The row is two-level (0 in
  the first half, 1 in the second), so every per-lane sum is an exact integer
  in binary32 and the expected values are exact: with H = V / 2,
      LSE = log H + log(1 + e),   logp(target in the upper half) = 1 - LSE,
      d = g (onehot - p),  p = e^0 / (H (1 + e)) below, e / (H (1 + e)) above.
  (Random logits this wide are outside the accuracy envelope of binary32
  per-lane sums; the two-level row checks the indexing, not the rounding.)
"""

import math

import numpy as np
import pytest
import torch

import oracle
import selected_token_logprob_gb300 as flp
import workloads
from parity_util import bits, check_backward, check_forward, run

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    flp._lib.load(build_if_missing=True)


def test_very_wide_rows_against_oracle():
    v = (1 << 24) + 37
    wl = workloads.Workload("wide", 3, v, 2.0, 8.0, 0.0, "normal", seed=21)
    x, y, g = workloads.make(wl, device=DEV)
    logp, lse, dl = run(x, y, g)
    yn, gn = y.cpu().numpy(), g.cpu().numpy()
    check_forward(bits(x), yn, logp, lse)
    check_backward(bits(x), yn, gn, dl)


def test_row_wider_than_2_31_elements():
    v = (1 << 31) + 24
    h = v // 2
    free = torch.cuda.mem_get_info()[0]
    if free < 3 * v * 2:
        pytest.skip("needs about 13 GB of free device memory")
    x = torch.zeros((1, v), dtype=torch.bfloat16, device=DEV)
    x[0, h:] = 1.0
    y = torch.tensor([v - 1], dtype=torch.int64, device=DEV)
    g = torch.tensor([3.0], dtype=torch.float32, device=DEV)
    logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True)
    lse_exact = math.log(h) + math.log1p(math.e)
    assert abs(lse.item() - lse_exact) <= 1e-4 + float(np.spacing(np.float32(lse_exact)))
    assert abs(logp.item() - (1.0 - lse_exact)) <= 1e-4
    dl = flp.fused_logp_backward(x, y, lse, g, lse_lo=lo)
    del x
    torch.cuda.synchronize()
    p_lo = 1.0 / (h * (1.0 + math.e))
    p_hi = math.e / (h * (1.0 + math.e))
    want = {"low": -3.0 * p_lo, "high": -3.0 * p_hi, "target": 3.0 * (1.0 - p_hi)}
    # positions across both halves, the 2^31 boundary and the ragged end
    cols = {"low": [0, 1, 12345, h - 1], "high": [h, h + 1, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, v - 2],
            "target": [v - 1]}
    for kind, cs in cols.items():
        got = dl[0, torch.tensor(cs, device=DEV)].float().cpu().numpy().astype(np.float64)
        ref = oracle.bf16_to_f64(oracle.round_bf16(np.full(len(cs), want[kind])))
        ulp = np.spacing(np.abs(ref).astype(np.float32)) * 2.0 ** 16     # one BF16 ulp
        assert np.all(np.abs(got - ref) <= ulp), (kind, got, ref)
    # every element of each half holds the same value (no stray writes)
    for a, b in ((0, h), (h, v - 1)):
        mn, mx = torch.aminmax(dl[0, a:b])
        assert mn.item() == mx.item(), (a, b, mn.item(), mx.item())
    assert flp.flp_device_error(0) == 0
