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
* The GRPO loss over more than 2^31 tokens (n = 2^31 + 777, sequences whose
  bounds straddle 2^31): with logp == old_logp the ratio is exactly 1 and
  each gradient is exactly -A times the token's FP32 weight (the KL = 0
  identity of PR 5), checked bitwise at positions on both sides of 2^31 and
  at the ragged end; the loss against an FP64 sum on the device.
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


def test_grpo_beyond_2_31_tokens():
    n = (1 << 31) + 777
    free = torch.cuda.mem_get_info()[0]
    if free < 5 * n * 4:
        pytest.skip("needs about 43 GB of free device memory")
    gen = torch.Generator(device=DEV).manual_seed(61)
    lp = torch.empty(n, device=DEV).uniform_(-5.0, -0.1, generator=gen)
    adv = torch.randn(n, device=DEV, generator=gen)
    b1, b2 = 1000, (1 << 31) - 5
    cu = torch.tensor([0, b1, b2, n], dtype=torch.int64, device=DEV)
    lens = np.array([b1, b2 - b1, n - b2], dtype=np.float64)
    ws = torch.empty(flp.logp_grpo_loss_workspace_size(n, 3), dtype=torch.uint8, device=DEV)
    idx = [0, 1, b1 - 1, b1, 123456789, b2 - 1, b2, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, n - 2, n - 1]
    seq = np.searchsorted(np.array([0, b1, b2, n]), np.array(idx), side="right") - 1
    a_s = adv[torch.tensor(idx, device=DEV)].cpu().numpy().astype(np.float32)
    sums = [float(adv[lo_:hi_].double().sum().item()) for lo_, hi_ in ((0, b1), (b1, b2), (b2, n))]
    for mode in ("token_mean", "seq_mean_token_mean"):
        loss, grad = flp.logp_grpo_loss(lp, lp, adv, cu_seqlens=cu, mode=mode, workspace=ws)
        got = grad[torch.tensor(idx, device=DEV)].cpu().numpy()
        if mode == "token_mean":
            w = np.full(len(idx), np.float32(1.0 / n), np.float32)     # the weight rounded once from 1/n
            want_loss = -sum(sums) / n
        else:                                                       # (1/den)(1/n_s), each rounded
            w = np.float32(1.0) / np.float32(3.0) * (np.float32(1.0) / lens[seq].astype(np.float32))
            want_loss = -np.mean([sums[k] / lens[k] for k in range(3)])
        want = (-a_s) * w.astype(np.float32)
        assert np.array_equal(got.view(np.int32), want.view(np.int32)), (mode, got, want)
        assert abs(loss.item() - want_loss) <= 1e-5 * abs(want_loss) + 1e-7, (mode, loss.item(), want_loss)
    assert flp.flp_device_error(0) == 0
