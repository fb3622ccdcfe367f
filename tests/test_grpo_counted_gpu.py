"""The GRPO loss in two parts: the normaliser counts of a batch layout
(logp_grpo_loss_counts) and the token pass on those counts
(logp_grpo_loss_counted).  The weights depend on the layout only (issue #241
PR 5's declared normaliser), so the counts may be taken on another stream
while the logp are produced, or once for several calls.  Checked here:

* counts on a second stream (joined by an event), then the counted call on
  the current stream, give the whole call's loss, gradient and token losses
  bit for bit, in every mode, with and without a mask, sequences and KL;
* counted calls repeat on the same counts (the fold's ticket is left at 0),
  and a whole call leaves counts that a counted call can use;
* counts taken for another layout (mode, mask tensor, normaliser) make the
  loss and the sequences' gradients NaN rather than wrong numbers;
* a caller's uniform weight and an empty batch."""

import math

import pytest
import torch

import selected_token_logprob_gb300 as flp

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MODES = ["token_mean", "seq_mean_token_mean", "seq_mean_token_sum"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    flp._lib.load(build_if_missing=True)


def _case(n, seed, nseq):
    g = torch.Generator().manual_seed(seed)
    lp = -torch.rand(n, generator=g) * 6 - 0.05
    old = lp + (torch.rand(n, generator=g) - 0.5) * 1.2
    ref = lp + (torch.rand(n, generator=g) - 0.5) * 1.0
    adv = torch.randn(n, generator=g)
    mask = (torch.rand(n, generator=g) > 0.1).to(torch.uint8)
    cuts = torch.sort(torch.randint(0, n + 1, (nseq - 1,), generator=g)).values
    cu = torch.cat([torch.zeros(1, dtype=torch.int64), cuts, torch.full((1,), n, dtype=torch.int64)])
    return [t.to(DEV) for t in (lp, old, ref, adv, mask, cu)]


def _bits(t):
    return t.view(torch.int32)


# (mode, mask, cu_seqlens, KL); without cu_seqlens only the token mean here (the
# sequence modes then take the whole batch as one sequence: the next test)
_CASES = [(m, True, True, True) for m in MODES] + [(m, True, True, False) for m in MODES] + \
         [(m, False, True, True) for m in MODES] + [("token_mean", True, False, True)]


@pytest.mark.parametrize("mode, with_mask, with_cu, kl", _CASES)
def test_counted_equals_whole_call_bitwise(mode, with_mask, with_cu, kl):
    n = 300017                                      # ragged last chunk
    lp, old, ref, adv, mask, cu = _case(n, 41, 1000)
    mask = mask if with_mask else None
    cu = cu if with_cu else None
    kw = dict(ref_logp=ref if kl else None, active_mask=mask, cu_seqlens=cu, mode=mode, eps_lo=0.2,
              eps_hi=0.28, beta=0.04 if kl else 0.0, token_loss=True)
    want = flp.logp_grpo_loss(lp, old, adv, **kw)
    nseq = 0 if cu is None else cu.shape[0] - 1
    ws = torch.full((flp.logp_grpo_loss_workspace_size(n, nseq),), 0xAB, dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    flp.logp_grpo_loss_counts(n, active_mask=mask, cu_seqlens=cu, mode=mode, workspace=ws, stream=side)
    done = torch.cuda.Event()
    done.record(side)
    torch.cuda.current_stream().wait_event(done)
    for _ in range(3):                              # the same counts, three times
        got = flp.logp_grpo_loss(lp, old, adv, workspace=ws, counted=True, **kw)
        torch.cuda.synchronize()
        for u, v in zip(got, want):
            assert torch.equal(_bits(u), _bits(v)), mode
    assert flp.flp_device_error(0) == 0


@pytest.mark.parametrize("mode", ["seq_mean_token_mean", "seq_mean_token_sum"])
def test_counted_whole_batch_as_one_sequence(mode):
    n = 70001
    lp, old, ref, adv, mask, _ = _case(n, 42, 2)
    kw = dict(ref_logp=ref, active_mask=mask, mode=mode, beta=0.02)
    want = flp.logp_grpo_loss(lp, old, adv, **kw)
    ws = flp.logp_grpo_loss_counts(n, active_mask=mask, mode=mode)
    got = flp.logp_grpo_loss(lp, old, adv, workspace=ws, counted=True, **kw)
    for u, v in zip(got, want):
        assert torch.equal(_bits(u), _bits(v))


def test_whole_call_leaves_counts_for_counted_calls():
    n = 123457
    lp, old, ref, adv, mask, cu = _case(n, 43, 300)
    ws = torch.empty(flp.logp_grpo_loss_workspace_size(n, 300), dtype=torch.uint8, device=DEV)
    kw = dict(ref_logp=ref, active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean", beta=0.03)
    want = flp.logp_grpo_loss(lp, old, adv, workspace=ws, **kw)
    # another step's logp on the same batch layout (a second optimisation epoch)
    lp2 = lp + 0.01 * torch.randn(n, generator=torch.Generator(device=DEV).manual_seed(5), device=DEV)
    want2 = flp.logp_grpo_loss(lp2, old, adv, **kw)
    got2 = flp.logp_grpo_loss(lp2, old, adv, workspace=ws, counted=True, **kw)
    for u, v in zip(got2, want2):
        assert torch.equal(_bits(u), _bits(v))
    assert not torch.equal(_bits(want[1]), _bits(want2[1]))


@pytest.mark.parametrize("change", ["mode", "mask_tensor", "normalizer", "sequences"])
def test_counts_of_another_layout_give_nan(change):
    n = 65536
    lp, old, ref, adv, mask, cu = _case(n, 44, 200)
    nseq = 200
    ws = torch.empty(flp.logp_grpo_loss_workspace_size(n, nseq), dtype=torch.uint8, device=DEV)
    flp.logp_grpo_loss_counts(n, active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean", workspace=ws)
    kw = dict(ref_logp=ref, active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean", beta=0.01)
    if change == "mode":
        kw["mode"] = "seq_mean_token_sum"
    elif change == "mask_tensor":
        kw["active_mask"] = mask.clone()           # same contents, another tensor: counts not known for it
    elif change == "normalizer":
        kw["normalizer"] = 150.0
    else:
        kw["cu_seqlens"] = cu[:-1].clone()         # one sequence fewer
    loss, grad = flp.logp_grpo_loss(lp, old, adv, workspace=ws, counted=True, **kw)
    torch.cuda.synchronize()
    assert math.isnan(loss.item())
    inside = torch.zeros(n, dtype=torch.bool, device=DEV)
    c = kw["cu_seqlens"]
    inside[int(c[0]):int(c[-1])] = True
    active = inside & (kw["active_mask"] != 0)
    assert torch.isnan(grad[active]).all()
    # and the right counts make it right again
    good = flp.logp_grpo_loss(lp, old, adv, **kw)
    flp.logp_grpo_loss_counts(n, active_mask=kw["active_mask"], cu_seqlens=kw["cu_seqlens"], mode=kw["mode"],
                              normalizer=kw.get("normalizer", 0.0), workspace=ws)
    again = flp.logp_grpo_loss(lp, old, adv, workspace=ws, counted=True, **kw)
    for u, v in zip(again, good):
        assert torch.equal(_bits(u), _bits(v))


def test_counted_with_a_callers_weight_and_empty_batch():
    n = 50000
    lp, old, ref, adv, mask, cu = _case(n, 45, 64)
    kw = dict(active_mask=mask, cu_seqlens=cu, mode="token_mean", normalizer=12345.0, beta=0.0)
    want = flp.logp_grpo_loss(lp, old, adv, **kw)
    ws = torch.empty(flp.logp_grpo_loss_workspace_size(n, 64), dtype=torch.uint8, device=DEV)
    got = flp.logp_grpo_loss(lp, old, adv, workspace=ws, counted=True, **kw)   # nothing to count
    for u, v in zip(got, want):
        assert torch.equal(_bits(u), _bits(v))
    e = torch.empty(0, dtype=torch.float32, device=DEV)
    ws0 = flp.logp_grpo_loss_counts(0, active_mask=torch.empty(0, dtype=torch.uint8, device=DEV),
                                    mode="token_mean")
    loss, grad = flp.logp_grpo_loss(e, e, e, active_mask=torch.empty(0, dtype=torch.uint8, device=DEV),
                                    workspace=ws0, counted=True)
    assert loss.item() == 0.0 and grad.numel() == 0


def _edge_layout(kind, n, g):
    """cu_seqlens (host, int64) of a layout kind: empty sequences, tokens
    outside every sequence, one sequence, many tiny ones."""
    if kind == "empty_and_outside":
        cuts = torch.sort(torch.randint(n // 10, n - n // 10, (40,), generator=g)).values
        cuts = torch.cat([cuts, cuts[5:9]])                                 # repeated bounds: empty sequences
        return torch.sort(cuts).values.to(torch.int64)
    if kind == "one":
        return torch.tensor([0, n], dtype=torch.int64)
    step = 3                                                                # many tiny sequences
    return torch.arange(0, n + 1, step, dtype=torch.int64) if n % step == 0 else \
        torch.cat([torch.arange(0, n, step, dtype=torch.int64), torch.tensor([n])])


@pytest.mark.parametrize("seed, n, kind, density, mode, offset", [
    (1, 100, "one", 0.9, "seq_mean_token_mean", 0),             # a single partial chunk
    (2, 4099, "empty_and_outside", 0.7, "seq_mean_token_mean", 0),
    (3, 4099, "empty_and_outside", 0.0, "seq_mean_token_mean", 0),   # no active token: loss 0, grads 0
    (4, 65537, "tiny", 0.5, "seq_mean_token_sum", 0),
    (5, 65537, "empty_and_outside", 1.0, "token_mean", 0),
    (6, 33333, "empty_and_outside", 0.8, "seq_mean_token_mean", 1),  # arrays one element off alignment
    (7, 33333, "tiny", 0.8, "token_mean", 3),
])
def test_counted_edge_layouts_against_whole_call_and_oracle(seed, n, kind, density, mode, offset):
    import numpy as np

    import oracle
    from grpo_checks import _assert_grad, _token_weights

    g = torch.Generator().manual_seed(100 + seed)
    lp = -torch.rand(n, generator=g) * 6 - 0.05
    old = lp + (torch.rand(n, generator=g) - 0.5) * 1.2
    ref = lp + (torch.rand(n, generator=g) - 0.5) * 1.0
    adv = torch.randn(n, generator=g)
    mask = (torch.rand(n, generator=g) < density).to(torch.uint8)
    cu = _edge_layout(kind, n, g)

    def dev(t):   # a device view `offset` elements into a larger buffer (off alignment when offset > 0)
        buf = torch.zeros(n + offset, dtype=t.dtype, device=DEV)
        buf[offset:] = t.to(DEV)
        return buf[offset:]

    d_lp, d_old, d_ref, d_adv, d_mask = [dev(t) for t in (lp, old, ref, adv, mask)]
    d_cu = cu.to(DEV)
    kw = dict(ref_logp=d_ref, active_mask=d_mask, cu_seqlens=d_cu, mode=mode, eps_lo=0.2, eps_hi=0.28, beta=0.03)
    want = flp.logp_grpo_loss(d_lp, d_old, d_adv, **kw)
    ws = flp.logp_grpo_loss_counts(n, active_mask=d_mask, cu_seqlens=d_cu, mode=mode)
    got = flp.logp_grpo_loss(d_lp, d_old, d_adv, workspace=ws, counted=True, **kw)
    for u, v in zip(got, want):
        assert torch.equal(_bits(u), _bits(v))
    f64 = [t.double().numpy() for t in (lp, old, adv, ref)]
    want_l, want_g = oracle.grpo_loss(f64[0], f64[1], f64[2], ref_logp=f64[3], mask=mask.numpy(),
                                      cu_seqlens=cu.numpy(), mode=mode, eps_lo=0.2, eps_hi=0.28, beta=0.03)
    got_g = got[1].double().cpu().numpy()
    assert abs(got[0].item() - want_l) <= 1e-5 * abs(want_l) + 1e-7, (got[0].item(), want_l)
    if density == 0.0:
        assert got[0].item() == 0.0 and np.all(got_g == 0)
    else:
        w = _token_weights(n, mask.numpy(), cu.numpy(), mode)
        _assert_grad(got_g, want_g, f64[0], f64[1], f64[2], f64[3], 0.03, 0.2, 0.28, w)
