"""GPU parity of the GRPO loss on the logp path (RL-Kernel issue #241, PR 5)
against the FP64 oracle, its KL = 0 identity, determinism, and the whole
RL step: logits -> fused logp -> GRPO loss and d loss / d logp -> fused
backward, against the same chain in FP64.

Tolerances: loss |d| <= 1e-5 |loss| + 1e-7; grad max |d| <= 1e-5 max |g|
(FP32 per-token arithmetic with an accurate exp, FP64 sums)."""

import numpy as np
import pytest
import torch

import oracle
import selected_token_logprob_gb300 as flp
import workloads
from grpo_checks import _assert_grad, _token_weights

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MODES = ["token_mean", "seq_mean_token_mean", "seq_mean_token_sum"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    flp._lib.load(build_if_missing=True)


def _case(n, seed, nseq=None):
    g = torch.Generator().manual_seed(seed)
    lp = -torch.rand(n, generator=g) * 6 - 0.05
    old = lp + (torch.rand(n, generator=g) - 0.5) * 1.2
    ref = lp + (torch.rand(n, generator=g) - 0.5) * 1.0
    adv = torch.randn(n, generator=g)
    mask = (torch.rand(n, generator=g) > 0.1).to(torch.uint8)
    cu = None
    if nseq:
        cuts = torch.sort(torch.randint(0, n + 1, (nseq - 1,), generator=g)).values
        cu = torch.cat([torch.zeros(1, dtype=torch.int64), cuts, torch.full((1,), n, dtype=torch.int64)])
    return lp, old, ref, adv, mask, cu


def _dev(*ts):
    return [None if t is None else t.to(DEV) for t in ts]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("kl", [False, True])
def test_grpo_parity(mode, kl):
    lp, old, ref, adv, mask, cu = _case(32768, 1, nseq=257)
    kw = dict(mode=mode, eps_lo=0.2, eps_hi=0.28, beta=0.05 if kl else 0.0)
    loss, grad = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0] if kl else None,
                                    active_mask=_dev(mask)[0], cu_seqlens=_dev(cu)[0], **kw)
    want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                                      ref_logp=ref.double().numpy() if kl else None, mask=mask.numpy(),
                                      cu_seqlens=cu.numpy(), **kw)
    got_g = grad.double().cpu().numpy()
    assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7, (loss.item(), want_l)
    assert np.max(np.abs(got_g - want_g)) <= 1e-5 * np.max(np.abs(want_g)), np.max(np.abs(got_g - want_g))
    assert np.all(got_g[mask.numpy() == 0] == 0)


def test_grpo_whole_batch_and_normalizer():
    lp, old, ref, adv, mask, _ = _case(5000, 2)
    for mode in MODES:
        for norm in (0.0, 12345.0):
            loss, grad = flp.logp_grpo_loss(*_dev(lp, old, adv), active_mask=_dev(mask)[0], mode=mode,
                                            normalizer=norm)
            want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(),
                                              adv.double().numpy(), mask=mask.numpy(), mode=mode,
                                              normalizer=norm)
            assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7
            assert np.max(np.abs(grad.double().cpu().numpy() - want_g)) <= 1e-5 * np.max(np.abs(want_g))


def test_grpo_kl_zero_identity_bitwise():
    """logp == old_logp: ratio exactly 1, grad exactly -A times the FP32 weight."""
    lp, _, _, adv, _, _ = _case(4096, 3)
    loss, grad = flp.logp_grpo_loss(*_dev(lp, lp, adv))
    w = np.float32(1.0 / 4096)
    want = (-adv.numpy().astype(np.float32)) * w
    assert np.array_equal(grad.cpu().numpy(), want)


def test_grpo_deterministic_and_token_loss():
    lp, old, ref, adv, mask, cu = _case(20000, 4, nseq=100)
    args = (*_dev(lp, old, adv),)
    kw = dict(ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0], cu_seqlens=_dev(cu)[0],
              mode="seq_mean_token_mean", beta=0.1, token_loss=True)
    a = flp.logp_grpo_loss(*args, **kw)
    for _ in range(3):
        b = flp.logp_grpo_loss(*args, **kw)
        for u, v in zip(a, b):
            assert torch.equal(u.view(torch.int32), v.view(torch.int32))
    tl = a[2].cpu()
    assert torch.all(tl[mask == 0] == 0)


def test_grpo_edge_cases():
    lp, old, ref, adv, mask, _ = _case(100, 5)
    none = torch.zeros(100, dtype=torch.uint8)
    loss, grad = flp.logp_grpo_loss(*_dev(lp, old, adv), active_mask=_dev(none)[0])
    assert loss.item() == 0.0 and torch.all(grad == 0)
    cu = torch.tensor([0, 0, 50, 50, 100], dtype=torch.int64)   # empty sequences
    loss, grad = flp.logp_grpo_loss(*_dev(lp, old, adv), cu_seqlens=_dev(cu)[0],
                                    mode="seq_mean_token_mean")
    want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                                      cu_seqlens=cu.numpy(), mode="seq_mean_token_mean")
    assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7
    with pytest.raises(flp.FusedLogpError, match="mode"):
        flp._lib.check("logp_grpo_loss", flp._lib.load().logp_grpo_loss(
            None, None, None, None, None, None, 0, 0, 7, 0.2, 0.2, 0.0, 0.0, None, 0, None, None, None, None))


def test_rl_step_chain_against_fp64():
    """logits -> logp (fused forward) -> GRPO loss and d loss / d logp ->
    dlogits (fused backward), against the FP64 oracle chain on the same inputs."""
    n, v = 512, workloads.QWEN3_VOCAB
    x, y, _ = workloads.make("mid", device=DEV, n=n)
    lpo, old, ref, adv, mask, cu = _case(n, 6, nseq=8)
    logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True)
    old_d = (logp.cpu() + (old - lpo)).to(DEV)        # old/ref defined relative to the
    ref_d = (logp.cpu() + (ref - lpo)).to(DEV)        # current logp so ratios stay moderate
    act = (y.cpu() >= 0).to(torch.uint8) * mask
    loss, g = flp.logp_grpo_loss(logp, old_d, adv.to(DEV), ref_logp=ref_d, active_mask=act.to(DEV),
                                 cu_seqlens=cu.to(DEV), mode="seq_mean_token_mean", beta=0.04)
    d = flp.fused_logp_backward(x, y, lse, g, lse_lo=lo)

    xb, yn = workloads.bf16_bits(x), y.cpu().numpy()
    lp64, _ = oracle.forward(xb, yn)
    old64 = lp64 + (old - lpo).double().numpy()
    ref64 = lp64 + (ref - lpo).double().numpy()
    l64, g64 = oracle.grpo_loss(lp64, old64, adv.double().numpy(), ref_logp=ref64, mask=act.numpy(),
                                cu_seqlens=cu.numpy(), mode="seq_mean_token_mean", beta=0.04)
    assert abs(loss.item() - l64) <= 1e-4 * abs(l64) + 1e-6
    st = oracle.backward_compare(xb, yn, g64.astype(np.float32), workloads.bf16_bits(d))
    # the GPU's upstream gradient differs from the FP64 one by ~1e-6 relative,
    # so the bound is the plain max-error bound (not the correctly rounded count)
    assert st["max_abs_diff"] <= max(2e-3 * st["max_abs_d"], 2 * st["max_rounding_gap"]), st


@pytest.mark.parametrize("mode", MODES)
def test_grpo_many_segments_against_oracle(mode):
    """A million tokens in 3000 packed sequences (many CTAs in the mask count,
    the sequence counts and the token pass) and the whole-batch form (1024
    chunks), against FP64."""
    n = 1 << 20
    lp, old, ref, adv, mask, cu = _case(n, 11, nseq=3000)
    for cuv in (cu, None):
        if cuv is None and mode != "token_mean":
            continue
        kw = dict(mode=mode, eps_lo=0.2, eps_hi=0.28, beta=0.02)
        loss, grad = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0],
                                        cu_seqlens=None if cuv is None else _dev(cuv)[0], **kw)
        want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                                          ref_logp=ref.double().numpy(), mask=mask.numpy(),
                                          cu_seqlens=None if cuv is None else cuv.numpy(), **kw)
        got_g = grad.double().cpu().numpy()
        assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7, (loss.item(), want_l)
        w = _token_weights(n, mask.numpy(), None if cuv is None else cuv.numpy(), mode)
        _assert_grad(got_g, want_g, lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                     ref.double().numpy(), kw["beta"], kw["eps_lo"], kw["eps_hi"], w)
        again = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0],
                                   cu_seqlens=None if cuv is None else _dev(cuv)[0], **kw)
        assert torch.equal(again[0].view(torch.int32), loss.view(torch.int32))
        assert torch.equal(again[1].view(torch.int32), grad.view(torch.int32))


def _layout(n, seed):
    """cu_seqlens that leave 37 tokens uncovered in front and 123 behind, with
    900 sequences of 0..3 tokens (so one 256-token chunk meets well over 31
    sequences), one sequence of 20000 tokens (about 80 chunks) and random
    lengths up to 700 after it."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, 4, (900,), generator=g).tolist() + [20000]
    pos = 37 + sum(lens)
    while True:
        ln = int(torch.randint(1, 700, (1,), generator=g))
        if pos + ln > n - 123:
            break
        lens.append(ln)
        pos += ln
    return torch.cumsum(torch.tensor([37] + lens, dtype=torch.int64), 0)


@pytest.mark.parametrize("mode", MODES)
def test_grpo_uncovered_tiny_and_long_sequences(mode):
    n = 60000
    lp, old, ref, adv, mask, _ = _case(n, 21)
    cu = _layout(n, 22)
    cover = torch.zeros(n, dtype=torch.bool)
    cover[int(cu[0]):int(cu[-1])] = True
    for norm in (0.0, 777.0):
        kw = dict(mode=mode, eps_lo=0.2, eps_hi=0.28, beta=0.03, normalizer=norm)
        loss, grad, tl = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0],
                                            cu_seqlens=_dev(cu)[0], token_loss=True, **kw)
        want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                                          ref_logp=ref.double().numpy(), mask=mask.numpy(), cu_seqlens=cu.numpy(),
                                          **kw)
        got_g = grad.double().cpu().numpy()
        assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7, (norm, loss.item(), want_l)
        assert np.max(np.abs(got_g - want_g)) <= 1e-5 * np.max(np.abs(want_g)), norm
        out = ~cover.numpy()
        assert np.all(got_g[out] == 0) and torch.all(tl.cpu()[~cover] == 0)


def test_grpo_one_long_sequence_mean_of_means():
    """One sequence of 300000 tokens given by cu_seqlens (its 1172 chunks on
    many warps, its count from the word prefixes at its two bounds) equals
    the whole-batch form."""
    n = 300000
    lp, old, ref, adv, mask, _ = _case(n, 23)
    cu = torch.tensor([0, n], dtype=torch.int64)
    kw = dict(mode="seq_mean_token_mean", beta=0.01)
    a = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0],
                           cu_seqlens=_dev(cu)[0], **kw)
    b = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0], **kw)
    want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                                      ref_logp=ref.double().numpy(), mask=mask.numpy(), **kw)
    for loss, grad in (a, b):
        assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7
        assert np.max(np.abs(grad.double().cpu().numpy() - want_g)) <= 1e-5 * np.max(np.abs(want_g))


def test_grpo_caller_weight_equals_counted_weight():
    """A normaliser equal to the active-token count (or the number of
    non-empty sequences) makes the weight the caller's, and nothing is
    counted: loss and gradient are bitwise those of the form that counts the
    mask on the device."""
    n = 100000
    lp, old, ref, adv, mask, cu = _case(n, 24, nseq=333)
    d = float(int(mask.sum()))
    for mode, den in (("token_mean", d), ("seq_mean_token_sum", None)):
        cnt = d
        if den is None:   # the number of sequences with an active token
            cnt = float(sum(int(mask[int(cu[s]):int(cu[s + 1])].sum()) > 0 for s in range(333)))
        kw = dict(ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0], cu_seqlens=_dev(cu)[0], mode=mode, beta=0.02)
        a = flp.logp_grpo_loss(*_dev(lp, old, adv), **kw)
        b = flp.logp_grpo_loss(*_dev(lp, old, adv), normalizer=cnt, **kw)
        assert torch.equal(a[0].view(torch.int32), b[0].view(torch.int32)), mode
        assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32)), mode


def test_grpo_unaligned_arrays_bitwise_equal():
    """Arrays that start 4 bytes past a 16-byte boundary take the scalar-access
    variant of the token passes; it computes the same tokens in the same
    order, so loss, gradient and token loss are bitwise those of aligned
    copies."""
    n = 70001
    lp, old, ref, adv, mask, cu = _case(n, 25, nseq=97)
    big = [torch.empty(n + 1, dtype=t.dtype, device=DEV) for t in (lp, old, ref, adv, mask)]
    views = []
    for b, t in zip(big, (lp, old, ref, adv, mask)):
        b[1:].copy_(t)
        views.append(b[1:])
    for mode in MODES:
        kw = dict(cu_seqlens=_dev(cu)[0], mode=mode, beta=0.05, token_loss=True)
        a = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0], **kw)
        b = flp.logp_grpo_loss(views[0], views[1], views[3], ref_logp=views[2], active_mask=views[4], **kw)
        assert views[0].data_ptr() % 16 == 4
        for u, v in zip(a, b):
            assert torch.equal(u.view(torch.int32), v.view(torch.int32)), mode


def test_grpo_bench_size_against_oracle():
    """The bench's workload and launch shape: 16,777,216 tokens in 16,384
    sequences, sequence mean of token means with KL; every loss and gradient
    value against the FP64 oracle, and a second call bitwise equal."""
    n, nseq = 1 << 24, 16384
    lp, old, ref, adv, mask, cu = _case(n, 41, nseq=nseq)
    kw = dict(mode="seq_mean_token_mean", eps_lo=0.2, eps_hi=0.28, beta=0.04)
    args = _dev(lp, old, adv)
    dk = dict(ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0], cu_seqlens=_dev(cu)[0], **kw)
    loss, grad = flp.logp_grpo_loss(*args, **dk)
    want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                                      ref_logp=ref.double().numpy(), mask=mask.numpy(), cu_seqlens=cu.numpy(), **kw)
    got_g = grad.double().cpu().numpy()
    assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7, (loss.item(), want_l)
    w = _token_weights(n, mask.numpy(), cu.numpy(), kw["mode"])
    _assert_grad(got_g, want_g, lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                 ref.double().numpy(), kw["beta"], kw["eps_lo"], kw["eps_hi"], w)
    again = flp.logp_grpo_loss(*args, **dk)
    assert torch.equal(again[0].view(torch.int32), loss.view(torch.int32))
    assert torch.equal(again[1].view(torch.int32), grad.view(torch.int32))


@pytest.mark.parametrize("mode", MODES)
def test_grpo_300k_short_sequences(mode):
    """2,097,152 tokens in 300,000 sequences (about 7 tokens each): the folds
    run at their largest shape (1024 CTAs, sequence shares of 293 that loop,
    the last CTA folding 4 partials per thread), and a 256-token chunk meets
    about 37 sequences (boundary windows reloaded in both token passes)."""
    n, nseq = 1 << 21, 300000
    lp, old, ref, adv, mask, cu = _case(n, 51, nseq=nseq)
    kw = dict(mode=mode, eps_lo=0.2, eps_hi=0.28, beta=0.03)
    loss, grad = flp.logp_grpo_loss(*_dev(lp, old, adv), ref_logp=_dev(ref)[0], active_mask=_dev(mask)[0],
                                    cu_seqlens=_dev(cu)[0], **kw)
    want_l, want_g = oracle.grpo_loss(lp.double().numpy(), old.double().numpy(), adv.double().numpy(),
                                      ref_logp=ref.double().numpy(), mask=mask.numpy(), cu_seqlens=cu.numpy(), **kw)
    assert abs(loss.item() - want_l) <= 1e-5 * abs(want_l) + 1e-7, (loss.item(), want_l)
    w = _token_weights(n, mask.numpy(), cu.numpy(), mode)
    _assert_grad(grad.double().cpu().numpy(), want_g, lp.double().numpy(), old.double().numpy(),
                 adv.double().numpy(), ref.double().numpy(), kw["beta"], kw["eps_lo"], kw["eps_hi"], w)
