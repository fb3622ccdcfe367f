"""The entry points only enqueue work on the caller's stream (no allocation,
no synchronisation inside a call), so a training step built from them can be
captured once as a CUDA graph and replayed: the replays give the eager
results bit for bit."""

import pytest
import torch

import selected_token_logprob_gb300 as flp
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    flp._lib.load(build_if_missing=True)


def _i(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def test_logits_step_replays_bitwise():
    x, y, g = workloads.make("mid", device=DEV, n=256)
    n, v = x.shape
    logp, lse, lo = (torch.empty(n, device=DEV) for _ in range(3))
    dl = torch.empty_like(x)

    def step():
        flp.fused_logp_forward(x, y, logp=logp, lse=lse, lse_lo=lo)
        flp.fused_logp_backward(x, y, lse, g, dlogits=dl, lse_lo=lo)

    step()                                   # one-time set-up happens outside the capture
    torch.cuda.synchronize()
    want = [t.clone() for t in (logp, lse, lo, dl)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for t in (logp, lse, lo, dl):
        t.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for got, ref in zip((logp, lse, lo, dl), want):
        assert torch.equal(_i(got), _i(ref))
    assert flp.flp_device_error(0) == 0


def test_linear_forward_replays_bitwise():
    n, d, v = 300, 512, 8000
    h, w, y = workloads.linear(n, d, v, seed=101, device=DEV)
    ws = torch.empty(flp.fused_linear_logp_workspace_size(n, v), dtype=torch.uint8, device=DEV)
    logp, lse = torch.empty(n, device=DEV), torch.empty(n, device=DEV)

    def step():
        flp.fused_linear_logp_forward(h, w, y, logp=logp, lse=lse, workspace=ws)

    step()
    torch.cuda.synchronize()
    want = [logp.clone(), lse.clone()]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    logp.zero_()
    lse.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_i(logp), _i(want[0])) and torch.equal(_i(lse), _i(want[1]))


def test_grpo_loss_replays_bitwise():
    """The GRPO loss (its count fix and token pass are launched as
    programmatic dependents of their predecessors) captured in a graph
    replays bitwise."""
    g = torch.Generator().manual_seed(31)
    n, nseq = 50000, 77
    lp = -torch.rand(n, generator=g) * 5
    old = lp + (torch.rand(n, generator=g) - 0.5)
    adv = torch.randn(n, generator=g)
    mask = (torch.rand(n, generator=g) > 0.2).to(torch.uint8)
    cu = torch.cat([torch.zeros(1, dtype=torch.int64),
                    torch.sort(torch.randint(0, n + 1, (nseq - 1,), generator=g)).values,
                    torch.full((1,), n, dtype=torch.int64)])
    lp, old, adv, mask, cu = (t.to(DEV) for t in (lp, old, adv, mask, cu))
    ws = torch.empty(flp.logp_grpo_loss_workspace_size(n, nseq), dtype=torch.uint8, device=DEV)
    for mode in ("token_mean", "seq_mean_token_mean"):
        kw = dict(ref_logp=old, active_mask=mask, cu_seqlens=cu, mode=mode, beta=0.02, workspace=ws)
        want = flp.logp_grpo_loss(lp, old, adv, **kw)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                got = flp.logp_grpo_loss(lp, old, adv, **kw)
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        for u, v in zip(got, want):
            assert torch.equal(u.view(torch.int32), v.view(torch.int32)), mode


def test_grpo_counts_and_counted_loss_replay_bitwise():
    """The two-part GRPO form (the layout's counts, then the token pass on
    them) captured in one graph replays bit for bit, and equals the one-call
    loss."""
    g = torch.Generator().manual_seed(32)
    n, nseq = 40000, 50
    lp = -torch.rand(n, generator=g) * 5
    old = lp + (torch.rand(n, generator=g) - 0.5)
    adv = torch.randn(n, generator=g)
    mask = (torch.rand(n, generator=g) > 0.3).to(torch.uint8)
    cu = torch.cat([torch.zeros(1, dtype=torch.int64),
                    torch.sort(torch.randint(0, n + 1, (nseq - 1,), generator=g)).values,
                    torch.full((1,), n, dtype=torch.int64)])
    lp, old, adv, mask, cu = (t.to(DEV) for t in (lp, old, adv, mask, cu))
    kw = dict(active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean", beta=0.0)
    want = flp.logp_grpo_loss(lp, old, adv, **kw)
    ws = torch.empty(flp.logp_grpo_loss_workspace_size(n, nseq), dtype=torch.uint8, device=DEV)
    flp.logp_grpo_loss_counts(n, active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean", workspace=ws)
    flp.logp_grpo_loss(lp, old, adv, workspace=ws, counted=True, **kw)       # eager first call
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            flp.logp_grpo_loss_counts(n, active_mask=mask, cu_seqlens=cu, mode="seq_mean_token_mean",
                                      workspace=ws, stream=s)
            got = flp.logp_grpo_loss(lp, old, adv, workspace=ws, counted=True, **kw)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        for u, v in zip(got, want):
            assert torch.equal(u.view(torch.int32), v.view(torch.int32))
