"""Vocabulary-parallel and row-parallel forms on the GPU.

In one process: the shard backward (PR #314's vocab-parallel logprob op has a
backward over the local shard: each shard writes -s g p on its columns plus
the one-hot term only where it holds the target, from the merged LSE) side by
side equals the unsharded backward bit for bit, including ignore rows, masked
rows and rows whose target lies in another shard; the merge over gathered
exchange blocks (issue #241 PR 3 / PR 6, PR #314 Tensor Parallel section)
equals the unsharded forward bit for bit.

Across processes: 2 and 4 ranks as processes on this one GPU, joined by a
gloo group (the exchange goes through host copies; no kernel of one rank
waits on another): the vocabulary-parallel forward gives every rank the
unsharded logp, LSE and LSE residual bit for bit, and each rank's backward
columns are the unsharded gradient's; the row-parallel form over one global
batch split unevenly gives the single call's bits."""

import numpy as np
import pytest
import torch

import oracle
import selected_token_logprob_gb300 as flp
import workloads
from dist_util import run_ranks
from parity_util import bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
V = workloads.QWEN3_VOCAB


@pytest.fixture(scope="module", autouse=True)
def _built():
    flp._lib.load(build_if_missing=True)


def _i(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _bounds(v, S, W):
    """S contiguous shards on the tile grid: tile counts as even as possible."""
    n_tiles = -(-v // W)
    cuts = [round(l * n_tiles / S) * W for l in range(S)] + [v]
    return [(cuts[l], min(v, cuts[l + 1]) - cuts[l]) for l in range(S)]


def _padded_shard(x, a, w, pad_to=128):
    n = x.shape[0]
    buf = torch.full((n, -(-w // pad_to) * pad_to), float("-inf"), dtype=x.dtype, device=x.device)
    buf[:, :w] = x[:, a:a + w]
    return buf


def _inputs(n, v, dtype=torch.bfloat16, seed=5):
    wl = workloads.Workload("vp", n, v, 2.0, 8.0, 0.05, "normal", seed=seed)
    return workloads.make(wl, device=DEV, dtype=dtype)


@pytest.mark.parametrize("S", [2, 4])
@pytest.mark.parametrize("dtype, temp, masked", [(torch.bfloat16, 1.0, False), (torch.bfloat16, 0.7, True),
                                                 (torch.float16, 1.0, False), (torch.float32, 0.8, True)])
def test_shard_backward_concatenated_is_unsharded_bitwise(S, dtype, temp, masked):
    n = 256
    x, y, g = _inputs(n, V, dtype)
    y[:3] = torch.tensor([V - 1, 0, V // 2 + 1])       # targets at the vocabulary's edges and mid-shard
    mask = (torch.arange(n, device=DEV) % 7 != 3).to(torch.uint8) if masked else None
    logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True, temperature=temp, active_mask=mask)
    want = flp.fused_logp_backward(x, y, lse, g, lse_lo=lo, temperature=temp, active_mask=mask)
    W = flp.flp_tile_width(V)
    for a, w in _bounds(V, S, W):
        buf = _padded_shard(x, a, w)
        d = flp.logp_shard_backward(buf, a, w, V, y, lse, g, lse_lo=lo, temperature=temp, active_mask=mask)
        assert torch.equal(_i(d), _i(want[:, a:a + w].contiguous())), (a, w)
    # bounds off the tile grid are fine for the elementwise backward
    a, w = 12345, 777
    d = flp.logp_shard_backward(x[:, a:a + w], a, w, V, y, lse, g, lse_lo=lo, temperature=temp, active_mask=mask)
    assert torch.equal(_i(d), _i(want[:, a:a + w].contiguous()))


def test_shard_backward_in_place_and_against_oracle():
    n, v = 96, 5000
    x, y, g = _inputs(n, v, seed=9)
    y[5] = 4999
    y[6] = -100
    logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True)
    a, w = 2048, 2952                                   # the last shard, in place over its own columns
    buf = x[:, a:].contiguous()
    flp.logp_shard_backward(buf, a, w, v, y, lse, g, lse_lo=lo, dshard=buf)
    torch.cuda.synchronize()
    ref = oracle.backward(bits(x), y.cpu().numpy(), g.cpu().numpy())[:, a:]      # FP64 [n, w]
    got = oracle.bf16_to_f64(bits(buf))
    cr = oracle.bf16_to_f64(oracle.round_bf16(ref))
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref)) <= max(2e-3 * np.max(np.abs(ref)), np.max(np.abs(cr - ref)))
    assert np.count_nonzero(got != cr) <= 1e-4 * got.size
    assert np.all(got[6] == 0) and np.any(got[5] != 0)
    with pytest.raises(flp.FusedLogpError, match="inside the vocabulary"):
        flp.logp_shard_backward(buf, 4000, w, v, y, lse, g)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 16])
def test_gathered_merge_equals_unsharded_bitwise(S):
    n = 512
    x, y, _ = _inputs(n, V, seed=11)
    temp = 0.7 if S == 3 else 1.0
    logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True, temperature=temp)
    W = flp.flp_tile_width(V)
    bounds = _bounds(V, S, W)
    blocks = torch.full((S, 33 * n + 7), float("nan"), device=DEV)   # a stride wider than one block
    for r, (a, w) in enumerate(bounds):
        pm, ps, sel = flp.partials_views(blocks[r], n)
        flp.logp_shard_partials(_padded_shard(x, a, w), a, w, V, y, pm, ps, sel, temperature=temp)
    # ranks listed in any order: the table says which rank holds which tile
    perm = list(range(S))[::-1]
    g_logp, g_lse, g_lo = flp.logp_merge_gathered_partials(
        blocks[perm], [bounds[r][0] for r in perm], [bounds[r][1] for r in perm], y, V, with_lse_lo=True,
        temperature=temp)
    for got, want in ((g_logp, logp), (g_lse, lse), (g_lo, lo)):
        assert torch.equal(_i(got), _i(want))


def test_gathered_merge_rejects_bad_layouts():
    n = 4
    y = torch.zeros(n, dtype=torch.int64, device=DEV)
    blocks = torch.zeros((2, 33 * n), device=DEV)
    W = flp.flp_tile_width(V)
    with pytest.raises(flp.FusedLogpError, match="held by no rank"):
        flp.logp_merge_gathered_partials(blocks, [0, 9 * W], [8 * W, V - 9 * W], y, V)
    with pytest.raises(flp.FusedLogpError, match="FLP_EUNSUPPORTED"):
        flp.logp_merge_gathered_partials(blocks, [0, 8 * W + 8], [8 * W + 8, V - 8 * W - 8], y, V)


# ---------------------------------------------------------------- several processes on this GPU

def _vocab_rank(rank, world, n, S_per_rank, temp):
    """Rank r holds shards [r S_per_rank, (r + 1) S_per_rank) of an S-way split
    as one contiguous slice; returns whether its results equal the unsharded
    call's bit for bit."""
    import torch

    import selected_token_logprob_gb300 as flp
    from selected_token_logprob_gb300 import distributed as fd

    torch.cuda.set_device(0)
    x, y, g = _inputs(n, V, seed=21)                    # every rank draws the same global batch
    y[0] = V - 1
    mask = (torch.arange(n, device=DEV) % 11 != 5).to(torch.uint8)
    logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True, temperature=temp, active_mask=mask)
    want_d = flp.fused_logp_backward(x, y, lse, g, lse_lo=lo, temperature=temp, active_mask=mask)
    W = flp.flp_tile_width(V)
    bounds = _bounds(V, world * S_per_rank, W)
    a = bounds[rank * S_per_rank][0]
    last = bounds[(rank + 1) * S_per_rank - 1]
    w = last[0] + last[1] - a
    shard = _padded_shard(x, a, w)
    shard.requires_grad_(True)
    got = fd.vocab_parallel_logp(shard, y, a, V, real_width=w, ignore_index=-100, temperature=temp,
                                 active_mask=mask)
    r_logp, r_lse, r_lo = fd.vocab_parallel_logp_forward(shard.detach(), y, a, V, real_width=w, temperature=temp,
                                                         active_mask=mask, with_lse_lo=True)
    (got * g).sum().backward()
    torch.cuda.synchronize()
    d = shard.grad[:, :w]
    return {"logp": torch.equal(_i(got.detach()), _i(logp)), "logp2": torch.equal(_i(r_logp), _i(logp)),
            "lse": torch.equal(_i(r_lse), _i(lse)), "lse_lo": torch.equal(_i(r_lo), _i(lo)),
            "dlogits": torch.equal(_i(d.contiguous()), _i(want_d[:, a:a + w].contiguous())),
            "pad_grad_zero": bool((shard.grad[:, w:] == 0).all().item()) if shard.shape[1] > w else True,
            "device_error": flp.flp_device_error(0)}


@pytest.mark.parametrize("world, S_per_rank, temp", [(2, 1, 1.0), (2, 2, 0.7), (4, 1, 1.0)])
def test_vocab_parallel_ranks_match_unsharded_bitwise(world, S_per_rank, temp):
    res = run_ranks(_vocab_rank, world, (1024, S_per_rank, temp), timeout=600)
    for rank in range(world):
        kind, val = res[rank]
        assert kind == "ok", (rank, val)
        assert all(v is True for k, v in val.items() if k != "device_error"), (rank, val)
        assert val["device_error"] == 0


def _row_rank(rank, world, counts):
    import torch

    import selected_token_logprob_gb300 as flp
    from selected_token_logprob_gb300 import distributed as fd

    torch.cuda.set_device(0)
    n = sum(counts)
    x, y, g = _inputs(n, V, seed=31)                    # the global batch; this rank keeps its rows
    logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True)
    want_d = flp.fused_logp_backward(x, y, lse, g, lse_lo=lo)
    a = sum(counts[:rank])
    b = a + counts[rank]
    xl = x[a:b].clone()
    (l_logp, l_lse, l_lo), (all_logp, all_lse) = fd.row_parallel_logp_forward(xl, y[a:b].clone())
    d = fd.row_parallel_logp_backward(xl, y[a:b].clone(), l_lse, g[a:b].clone(), lse_lo=l_lo)
    torch.cuda.synchronize()
    return {"logp": torch.equal(_i(all_logp), _i(logp)), "lse": torch.equal(_i(all_lse), _i(lse)),
            "dlogits": torch.equal(_i(d), _i(want_d[a:b]))}


def test_row_parallel_global_batch_matches_one_call_bitwise():
    res = run_ranks(_row_rank, 2, ([600, 424],), timeout=600)
    for rank in range(2):
        kind, val = res[rank]
        assert kind == "ok", (rank, val)
        assert all(val.values()), (rank, val)


def _vocab_rank_device_transport(rank, world, n):
    """As _vocab_rank, with the exchange on device tensors the way it runs on
    NCCL (one all_gather_into_tensor into a rank-major [world, L] buffer).  Two
    NCCL ranks cannot share one GPU, so gloo stands in for the transport with
    NCCL's documented semantics (the output is the inputs concatenated in rank
    order); the library code path is the one a NCCL group takes."""
    import torch
    import torch.distributed as dist

    import selected_token_logprob_gb300 as flp
    from selected_token_logprob_gb300 import distributed as fd

    torch.cuda.set_device(0)
    calls = []

    def all_gather_into_tensor(out, inp, group=None):
        assert out.is_cuda and inp.is_cuda and out.numel() == world * inp.numel()
        parts = [torch.empty_like(inp, device="cpu") for _ in range(world)]
        dist.all_gather(parts, inp.cpu(), group=group)
        out.copy_(torch.cat(parts).to(out.device))
        calls.append(inp.numel())

    real_backend = fd.dist.get_backend
    fd.dist.get_backend = lambda group=None: "nccl"
    fd.dist.all_gather_into_tensor = all_gather_into_tensor
    try:
        x, y, g = _inputs(n, V, seed=23)
        logp, lse, lo = flp.fused_logp_forward(x, y, with_lse_lo=True)
        W = flp.flp_tile_width(V)
        a, w = _bounds(V, world, W)[rank]
        shard = _padded_shard(x, a, w)
        r_logp, r_lse, r_lo = fd.vocab_parallel_logp_forward(shard, y, a, V, real_width=w, with_lse_lo=True)
        torch.cuda.synchronize()
        return {"logp": torch.equal(_i(r_logp), _i(logp)), "lse": torch.equal(_i(r_lse), _i(lse)),
                "lse_lo": torch.equal(_i(r_lo), _i(lo)), "device_transport_used": calls == [33 * n]}
    finally:
        fd.dist.get_backend = real_backend


def test_vocab_parallel_device_tensor_transport_path():
    res = run_ranks(_vocab_rank_device_transport, 2, (512,), timeout=600)
    for rank in range(2):
        kind, val = res[rank]
        assert kind == "ok", (rank, val)
        assert all(val.values()), (rank, val)


# ---------------------------------------------------------------- the fused LM head, vocabulary parallel

@pytest.mark.parametrize("bounds", [(0, 10240, 20000), (0, 5120, 12800, 20000), (0, 256, 512, 19968, 20000)])
def test_linear_gathered_merge_equals_unsharded_bitwise(bounds):
    """Each slice of the LM-head weight writes its tiles' partials into its
    own workspace; the merge over the stacked workspaces (ranks listed in any
    order) gives the one-GPU forward's logp, lse and lse_lo bit for bit, with
    temperature and a mask."""
    n, d, v = 300, 512, 20000
    h, w, y = workloads.linear(n, d, v, seed=91, device=DEV)
    mask = (torch.arange(n, device=DEV) % 7 != 3)
    ref = flp.fused_linear_logp_forward(h, w, y, with_lse_lo=True, temperature=0.7, active_mask=mask)
    nbytes = flp.fused_linear_logp_workspace_size(n, v)
    slices = list(zip(bounds[:-1], bounds[1:]))
    blocks = torch.full((len(slices), nbytes // 4 + 5), float("nan"), device=DEV)   # a stride wider than a block
    for r, (a, b) in enumerate(slices):
        ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)            # other ranks' tiles: garbage
        flp.fused_linear_logp_shard_partials(h, w[a:b].clone(), a, v, y, ws, temperature=0.7)
        blocks[r, :nbytes // 4] = ws.view(torch.float32)
    perm = list(range(len(slices)))[::-1]
    out = flp.fused_linear_logp_merge_gathered(blocks[perm], [slices[r][0] for r in perm],
                                               [slices[r][1] - slices[r][0] for r in perm], y, v,
                                               with_lse_lo=True, temperature=0.7, active_mask=mask)
    for r, o in zip(ref, out):
        assert torch.equal(_i(r), _i(o))


def test_sum_blocks_is_the_rank_order_sum():
    g = torch.Generator(device=DEV).manual_seed(3)
    blocks = torch.randn((4, 333, 257), generator=g, device=DEV) * torch.tensor([1.0, 1e4, 1e-4, 1.0],
                                                                               device=DEV).view(4, 1, 1)
    want = ((blocks[0] + blocks[1]) + blocks[2]) + blocks[3]          # the same IEEE additions, in order
    assert torch.equal(_i(flp.sum_blocks(blocks)), _i(want))
    assert torch.equal(_i(flp.sum_blocks(blocks[:1])), _i(blocks[0]))


def _linear_rank(rank, world, n, d, v, cut):
    import torch

    import selected_token_logprob_gb300 as flp
    from selected_token_logprob_gb300 import distributed as fd

    torch.cuda.set_device(0)
    h, w, y = workloads.linear(n, d, v, seed=97, device=DEV)        # every rank: the same hidden states
    mask = (torch.arange(n, device=DEV) % 5 != 2)
    g = torch.randn(n, generator=torch.Generator().manual_seed(98)).to(DEV)
    bounds = [(0, cut), (cut, v)]
    # the one-GPU references: the unsharded forward, the sharded backward in slice order
    ref = flp.fused_linear_logp_forward(h, w, y, with_lse_lo=True, temperature=0.7, active_mask=mask)
    dh_ref = torch.empty((n, d), device=DEV)
    dw_ref = [flp.fused_linear_logp_shard_backward(h, w[a:b].clone(), a, v, y, ref[1], g, dh_ref, k > 0,
                                                   lse_lo=ref[2], temperature=0.7, active_mask=mask)
              for k, (a, b) in enumerate(bounds)]
    dh_all, _ = flp.fused_linear_logp_backward(h, w, y, ref[1], g, lse_lo=ref[2], temperature=0.7,
                                               active_mask=mask)
    a, b = bounds[rank]
    hh = h.clone().requires_grad_(True)
    ws = w[a:b].clone().requires_grad_(True)
    logp = fd.vocab_parallel_linear_logp(hh, ws, y, a, v, temperature=0.7, active_mask=mask)
    (logp * g).sum().backward()
    torch.cuda.synchronize()
    rel = (torch.max(torch.abs(hh.grad.float() - dh_all)) / torch.max(torch.abs(dh_all))).item()
    return {"logp": torch.equal(_i(logp.detach()), _i(ref[0])),
            # autograd returns dhidden in hidden's dtype (BF16): compare with the reference cast the same way
            "dhidden_sharded_bits": torch.equal(hh.grad.view(torch.int16), dh_ref.to(torch.bfloat16).view(torch.int16)),
            "dweight_rows_bits": torch.equal(ws.grad.view(torch.int16), dw_ref[rank].to(torch.bfloat16).view(torch.int16)),
            "dhidden_close_to_unsharded": rel <= 1e-2,
            "device_error": flp.flp_device_error(0)}


def test_vocab_parallel_lm_head_two_ranks_match_one_gpu():
    res = run_ranks(_linear_rank, 2, (300, 512, 20000, 10240), timeout=600)
    for rank in range(2):
        kind, val = res[rank]
        assert kind == "ok", (rank, val)
        assert all(v is True for k, v in val.items() if k != "device_error"), (rank, val)
        assert val["device_error"] == 0
