"""Bitwise determinism on the GPU: repeated runs, the batch-size sweep of
RL-Kernel PR #495 (Prior art: eight rows alone vs at the front, middle and back
of batches of every size 1-9 and 2^k-1, 2^k, 2^k+1 up to 2048, three seeds,
logp and dlogits), and the vocab-sharded partials/merge against the unsharded
forward (issue #241 PR 3 acceptance: the sharded result bitwise equals the
unsharded one), plus the shard partials against the oracle's range partials."""

import numpy as np
import pytest
import torch

import oracle
import selected_token_logprob_gb300 as flp
import workloads
from parity_util import bits, run

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
V = workloads.QWEN3_VOCAB


@pytest.fixture(scope="module", autouse=True)
def _built():
    flp._lib.load(build_if_missing=True)


def _i(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def test_repeat_runs_are_bitwise_identical():
    x, y, g = workloads.make("mid", device=DEV)
    ref = [r.clone() for r in run(x, y, g)]
    for _ in range(3):
        out = run(x, y, g)
        for a, b in zip(ref, out):
            assert torch.equal(_i(a), _i(b))


def sweep_sizes():
    sizes = list(range(2, 10))
    for k in range(4, 11):
        sizes += [2 ** k - 1, 2 ** k, 2 ** k + 1]
    sizes += [2047, 2048]
    return sizes


def test_batch_invariance_sweep_2232():
    sizes = sweep_sizes()
    assert len(sizes) == 31
    wl = workloads.WORKLOADS["sweep"]
    cap = max(sizes)
    F = None
    compared = differing = 0
    for seed in (0, 1, 2):
        px, py, pg = workloads.sweep_rows(8, V, wl.sigma, seed, 0, device=DEV)
        del F
        F, fy, fg = workloads.sweep_rows(cap, V, wl.sigma, seed, 1, device=DEV)
        dl_buf = torch.empty((cap, V), dtype=torch.bfloat16, device=DEV)
        refs = []
        for k in range(8):
            lp, ls, d = run(px[k:k + 1], py[k:k + 1], pg[k:k + 1])
            refs.append((lp.clone(), ls.clone(), d.clone()))
        for B in sizes:
            for pos in (0, B // 2, B - 1):
                save_x, save_y, save_g = F[pos].clone(), fy[pos].clone(), fg[pos].clone()
                for k in range(8):
                    F[pos].copy_(px[k]); fy[pos] = py[k]; fg[pos] = pg[k]
                    lp, ls, lo = flp.fused_logp_forward(F[:B], fy[:B], with_lse_lo=True)
                    flp.fused_logp_backward(F[:B], fy[:B], ls, fg[:B], dlogits=dl_buf[:B],
                                            lse_lo=lo)
                    r_lp, r_ls, r_d = refs[k]
                    same = (torch.equal(_i(lp[pos:pos + 1]), _i(r_lp))
                            and torch.equal(_i(ls[pos:pos + 1]), _i(r_ls))
                            and torch.equal(_i(dl_buf[pos:pos + 1]), _i(r_d)))
                    compared += 1
                    differing += 0 if same else 1
                F[pos].copy_(save_x); fy[pos] = save_y; fg[pos] = save_g
    print(f"batch sweep: {differing} of {compared} comparisons differ")
    assert compared == 2232
    assert differing == 0


def _shards(x, S, pad_to=128):
    """S contiguous equal shards of the vocabulary, each in its own buffer
    padded with -inf columns to a multiple of pad_to."""
    n, v = x.shape
    out = []
    for l in range(S):
        a, b = l * v // S, (l + 1) * v // S
        w = b - a
        wpad = -(-w // pad_to) * pad_to
        buf = torch.full((n, wpad), float("-inf"), dtype=torch.bfloat16, device=x.device)
        buf[:, :w] = x[:, a:b]
        out.append((buf, a, w))
    return out


def _sharded_forward(shards, y, v_total, order=None):
    n = y.shape[0]
    pm = torch.full((n, 16), float("nan"), device=DEV)
    ps = torch.full((n, 16), float("nan"), device=DEV)
    sel = torch.full((n,), float("nan"), device=DEV)
    for l in (order or range(len(shards))):
        buf, a, w = shards[l]
        flp.logp_shard_partials(buf, a, w, v_total, y, pm, ps, sel)
    logp, lse, lse_lo = flp.logp_merge_partials(pm, ps, sel, y, v_total, with_lse_lo=True)
    _sharded_forward.lse_lo = lse_lo
    return logp, lse, pm, ps


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
def test_sharded_equals_unsharded_bitwise(S):
    x, y, _ = workloads.make("sharded", device=DEV)
    logp, lse, lse_lo = flp.fused_logp_forward(x, y, with_lse_lo=True)
    s_logp, s_lse, pm, ps = _sharded_forward(_shards(x, S), y, V)
    assert torch.equal(_i(s_lse), _i(lse))
    assert torch.equal(_i(s_logp), _i(logp))
    assert torch.equal(_i(_sharded_forward.lse_lo), _i(lse_lo))
    # the shard launch order does not matter either
    if S > 1:
        r_logp, r_lse, _, _ = _sharded_forward(_shards(x, S), y, V, order=list(range(S))[::-1])
        assert torch.equal(_i(r_lse), _i(lse)) and torch.equal(_i(r_logp), _i(logp))


def test_shard_partials_against_oracle():
    """Tile maxima are exact; tile sums are within FP32 accumulation error of
    the FP64 range sums (tolerance on the rank-local kernel, issue #241 PR 6)."""
    x, y, _ = workloads.make("sharded", device=DEV, n=256)
    W = flp.flp_tile_width(V)
    _, _, pm, ps = _sharded_forward(_shards(x, 4), y, V)
    ref_m, ref_s = oracle.range_partials(bits(x), W, 16)
    got_m = pm.cpu().numpy().astype(np.float64)
    got_s = ps.cpu().numpy().astype(np.float64)
    assert np.array_equal(got_m, ref_m)
    rel = np.max(np.abs(got_s - ref_s) / ref_s)
    print("tile sumexp max rel err:", rel)
    assert rel <= 4e-6


def test_misaligned_shard_buffers_are_bitwise_equal():
    x, y, _ = workloads.make("sharded", device=DEV, n=64)
    logp, lse = flp.fused_logp_forward(x, y)
    shards = []
    for buf, a, w in _shards(x, 2):
        n, wpad = buf.shape
        big = torch.full((n * (wpad + 3) + 1,), float("-inf"), dtype=torch.bfloat16, device=DEV)
        view = big[1:1 + n * (wpad + 3)].view(n, wpad + 3)[:, :wpad]
        view.copy_(buf)
        shards.append((view, a, w))
    s_logp, s_lse, _, _ = _sharded_forward(shards, y, V)
    assert torch.equal(_i(s_lse), _i(lse)) and torch.equal(_i(s_logp), _i(logp))


def test_ragged_vocab_sharding():
    """V = 1031: W = 72, 15 non-empty tiles; a last shard that ends the
    vocabulary may be ragged."""
    v = 1031
    W = flp.flp_tile_width(v)
    wl = workloads.Workload("rag", 40, v, 2.0, 8.0, 0.1, "normal", seed=2)
    x, y, _ = workloads.make(wl, device=DEV)
    logp, lse = flp.fused_logp_forward(x, y)
    cut = 8 * W
    shards = [(x[:, :cut].contiguous(), 0, cut), (x[:, cut:].contiguous(), cut, v - cut)]
    s_logp, s_lse, _, _ = _sharded_forward(shards, y, v)
    assert torch.equal(_i(s_lse), _i(lse)) and torch.equal(_i(s_logp), _i(logp))
    bad = x[:, :100].contiguous()
    with pytest.raises(flp.FusedLogpError, match="FLP_EUNSUPPORTED"):
        flp.logp_shard_partials(bad, 0, 100, v, y, torch.empty((40, 16), device=DEV),
                                torch.empty((40, 16), device=DEV), torch.empty(40, device=DEV))
