"""Host logic of the multi-process forms (no GPU): the preflight agreement of
a vocabulary-parallel group (issue #241 / PR #314: mismatched all-gather
shapes must be caught before any exchange), the transport of the exchange
blocks and of ragged row blocks, on world-size-2 and -3 gloo groups of CPU
processes.  A preflight that finds a mismatch raises on every rank; no test
waits beyond its time limit."""

import pytest
import torch

import selected_token_logprob_gb300 as flp
from selected_token_logprob_gb300 import _lib, distributed as fd
from dist_util import run_ranks

V = 151936
W = 9496


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    _lib.load(build_if_missing=True)


def _spec(**kw):
    base = dict(mode="vocab", n=64, v_total=V, vocab_start=0, real_width=V, dtype="torch.bfloat16",
                temperature=1.0, ignore_index=-100, masked=False)
    base.update(kw)
    return base


def test_check_specs_accepts_tile_grid_partitions():
    for bounds in ([(0, V)], [(0, 8 * W), (8 * W, 8 * W)], [(0, 4 * W), (4 * W, 4 * W), (8 * W, 8 * W)],
                   [(8 * W, 8 * W), (0, 8 * W)], [(k * W, W) for k in range(16)]):
        specs = [_spec(vocab_start=a, real_width=b) for a, b in bounds]
        assert fd._check_specs(specs) == ([a for a, _ in bounds], [b for _, b in bounds])
    # a ragged vocabulary: the last shard ends the vocabulary off the grid
    v = 5000
    w = flp.flp_tile_width(v)
    specs = [_spec(v_total=v, vocab_start=0, real_width=3 * w), _spec(v_total=v, vocab_start=3 * w,
                                                                     real_width=v - 3 * w)]
    fd._check_specs(specs)


@pytest.mark.parametrize("bad, match", [
    ([(0, 8 * W), (8 * W + 8, 8 * W - 8)], "tile grid"),          # second shard starts off the grid
    ([(0, 8 * W - 8), (8 * W - 8, 8 * W + 8)], "tile grid"),      # first shard ends off the grid
    ([(0, 8 * W), (7 * W, 9 * W)], "held by rank 0 and rank 1"),  # overlap
    ([(0, 7 * W), (8 * W, 8 * W)], "held by no rank"),            # gap
    ([(0, 8 * W), (8 * W, 9 * W)], "not inside"),                 # past the vocabulary
])
def test_check_specs_rejects_bad_partitions(bad, match):
    specs = [_spec(vocab_start=a, real_width=b) for a, b in bad]
    with pytest.raises(fd.PreflightError, match=match):
        fd._check_specs(specs)


@pytest.mark.parametrize("key, other", [("temperature", 0.7), ("n", 65), ("v_total", V - 8),
                                        ("dtype", "torch.float16"), ("ignore_index", -1), ("masked", True),
                                        ("mode", "rows")])
def test_check_specs_rejects_disagreement(key, other):
    specs = [_spec(vocab_start=0, real_width=8 * W), _spec(vocab_start=8 * W, real_width=8 * W)]
    specs[1][key] = other
    with pytest.raises(fd.PreflightError, match=f"ranks disagree on {key}"):
        fd._check_specs(specs)


def test_row_mode_allows_different_row_counts():
    specs = [_spec(mode="rows", n=10), _spec(mode="rows", n=7)]
    fd._check_specs(specs)
    specs[1]["temperature"] = 0.5
    with pytest.raises(fd.PreflightError, match="temperature"):
        fd._check_specs(specs)


def _preflight_rank(rank, world, case):
    """Each rank describes its call; `case` plants one mismatch on rank 1."""
    half = 8 * W
    start, width, temp, n = (0, half, 1.0, 64) if rank == 0 else (half, V - half, 1.0, 64)
    if rank == 1 and case == "grid":
        start, width = half + 8, V - half - 8
    if rank == 1 and case == "temperature":
        temp = 0.7
    if rank == 1 and case == "rows":
        n = 63
    return fd.preflight("vocab", n, V, start, width, torch.bfloat16, temp, -100, False)


@pytest.mark.parametrize("case, match", [("grid", "tile grid"), ("temperature", "ranks disagree on temperature"),
                                         ("rows", "ranks disagree on n")])
def test_preflight_mismatch_raises_on_every_rank(case, match):
    res = run_ranks(_preflight_rank, 2, (case,), timeout=120)
    for rank in range(2):
        kind, val = res[rank]
        assert kind == "raised", (rank, val)
        assert val[0] == "PreflightError" and match in val[1], val


def test_preflight_agreement_returns_every_shard():
    res = run_ranks(_preflight_rank, 2, ("none",), timeout=120)
    for rank in range(2):
        assert res[rank] == ("ok", ([0, 8 * W], [8 * W, V - 8 * W]))


def _exchange_rank(rank, world, n):
    """Every rank fills its exchange block with values that name the rank and
    the position; returns the gathered [world, 33 n]."""
    block = flp.partials_block(n, "cpu")
    block.copy_(torch.arange(block.numel(), dtype=torch.float32) + 1000.0 * rank)
    pm, ps, sel = flp.partials_views(block, n)
    assert pm.shape == (n, 16) and ps.shape == (n, 16) and sel.shape == (n,)
    assert ps.data_ptr() - pm.data_ptr() == 4 * 16 * n and sel.data_ptr() - pm.data_ptr() == 4 * 32 * n
    return fd._all_gather_flat(block, None).numpy()   # plain arrays cross the result queue


def test_exchange_blocks_land_in_rank_order():
    n = 5
    res = run_ranks(_exchange_rank, 3, (n,), timeout=120)
    for rank in range(3):
        kind, got = res[rank]
        assert kind == "ok", got
        assert got.shape == (3, 33 * n)
        for r in range(3):
            assert torch.equal(torch.from_numpy(got[r]), torch.arange(33 * n, dtype=torch.float32) + 1000.0 * r)


def _gather_rows_rank(rank, world):
    rows = [3, 0, 5][rank]
    t = torch.arange(rows * 2, dtype=torch.float32).view(rows, 2) + 100 * rank
    return fd.gather_rows(t).numpy()


def test_gather_rows_uneven_counts():
    res = run_ranks(_gather_rows_rank, 3, (), timeout=120)
    want = torch.cat([torch.arange(6, dtype=torch.float32).view(3, 2),
                      torch.arange(10, dtype=torch.float32).view(5, 2) + 200])
    for rank in range(3):
        kind, got = res[rank]
        assert kind == "ok", got
        assert torch.equal(torch.from_numpy(got), want)


def _lspec(**kw):
    base = _spec(mode="linear", d=512, v_total=20000)
    base.update(kw)
    return base


def test_linear_mode_checks_the_256_grid_and_the_hidden_size():
    """The fused LM head's vocabulary-parallel preflight: slices on the
    256-column grid of the fused kernel (not the logits path's tile width),
    covering every tile once, and the same hidden size on every rank."""
    v = 20000
    fd._check_specs([_lspec(vocab_start=0, real_width=10240), _lspec(vocab_start=10240, real_width=v - 10240)])
    fd._check_specs([_lspec(vocab_start=19968, real_width=32), _lspec(vocab_start=0, real_width=19968)])
    with pytest.raises(fd.PreflightError, match="256-column tile grid"):
        fd._check_specs([_lspec(vocab_start=0, real_width=10000), _lspec(vocab_start=10000, real_width=10000)])
    with pytest.raises(fd.PreflightError, match="held by no rank"):
        fd._check_specs([_lspec(vocab_start=0, real_width=9984), _lspec(vocab_start=10240, real_width=v - 10240)])
    specs = [_lspec(vocab_start=0, real_width=10240), _lspec(vocab_start=10240, real_width=v - 10240)]
    specs[1]["d"] = 1024
    with pytest.raises(fd.PreflightError, match="ranks disagree on d"):
        fd._check_specs(specs)
