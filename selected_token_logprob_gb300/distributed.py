"""Multi-process forms of the selected-token logp path: vocabulary parallel
and row parallel, on top of the library's kernels.

Vocabulary parallel (RL-Kernel issue #241 "TP-aware deterministic logprob",
PR 3 and PR 6 bullets; PR #314 "Deterministic config option", Tensor Parallel
section): every rank holds the logits of its own slice of the vocabulary,
[vocab_start, vocab_start + real_width), on the tile grid of the whole
vocabulary.  Per call:

1. preflight: every rank publishes its shape, shard and mode, and all check
   that they agree (PR #314 review thread on the cross-rank agreement check:
   mismatched all-gather shapes hang or corrupt, so the check always runs
   when the group has more than one rank);
2. ``logp_shard_partials_ex`` writes this rank's tile partials and the
   selected logits it owns into one exchange block (``partials_block``);
3. one all-gather of the blocks, transport only (NCCL on device tensors,
   gloo through host copies);
4. every rank runs the same ``logp_merge_gathered_partials`` over the gathered
   blocks.  The result is bitwise the unsharded forward on every rank.

The backward needs no collective: the merged LSE is global and the upstream
gradient of logp is the same on every rank, so each rank writes its own
columns with ``logp_shard_backward``; the ranks' columns side by side are the
unsharded gradient bit for bit.

Row parallel (issue #241: the sequence / context axis is not a merge axis):
rows are independent and each row's bits do not depend on the batch, so each
rank runs the ordinary forward and backward on its rows; ``gather_rows``
assembles per-row results in global row order when a caller wants them.

The fused LM head in the same vocabulary-parallel layout (the
tensor-parallel output layer: each rank holds a slice of the weight's rows
on the 256-column tile grid, the hidden states on every rank): each rank
writes its tiles' partials into its own workspace, one all-gather of the
workspaces, the same merge on every rank (``fused_linear_logp_merge_gathered``)
-- bitwise the one-GPU result.  Its backward: each rank's slice gives its
dweight rows and its term of dhidden; the terms are all-gathered and summed
in rank order by the library (``sum_blocks``), the sum the one-GPU sharded
backward forms, so every rank has the same dhidden.

Nothing here computes: the arithmetic is in the library's kernels; this
module checks agreement, moves bytes and calls the C ABI.
"""

from __future__ import annotations

from dataclasses import asdict, dataclass

import torch
import torch.distributed as dist

from . import (IGNORE_INDEX, NUM_TILES, flp_tile_width, fused_linear_logp_merge_gathered,
               fused_linear_logp_shard_backward, fused_linear_logp_shard_partials, fused_linear_logp_workspace_size,
               fused_logp_backward, fused_logp_forward, logp_merge_gathered_partials, logp_shard_backward,
               logp_shard_partials, partials_block, partials_views, sum_blocks)

LINEAR_TILE = 256   # vocabulary columns per tile of the fused LM head

__all__ = [
    "PreflightError",
    "VocabParallelLinearLogp",
    "VocabParallelLogp",
    "gather_rows",
    "preflight",
    "row_parallel_logp_backward",
    "row_parallel_logp_forward",
    "vocab_parallel_linear_logp",
    "vocab_parallel_linear_logp_backward",
    "vocab_parallel_linear_logp_forward",
    "vocab_parallel_logp",
    "vocab_parallel_logp_backward",
    "vocab_parallel_logp_forward",
]


class PreflightError(ValueError):
    """Raised on every rank when the ranks of a group disagree on the call."""


@dataclass(frozen=True)
class _Spec:
    mode: str
    n: int
    v_total: int
    vocab_start: int
    real_width: int
    dtype: str
    temperature: float
    ignore_index: int
    masked: bool
    d: int = 0          # hidden size (the fused LM head)


def _world(group) -> tuple[int, int]:
    if not dist.is_available() or not dist.is_initialized():
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def _check_specs(specs: list[dict]) -> tuple[list[int], list[int]]:
    """The agreement rules; raises PreflightError naming the first mismatch.
    Returns the ranks' (vocab_starts, real_widths)."""
    first = specs[0]
    same = ["mode", "v_total", "dtype", "temperature", "ignore_index", "masked"]
    if first["mode"] in ("vocab", "linear"):
        same.insert(1, "n")
    if first["mode"] == "linear":
        same.insert(2, "d")
    for key in same:
        vals = [s[key] for s in specs]
        if any(v != vals[0] for v in vals):
            raise PreflightError(f"ranks disagree on {key}: " +
                                 ", ".join(f"rank {r}: {v!r}" for r, v in enumerate(vals)))
    starts = [s["vocab_start"] for s in specs]
    widths = [s["real_width"] for s in specs]
    if first["mode"] not in ("vocab", "linear"):
        return starts, widths
    v_total = first["v_total"]
    if len(specs) > NUM_TILES:
        raise PreflightError(f"a vocabulary-parallel group has at most {NUM_TILES} ranks (got {len(specs)})")
    w = flp_tile_width(v_total) if first["mode"] == "vocab" else LINEAR_TILE
    n_tiles = -(-v_total // w)
    owner = [-1] * n_tiles
    for r, (a, b) in enumerate(zip(starts, widths)):
        if b < 1 or a < 0 or a + b > v_total:
            raise PreflightError(f"rank {r}: shard [{a}, {a + b}) is not inside the vocabulary [0, {v_total})")
        if a % w or (a + b != v_total and b % w):
            raise PreflightError(f"rank {r}: shard [{a}, {a + b}) is off the {w}-column tile grid of "
                                 f"a {v_total}-entry vocabulary (bounds must be multiples of {w})")
        for k in range(a // w, -(-(a + b) // w)):
            if owner[k] >= 0:
                raise PreflightError(f"tile {k} (columns from {k * w}) is held by rank {owner[k]} and rank {r}")
            owner[k] = r
    missing = [k for k, o in enumerate(owner) if o < 0]
    if missing:
        raise PreflightError(f"tiles {missing} (columns from {missing[0] * w}) are held by no rank")
    return starts, widths


def preflight(mode: str, n: int, v_total: int, vocab_start: int, real_width: int, dtype: torch.dtype,
              temperature: float, ignore_index: int, masked: bool, group=None,
              d: int = 0) -> tuple[list[int], list[int]]:
    """All ranks publish their call and check that they agree; on a mismatch
    every rank raises the same PreflightError, before any exchange of
    tensors.  mode "vocab": the same N, vocabulary, dtype, temperature,
    ignore_index and mask use, and shards on the tile grid covering every
    tile exactly once; mode "linear" (the fused LM head): the same, with the
    hidden size d, on the 256-column grid.  mode "rows": the same vocabulary
    and mode (row counts may differ).  Returns every rank's (vocab_start,
    real_width)."""
    spec = asdict(_Spec(mode, int(n), int(v_total), int(vocab_start), int(real_width), str(dtype),
                        float(temperature), int(ignore_index), bool(masked), int(d)))
    world, _ = _world(group)
    specs = [spec]
    if world > 1:
        specs = [None] * world
        dist.all_gather_object(specs, spec, group=group)
    return _check_specs(specs)


def _all_gather_flat(block: torch.Tensor, group) -> torch.Tensor:
    """[world, L] of every rank's [L] block, in rank order (transport only)."""
    world, _ = _world(group)
    if world == 1:
        return block.view(1, -1)
    if block.is_cuda and dist.get_backend(group) == "nccl":
        out = torch.empty((world, block.numel()), dtype=block.dtype, device=block.device)
        dist.all_gather_into_tensor(out.view(-1), block.contiguous(), group=group)
        return out
    host = block.detach().to("cpu")
    out = torch.empty((world, block.numel()), dtype=block.dtype)
    dist.all_gather(list(out.unbind(0)), host, group=group)
    return out.to(block.device)


def vocab_parallel_logp_forward(shard_logits: torch.Tensor, targets: torch.Tensor, vocab_start: int,
                                v_total: int, real_width: int | None = None, group=None,
                                ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                                active_mask: torch.Tensor | None = None, with_lse_lo: bool = False):
    """(logp, lse[, lse_lo]) FP32 [N] of the whole vocabulary on every rank,
    from this rank's shard_logits [N, >= real_width] (global columns
    [vocab_start, vocab_start + real_width)); bitwise the unsharded
    forward."""
    n = shard_logits.shape[0]
    width = shard_logits.shape[1] if real_width is None else int(real_width)
    starts, widths = preflight("vocab", n, v_total, vocab_start, width, shard_logits.dtype, temperature,
                               ignore_index, active_mask is not None, group)
    block = partials_block(n, shard_logits.device)
    pm, ps, sel = partials_views(block, n)
    logp_shard_partials(shard_logits[:, :width] if width < shard_logits.shape[1] else shard_logits,
                        vocab_start, width, v_total, targets, pm, ps, sel, temperature=temperature)
    gathered = _all_gather_flat(block, group)
    return logp_merge_gathered_partials(gathered, starts, widths, targets, v_total, ignore_index,
                                        with_lse_lo=with_lse_lo, temperature=temperature,
                                        active_mask=active_mask)


def vocab_parallel_logp_backward(shard_logits: torch.Tensor, targets: torch.Tensor, vocab_start: int,
                                 v_total: int, lse: torch.Tensor, grad: torch.Tensor,
                                 lse_lo: torch.Tensor | None = None, real_width: int | None = None,
                                 ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                                 active_mask: torch.Tensor | None = None, dshard: torch.Tensor | None = None):
    """This rank's columns of the gradient (no collective): [N, real_width]."""
    width = shard_logits.shape[1] if real_width is None else int(real_width)
    return logp_shard_backward(shard_logits, vocab_start, width, v_total, targets, lse, grad, ignore_index,
                               dshard=dshard, lse_lo=lse_lo, temperature=temperature, active_mask=active_mask)


class VocabParallelLogp(torch.autograd.Function):
    """logp = VocabParallelLogp.apply(shard_logits, targets, vocab_start,
    v_total, real_width, group, ignore_index, temperature, active_mask): the
    selected-token logp over a vocabulary split across the group's ranks.
    Saves only the O(N) merged LSE and its residual; the backward writes this
    rank's columns of dlogits (padding columns past real_width get 0)."""

    @staticmethod
    def forward(ctx, shard_logits, targets, vocab_start, v_total, real_width=None, group=None,
                ignore_index=IGNORE_INDEX, temperature=1.0, active_mask=None):
        width = shard_logits.shape[1] if real_width is None else int(real_width)
        logp, lse, lse_lo = vocab_parallel_logp_forward(shard_logits, targets, vocab_start, v_total,
                                                        real_width=width, group=group, ignore_index=ignore_index,
                                                        temperature=temperature, active_mask=active_mask,
                                                        with_lse_lo=True)
        ctx.save_for_backward(shard_logits, targets, lse, lse_lo, active_mask)
        ctx.args = (int(vocab_start), int(v_total), width, int(ignore_index), float(temperature))
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        shard_logits, targets, lse, lse_lo, active_mask = ctx.saved_tensors
        vocab_start, v_total, width, ignore_index, temperature = ctx.args
        g = grad_logp.to(torch.float32).contiguous()
        full = shard_logits.shape[1]
        d = torch.empty(shard_logits.shape, dtype=shard_logits.dtype, device=shard_logits.device)
        if width < full:
            d[:, width:].zero_()
        vocab_parallel_logp_backward(shard_logits, targets, vocab_start, v_total, lse, g, lse_lo=lse_lo,
                                     real_width=width, ignore_index=ignore_index, temperature=temperature,
                                     active_mask=active_mask, dshard=d[:, :width])
        return d, None, None, None, None, None, None, None, None


def vocab_parallel_logp(shard_logits: torch.Tensor, targets: torch.Tensor, vocab_start: int, v_total: int,
                        real_width: int | None = None, group=None, ignore_index: int = IGNORE_INDEX,
                        temperature: float = 1.0, active_mask: torch.Tensor | None = None) -> torch.Tensor:
    """Autograd-aware vocabulary-parallel selected-token logp (FP32 [N]) of
    this rank's shard_logits [N, >= real_width] (global columns
    [vocab_start, vocab_start + real_width); real_width defaults to the
    buffer's width)."""
    return VocabParallelLogp.apply(shard_logits, targets, vocab_start, v_total, real_width, group,
                                   ignore_index, temperature, active_mask)


def vocab_parallel_linear_logp_forward(hidden: torch.Tensor, weight_shard: torch.Tensor, targets: torch.Tensor,
                                       vocab_start: int, v_total: int, group=None, ignore_index: int = IGNORE_INDEX,
                                       temperature: float = 1.0, active_mask: torch.Tensor | None = None,
                                       with_lse_lo: bool = False):
    """(logp, lse[, lse_lo]) FP32 [N] of hidden [N, D] @ weight.T over the
    whole vocabulary, on every rank, from this rank's weight rows
    weight_shard [w, D] (global columns [vocab_start, vocab_start + w));
    bitwise the one-GPU fused LM head."""
    n, d = hidden.shape
    w = weight_shard.shape[0]
    starts, widths = preflight("linear", n, v_total, vocab_start, w, hidden.dtype, temperature, ignore_index,
                               active_mask is not None, group, d=d)
    ws = torch.empty(fused_linear_logp_workspace_size(n, v_total), dtype=torch.uint8, device=hidden.device)
    if n > 0:
        fused_linear_logp_shard_partials(hidden, weight_shard, vocab_start, v_total, targets, ws,
                                         temperature=temperature)
    gathered = _all_gather_flat(ws.view(torch.float32), group)
    return fused_linear_logp_merge_gathered(gathered, starts, widths, targets, v_total, ignore_index,
                                            with_lse_lo=with_lse_lo, temperature=temperature,
                                            active_mask=active_mask)


def vocab_parallel_linear_logp_backward(hidden: torch.Tensor, weight_shard: torch.Tensor, targets: torch.Tensor,
                                        vocab_start: int, v_total: int, lse: torch.Tensor, grad: torch.Tensor,
                                        group=None, lse_lo: torch.Tensor | None = None,
                                        ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                                        active_mask: torch.Tensor | None = None):
    """(dhidden [N, D] FP32, the same on every rank; this rank's dweight
    rows [w, D] FP32) of Σ_t g_t logp_t.  Each rank computes its slice's
    term of dhidden; the terms are all-gathered and summed in rank order, the
    order in which the one-GPU sharded backward adds its shards' terms when
    the ranks hold increasing slices."""
    n, d = hidden.shape
    term = torch.empty((n, d), dtype=torch.float32, device=hidden.device)
    dw = fused_linear_logp_shard_backward(hidden, weight_shard, vocab_start, v_total, targets, lse, grad, term,
                                          False, ignore_index, lse_lo=lse_lo, temperature=temperature,
                                          active_mask=active_mask)
    world, _ = _world(group)
    if world == 1:
        return term, dw
    gathered = _all_gather_flat(term.view(-1), group)
    return sum_blocks(gathered.view(world, n, d)), dw


class VocabParallelLinearLogp(torch.autograd.Function):
    """logp = VocabParallelLinearLogp.apply(hidden, weight_shard, targets,
    vocab_start, v_total, group, ignore_index, temperature, active_mask): the
    fused LM head with the weight's vocabulary rows split across the group's
    ranks.  Saves the O(N) merged LSE; the backward returns dhidden (the same
    on every rank) and this rank's dweight rows, in the dtypes of hidden and
    weight_shard."""

    @staticmethod
    def forward(ctx, hidden, weight_shard, targets, vocab_start, v_total, group=None, ignore_index=IGNORE_INDEX,
                temperature=1.0, active_mask=None):
        logp, lse, lse_lo = vocab_parallel_linear_logp_forward(hidden, weight_shard, targets, vocab_start, v_total,
                                                               group=group, ignore_index=ignore_index,
                                                               temperature=temperature, active_mask=active_mask,
                                                               with_lse_lo=True)
        ctx.save_for_backward(hidden, weight_shard, targets, lse, lse_lo, active_mask)
        ctx.args = (int(vocab_start), int(v_total), group, int(ignore_index), float(temperature))
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        hidden, weight_shard, targets, lse, lse_lo, active_mask = ctx.saved_tensors
        vocab_start, v_total, group, ignore_index, temperature = ctx.args
        g = grad_logp.to(torch.float32).contiguous()
        dh, dw = vocab_parallel_linear_logp_backward(hidden, weight_shard, targets, vocab_start, v_total, lse, g,
                                                     group=group, lse_lo=lse_lo, ignore_index=ignore_index,
                                                     temperature=temperature, active_mask=active_mask)
        dh = dh if hidden.dtype == torch.float32 else dh.to(hidden.dtype)
        dw = dw if weight_shard.dtype == torch.float32 else dw.to(weight_shard.dtype)
        return dh, dw, None, None, None, None, None, None, None


def vocab_parallel_linear_logp(hidden: torch.Tensor, weight_shard: torch.Tensor, targets: torch.Tensor,
                               vocab_start: int, v_total: int, group=None, ignore_index: int = IGNORE_INDEX,
                               temperature: float = 1.0, active_mask: torch.Tensor | None = None) -> torch.Tensor:
    """Autograd-aware vocabulary-parallel fused LM head + selected-token logp
    (FP32 [N]) of hidden [N, D] @ weight.T, this rank holding weight rows
    [vocab_start, vocab_start + weight_shard.shape[0])."""
    return VocabParallelLinearLogp.apply(hidden, weight_shard, targets, vocab_start, v_total, group, ignore_index,
                                         temperature, active_mask)


def gather_rows(t: torch.Tensor, group=None) -> torch.Tensor:
    """Concatenation over the group's ranks, in rank order, of each rank's
    [n_r, ...] tensor (row counts may differ): pure transport."""
    world, _ = _world(group)
    if world == 1:
        return t
    counts = [None] * world
    dist.all_gather_object(counts, int(t.shape[0]), group=group)
    width = max(counts)
    pad = torch.zeros((width,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    pad[:t.shape[0]] = t
    out = _all_gather_flat(pad.view(-1), group).view((world, width) + tuple(t.shape[1:]))
    return torch.cat([out[r, :counts[r]] for r in range(world)], dim=0)


def row_parallel_logp_forward(logits: torch.Tensor, targets: torch.Tensor, group=None,
                              ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                              active_mask: torch.Tensor | None = None, gather: bool = True):
    """This rank's rows of one global batch: the ordinary forward on them,
    after a preflight that the ranks agree on the vocabulary and the mode.
    Returns (logp, lse, lse_lo) of the local rows and, with ``gather``, the
    global (logp, lse) in rank order as well.  No collective is needed for
    the backward: ``fused_logp_backward`` on the local rows."""
    preflight("rows", logits.shape[0], logits.shape[1], 0, logits.shape[1], logits.dtype, temperature,
              ignore_index, active_mask is not None, group)
    local = fused_logp_forward(logits, targets, ignore_index, with_lse_lo=True, temperature=temperature,
                               active_mask=active_mask)
    if not gather:
        return local
    return local, (gather_rows(local[0], group), gather_rows(local[1], group))


def row_parallel_logp_backward(logits: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                               grad: torch.Tensor, lse_lo: torch.Tensor | None = None,
                               ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                               active_mask: torch.Tensor | None = None) -> torch.Tensor:
    """The local rows' dlogits (no collective)."""
    return fused_logp_backward(logits, targets, lse, grad, ignore_index, lse_lo=lse_lo, temperature=temperature,
                               active_mask=active_mask)
