"""Selected-token log-probability on GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/fused_logp.h``: argument
checking and marshalling of torch tensors into pointers, sizes and the current
CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; torch only provides device memory and streams.  There is no CPU or
PyTorch fallback: without the built library every call raises.

Entry points (same names as the C ABI):
    fused_logp_forward(logits, targets, ignore_index) -> (logp, lse)
        (with_lse_lo=True also returns lse_lo, the FP32 rounding residual of
        the LSE, which the backward accepts to avoid the FP32 quantisation)
    fused_logp_backward(logits, targets, lse, grad, ignore_index, lse_lo=None)
        -> dlogits
    logp_shard_partials(shard_logits, vocab_start, real_width, v_total, targets,
                        part_max, part_sum, sel)
    logp_merge_partials(part_max, part_sum, sel, targets, v_total,
                        ignore_index) -> (logp, lse)
``FusedLogp``, an autograd function that saves only the O(N) LSE (and its
residual), and ``flp_device_error`` / ``flp_selftest_wait_timeout`` for the
device-side health word.

Logits are BF16, FP16 or FP32 [N, V] (row stride may exceed V: pass a column
slice of a wider buffer), targets int64 [N], the upstream gradient FP32 [N];
logp and lse are FP32 [N]; the gradient has the logits' dtype.
``ignore_index`` defaults to -100.  ``temperature`` T scales the logits by
1/T before the log-softmax (the gradient is with respect to the unscaled
logits); ``active_mask`` (bool or uint8 [N]) excludes rows explicitly.  The
shard partials and their merge must use the same temperature.
"""

from __future__ import annotations

import torch

from . import _lib
from ._lib import FusedLogpError

IGNORE_INDEX = -100
NUM_TILES = 16
_DTYPES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}

__all__ = [
    "FusedLinearLogp",
    "FusedLogp",
    "FusedLogpError",
    "IGNORE_INDEX",
    "NUM_TILES",
    "flp_device_error",
    "flp_selftest_ex2_bias",
    "flp_selftest_wait_timeout",
    "flp_tile_width",
    "fused_logp",
    "fused_logp_backward",
    "fused_logp_forward",
    "fused_linear_logp",
    "fused_linear_logp_backward",
    "fused_linear_logp_backward_workspace_size",
    "fused_linear_logp_forward",
    "fused_linear_logp_forward_noalloc",
    "fused_linear_logp_merge",
    "fused_linear_logp_shard_backward",
    "fused_linear_logp_shard_partials",
    "fused_linear_logp_workspace_size",
    "fused_linear_logp_merge_gathered",
    "sum_blocks",
    "logp_grpo_loss",
    "logp_grpo_loss_counts",
    "logp_grpo_loss_workspace_size",
    "logp_merge_gathered_partials",
    "logp_merge_partials",
    "logp_shard_backward",
    "logp_shard_partials",
]
GRPO_MODES = {"token_mean": 0, "seq_mean_token_mean": 1, "seq_mean_token_sum": 2}


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _rows(x: torch.Tensor, name: str):
    """(n, v, ld) of a 2-D tensor whose rows are contiguous."""
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D [N, V], got shape {tuple(x.shape)}")
    n, v = x.shape
    if v > 1 and x.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous (stride(1) == 1)")
    ld = x.stride(0) if n > 1 else max(v, x.stride(0))
    if ld < v:
        raise ValueError(f"{name} row stride {ld} is smaller than its width {v}")
    return n, v, ld


def _vec(t: torch.Tensor, name: str, n: int, dtype: torch.dtype) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 1 or t.shape[0] != n:
        raise ValueError(f"{name} must have shape [{n}], got {tuple(t.shape)}")
    if n > 1 and t.stride(0) != 1:
        raise ValueError(f"{name} must be contiguous")


def _cuda(*ts) -> None:
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")


def flp_tile_width(v: int) -> int:
    """Tile width W = 8 * ceil(v / 128) of a v-column vocabulary."""
    return int(_lib.load().flp_tile_width(int(v)))


def _opt_ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _dtype(x: torch.Tensor, name: str) -> int:
    if x.dtype not in _DTYPES:
        raise TypeError(f"{name} must be bfloat16, float16 or float32, got {x.dtype}")
    return _DTYPES[x.dtype]


def _inv_temperature(temperature: float) -> float:
    t = float(temperature)
    if not (t > 0.0) or t == float("inf"):
        raise ValueError(f"temperature must be finite and > 0, got {temperature}")
    return 1.0 / t   # rounded to binary32 at the C boundary


def _mask(active_mask: torch.Tensor | None, n: int) -> int | None:
    if active_mask is None:
        return None
    if active_mask.dtype not in (torch.bool, torch.uint8):
        raise TypeError("active_mask must be bool or uint8")
    if active_mask.dim() != 1 or active_mask.shape[0] != n or (n > 1 and active_mask.stride(0) != 1):
        raise ValueError(f"active_mask must be a contiguous [{n}] tensor")
    _cuda(active_mask)
    return active_mask.data_ptr()


def fused_logp_forward(logits: torch.Tensor, targets: torch.Tensor,
                       ignore_index: int = IGNORE_INDEX,
                       logp: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                       lse_lo: torch.Tensor | None = None, with_lse_lo: bool = False,
                       temperature: float = 1.0, active_mask: torch.Tensor | None = None):
    """(logp, lse), FP32 [N] each, of logits [N, V]; (logp, lse, lse_lo)
    when ``with_lse_lo`` is true or an ``lse_lo`` buffer is given."""
    n, v, ld = _rows(logits, "logits")
    dt = _dtype(logits, "logits")
    inv_t = _inv_temperature(temperature)
    _vec(targets, "targets", n, torch.int64)
    dev = logits.device
    logp = torch.empty(n, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(n, dtype=torch.float32, device=dev) if lse is None else lse
    want_lo = with_lse_lo or lse_lo is not None
    if want_lo and lse_lo is None:
        lse_lo = torch.empty(n, dtype=torch.float32, device=dev)
    _vec(logp, "logp", n, torch.float32)
    _vec(lse, "lse", n, torch.float32)
    _cuda(logits, targets, logp, lse)
    if want_lo:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    mp = _mask(active_mask, n)
    if n > 0:
        st = _lib.load().fused_logp_forward_ex(logits.data_ptr(), dt, n, v, ld, targets.data_ptr(),
                                               int(ignore_index), mp, inv_t, logp.data_ptr(),
                                               lse.data_ptr(), _opt_ptr(lse_lo), _stream(logits))
        _lib.check("fused_logp_forward", st)
    return (logp, lse, lse_lo) if want_lo else (logp, lse)


def fused_logp_backward(logits: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                        grad: torch.Tensor, ignore_index: int = IGNORE_INDEX,
                        dlogits: torch.Tensor | None = None,
                        lse_lo: torch.Tensor | None = None, temperature: float = 1.0,
                        active_mask: torch.Tensor | None = None) -> torch.Tensor:
    """dlogits [N, V] (the logits' dtype) = grad / T * (onehot(targets) -
    softmax(logits / T)).

    ``dlogits`` may be ``logits`` itself (in-place gradient).  ``lse_lo`` is
    the residual returned by the forward with ``with_lse_lo=True``."""
    n, v, ld = _rows(logits, "logits")
    dt = _dtype(logits, "logits")
    inv_t = _inv_temperature(temperature)
    _vec(targets, "targets", n, torch.int64)
    _vec(lse, "lse", n, torch.float32)
    _vec(grad, "grad", n, torch.float32)
    if lse_lo is not None:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    if dlogits is None:
        dlogits = torch.empty((n, v), dtype=logits.dtype, device=logits.device)
    if dlogits.dtype != logits.dtype or tuple(dlogits.shape) != (n, v):
        raise ValueError("dlogits must have the logits' dtype and shape")
    _, _, ld_out = _rows(dlogits, "dlogits")
    _cuda(logits, targets, lse, grad, dlogits)
    mp = _mask(active_mask, n)
    if n == 0:
        return dlogits
    st = _lib.load().fused_logp_backward_ex(logits.data_ptr(), dt, n, v, ld, targets.data_ptr(),
                                            int(ignore_index), mp, inv_t, lse.data_ptr(),
                                            _opt_ptr(lse_lo), grad.data_ptr(), dlogits.data_ptr(),
                                            ld_out, _stream(logits))
    _lib.check("fused_logp_backward", st)
    return dlogits


def logp_shard_partials(shard_logits: torch.Tensor, vocab_start: int, real_width: int,
                        v_total: int, targets: torch.Tensor, part_max: torch.Tensor,
                        part_sum: torch.Tensor, sel: torch.Tensor,
                        temperature: float = 1.0) -> None:
    """Write one vocab shard's tile partials into part_max/part_sum [N, 16]
    and, for rows whose target it owns, the selected logit into sel [N].

    shard_logits is BF16 [N, W_pad] holding global columns
    [vocab_start, vocab_start + real_width); columns >= real_width are padding
    and are never read."""
    n, wpad, ld = _rows(shard_logits, "shard_logits")
    dt = _dtype(shard_logits, "shard_logits")
    inv_t = _inv_temperature(temperature)
    if real_width > wpad:
        raise ValueError(f"real_width {real_width} exceeds the shard width {wpad}")
    _vec(targets, "targets", n, torch.int64)
    for name, t in (("part_max", part_max), ("part_sum", part_sum)):
        if t.dtype != torch.float32 or tuple(t.shape) != (n, NUM_TILES) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous FP32 [{n}, {NUM_TILES}] tensor")
    _vec(sel, "sel", n, torch.float32)
    _cuda(shard_logits, targets, part_max, part_sum, sel)
    if n == 0:
        return
    st = _lib.load().logp_shard_partials_ex(shard_logits.data_ptr(), dt, n, ld, int(vocab_start),
                                            int(real_width), int(v_total), inv_t,
                                            targets.data_ptr(), part_max.data_ptr(),
                                            part_sum.data_ptr(), sel.data_ptr(),
                                            _stream(shard_logits))
    _lib.check("logp_shard_partials", st)


def logp_merge_partials(part_max: torch.Tensor, part_sum: torch.Tensor, sel: torch.Tensor,
                        targets: torch.Tensor, v_total: int,
                        ignore_index: int = IGNORE_INDEX,
                        logp: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                        lse_lo: torch.Tensor | None = None, with_lse_lo: bool = False,
                        temperature: float = 1.0, active_mask: torch.Tensor | None = None):
    """(logp, lse) [or (logp, lse, lse_lo)] from the tile partials of shards
    covering [0, v_total)."""
    inv_t = _inv_temperature(temperature)
    n = targets.shape[0] if targets.dim() == 1 else -1
    _vec(targets, "targets", n, torch.int64)
    for name, t in (("part_max", part_max), ("part_sum", part_sum)):
        if t.dtype != torch.float32 or tuple(t.shape) != (n, NUM_TILES) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous FP32 [{n}, {NUM_TILES}] tensor")
    _vec(sel, "sel", n, torch.float32)
    dev = targets.device
    logp = torch.empty(n, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(n, dtype=torch.float32, device=dev) if lse is None else lse
    want_lo = with_lse_lo or lse_lo is not None
    if want_lo and lse_lo is None:
        lse_lo = torch.empty(n, dtype=torch.float32, device=dev)
    _vec(logp, "logp", n, torch.float32)
    _vec(lse, "lse", n, torch.float32)
    _cuda(part_max, part_sum, sel, targets, logp, lse)
    if want_lo:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    mp = _mask(active_mask, n)
    if n > 0:
        st = _lib.load().logp_merge_partials_ex(part_max.data_ptr(), part_sum.data_ptr(),
                                                sel.data_ptr(), targets.data_ptr(),
                                                int(ignore_index), mp, n, int(v_total), inv_t,
                                                logp.data_ptr(), lse.data_ptr(), _opt_ptr(lse_lo),
                                                _stream(targets))
        _lib.check("logp_merge_partials", st)
    return (logp, lse, lse_lo) if want_lo else (logp, lse)


def logp_shard_backward(shard_logits: torch.Tensor, vocab_start: int, real_width: int, v_total: int,
                        targets: torch.Tensor, lse: torch.Tensor, grad: torch.Tensor,
                        ignore_index: int = IGNORE_INDEX, dshard: torch.Tensor | None = None,
                        lse_lo: torch.Tensor | None = None, temperature: float = 1.0,
                        active_mask: torch.Tensor | None = None) -> torch.Tensor:
    """Gradient [N, real_width] (the shard's dtype) of one vocabulary shard
    holding global columns [vocab_start, vocab_start + real_width) of a
    v_total-column vocabulary, from the merged (global) lse / lse_lo.  The
    shards' outputs side by side are the unsharded fused_logp_backward
    bitwise.  ``dshard`` may be the shard's own columns (in place)."""
    n, wpad, ld = _rows(shard_logits, "shard_logits")
    dt = _dtype(shard_logits, "shard_logits")
    inv_t = _inv_temperature(temperature)
    if not 0 < real_width <= wpad:
        raise ValueError(f"real_width {real_width} must be in [1, {wpad}]")
    _vec(targets, "targets", n, torch.int64)
    _vec(lse, "lse", n, torch.float32)
    _vec(grad, "grad", n, torch.float32)
    if lse_lo is not None:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    if dshard is None:
        dshard = torch.empty((n, real_width), dtype=shard_logits.dtype, device=shard_logits.device)
    if dshard.dtype != shard_logits.dtype or tuple(dshard.shape) != (n, real_width):
        raise ValueError(f"dshard must be a [{n}, {real_width}] tensor of the shard's dtype")
    _, _, ld_out = _rows(dshard, "dshard")
    _cuda(shard_logits, targets, lse, grad, dshard)
    mp = _mask(active_mask, n)
    if n == 0:
        return dshard
    st = _lib.load().logp_shard_backward_ex(shard_logits.data_ptr(), dt, n, ld, int(vocab_start),
                                            int(real_width), int(v_total), targets.data_ptr(),
                                            int(ignore_index), mp, inv_t, lse.data_ptr(), _opt_ptr(lse_lo),
                                            grad.data_ptr(), dshard.data_ptr(), ld_out,
                                            _stream(shard_logits))
    _lib.check("logp_shard_backward", st)
    return dshard


def partials_block(n: int, device) -> torch.Tensor:
    """One rank's exchange block for the vocabulary-parallel merge: FP32
    [33 n] = tile maxima [n, 16], tile sums [n, 16], selected logits [n]."""
    return torch.empty((2 * NUM_TILES + 1) * n, dtype=torch.float32, device=device)


def partials_views(block: torch.Tensor, n: int):
    """(part_max [n, 16], part_sum [n, 16], sel [n]) views of an exchange
    block, in the layout logp_merge_gathered_partials reads."""
    k = NUM_TILES * n
    return block[:k].view(n, NUM_TILES), block[k:2 * k].view(n, NUM_TILES), block[2 * k:2 * k + n]


def logp_merge_gathered_partials(gathered: torch.Tensor, vocab_starts, real_widths, targets: torch.Tensor,
                                 v_total: int, ignore_index: int = IGNORE_INDEX,
                                 logp: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                                 lse_lo: torch.Tensor | None = None, with_lse_lo: bool = False,
                                 temperature: float = 1.0, active_mask: torch.Tensor | None = None):
    """(logp, lse[, lse_lo]) from the exchange blocks of every rank of a
    vocabulary-parallel group, gathered as FP32 [world, 33 N] (rank r's block
    in row r; see ``partials_block``).  ``vocab_starts`` / ``real_widths`` give
    each rank's shard; the result is bitwise the unsharded forward."""
    import ctypes

    inv_t = _inv_temperature(temperature)
    n = targets.shape[0] if targets.dim() == 1 else -1
    _vec(targets, "targets", n, torch.int64)
    world = len(vocab_starts)
    if len(real_widths) != world:
        raise ValueError("vocab_starts and real_widths must have one entry per rank")
    block = (2 * NUM_TILES + 1) * n
    if (gathered.dtype != torch.float32 or gathered.dim() != 2 or gathered.shape[0] != world
            or gathered.shape[1] < block or gathered.stride(1) != 1):
        raise ValueError(f"gathered must be FP32 [{world}, >= {block}] with contiguous rows")
    dev = targets.device
    logp = torch.empty(n, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(n, dtype=torch.float32, device=dev) if lse is None else lse
    want_lo = with_lse_lo or lse_lo is not None
    if want_lo and lse_lo is None:
        lse_lo = torch.empty(n, dtype=torch.float32, device=dev)
    _vec(logp, "logp", n, torch.float32)
    _vec(lse, "lse", n, torch.float32)
    _cuda(gathered, targets, logp, lse)
    if want_lo:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    mp = _mask(active_mask, n)
    starts = (ctypes.c_int64 * max(1, world))(*[int(a) for a in vocab_starts])
    widths = (ctypes.c_int64 * max(1, world))(*[int(w) for w in real_widths])
    st = _lib.load().logp_merge_gathered_partials_ex(
        gathered.data_ptr(), gathered.stride(0) if world > 1 else 0, world, starts, widths, targets.data_ptr(),
        int(ignore_index), mp, n, int(v_total), inv_t, logp.data_ptr(), lse.data_ptr(), _opt_ptr(lse_lo),
        _stream(targets))
    _lib.check("logp_merge_gathered_partials", st)
    return (logp, lse, lse_lo) if want_lo else (logp, lse)


def _grpo_layout(cu_seqlens):
    """(cu_seqlens contiguous or None, number of sequences)."""
    if cu_seqlens is None:
        return None, 0
    if cu_seqlens.dtype != torch.int64 or cu_seqlens.dim() != 1 or cu_seqlens.shape[0] < 1:
        raise ValueError("cu_seqlens must be an int64 [S + 1] tensor")
    _cuda(cu_seqlens)
    cu_seqlens = cu_seqlens.contiguous()
    return cu_seqlens, cu_seqlens.shape[0] - 1


def logp_grpo_loss(logp: torch.Tensor, old_logp: torch.Tensor, advantages: torch.Tensor,
                   ref_logp: torch.Tensor | None = None, active_mask: torch.Tensor | None = None,
                   cu_seqlens: torch.Tensor | None = None, mode: str = "token_mean",
                   eps_lo: float = 0.2, eps_hi: float = 0.2, beta: float = 0.0,
                   normalizer: float = 0.0, token_loss: bool = False,
                   workspace: torch.Tensor | None = None, counted: bool = False):
    """GRPO clipped-surrogate loss of per-token logp: (loss FP32 [1], grad
    FP32 [N] = d loss / d logp) [+ per-token loss FP32 [N] if token_loss].
    ``grad`` is the upstream gradient for ``fused_logp_backward``.
    ``workspace`` (a CUDA byte tensor of logp_grpo_loss_workspace_size(N, S)
    bytes) is allocated when not given.  With ``counted`` the normaliser
    counts are not taken again: ``workspace`` must hold the counts of an
    earlier ``logp_grpo_loss_counts`` (or ``logp_grpo_loss``) call for the
    same active_mask, cu_seqlens, mode and normalizer tensors and values."""
    if mode not in GRPO_MODES:
        raise ValueError(f"mode must be one of {sorted(GRPO_MODES)} (got {mode!r})")
    n = logp.shape[0] if logp.dim() == 1 else -1
    for name, t in (("logp", logp), ("old_logp", old_logp), ("advantages", advantages)):
        _vec(t, name, n, torch.float32)
        _cuda(t)
    if ref_logp is not None:
        _vec(ref_logp, "ref_logp", n, torch.float32)
        _cuda(ref_logp)
    mp = _mask(active_mask, n)
    cu_seqlens, nseq = _grpo_layout(cu_seqlens)
    dev = logp.device
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    grad = torch.empty(n, dtype=torch.float32, device=dev)
    tl = torch.empty(n, dtype=torch.float32, device=dev) if token_loss else None
    if workspace is None:
        if counted:
            raise ValueError("counted=True needs the workspace that holds the counts")
        workspace = torch.empty(logp_grpo_loss_workspace_size(n, nseq), dtype=torch.uint8, device=dev)
    _cuda(workspace)
    fn = "logp_grpo_loss_counted" if counted else "logp_grpo_loss"
    st = getattr(_lib.load(), fn)(logp.data_ptr(), old_logp.data_ptr(), _opt_ptr(ref_logp),
                                  advantages.data_ptr(), mp, _opt_ptr(cu_seqlens), nseq, n,
                                  GRPO_MODES[mode], float(eps_lo), float(eps_hi), float(beta),
                                  float(normalizer), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), loss.data_ptr(),
                                  grad.data_ptr(), _opt_ptr(tl), _stream(logp))
    _lib.check(fn, st)
    return (loss, grad, tl) if token_loss else (loss, grad)


def logp_grpo_loss_counts(n: int, active_mask: torch.Tensor | None = None,
                          cu_seqlens: torch.Tensor | None = None, mode: str = "token_mean",
                          normalizer: float = 0.0, workspace: torch.Tensor | None = None,
                          stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """The normaliser counts of a GRPO batch layout (n tokens, the active
    mask, the sequences, the mode and normalizer) into ``workspace``
    (allocated when not given on the mask's or cu_seqlens' device), on
    ``stream`` (default: the current stream); returns the workspace for
    ``logp_grpo_loss(..., counted=True, workspace=...)``."""
    if mode not in GRPO_MODES:
        raise ValueError(f"mode must be one of {sorted(GRPO_MODES)} (got {mode!r})")
    n = int(n)
    mp = _mask(active_mask, n)
    cu_seqlens, nseq = _grpo_layout(cu_seqlens)
    if workspace is None:
        ref = active_mask if active_mask is not None else cu_seqlens
        if ref is None:
            raise ValueError("give the workspace when there is neither a mask nor cu_seqlens")
        workspace = torch.empty(logp_grpo_loss_workspace_size(n, nseq), dtype=torch.uint8, device=ref.device)
    _cuda(workspace)
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    st = _lib.load().logp_grpo_loss_counts(mp, _opt_ptr(cu_seqlens), nseq, n, GRPO_MODES[mode],
                                           float(normalizer), workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(), s.cuda_stream)
    _lib.check("logp_grpo_loss_counts", st)
    return workspace


def logp_grpo_loss_workspace_size(n: int, num_seqs: int = 0) -> int:
    """Bytes of device scratch that logp_grpo_loss needs."""
    import ctypes

    b = ctypes.c_int64(0)
    _lib.check("logp_grpo_loss_workspace_size",
               _lib.load().logp_grpo_loss_workspace_size(int(n), int(num_seqs), ctypes.byref(b)))
    return int(b.value)


def fused_linear_logp_workspace_size(n: int, v: int) -> int:
    """Bytes of device scratch that fused_linear_logp_forward needs for n rows
    and a v-entry vocabulary."""
    import ctypes

    b = ctypes.c_int64(0)
    _lib.check("fused_linear_logp_workspace_size",
               _lib.load().fused_linear_logp_workspace_size(int(n), int(v), ctypes.byref(b)))
    return int(b.value)


def fused_linear_logp_forward(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                              ignore_index: int = IGNORE_INDEX,
                              logp: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                              lse_lo: torch.Tensor | None = None, with_lse_lo: bool = False,
                              temperature: float = 1.0, active_mask: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None):
    """(logp, lse) FP32 [N] of the logits hidden @ weight.T (BF16 hidden
    [N, D], BF16 LM-head weight [V, D]) without materialising the logits;
    (logp, lse, lse_lo) when ``with_lse_lo`` or an ``lse_lo`` buffer is given.
    ``workspace`` (a CUDA byte tensor of at least
    ``fused_linear_logp_workspace_size(N, V)`` bytes) is allocated when not
    given."""
    n, d, ld_h = _rows(hidden, "hidden")
    v, d_w, ld_w = _rows(weight, "weight")
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("hidden and weight must be bfloat16")
    if d_w != d:
        raise ValueError(f"hidden has {d} columns but weight has {d_w}")
    inv_t = _inv_temperature(temperature)
    _vec(targets, "targets", n, torch.int64)
    dev = hidden.device
    logp = torch.empty(n, dtype=torch.float32, device=dev) if logp is None else logp
    lse = torch.empty(n, dtype=torch.float32, device=dev) if lse is None else lse
    want_lo = with_lse_lo or lse_lo is not None
    if want_lo and lse_lo is None:
        lse_lo = torch.empty(n, dtype=torch.float32, device=dev)
    _vec(logp, "logp", n, torch.float32)
    _vec(lse, "lse", n, torch.float32)
    _cuda(hidden, weight, targets, logp, lse)
    if want_lo:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    mp = _mask(active_mask, n)
    if n > 0:
        need = fused_linear_logp_workspace_size(n, v)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _cuda(workspace)
        wbytes = workspace.numel() * workspace.element_size()
        st = _lib.load().fused_linear_logp_forward(
            hidden.data_ptr(), n, d, ld_h, weight.data_ptr(), v, ld_w, targets.data_ptr(),
            int(ignore_index), mp, inv_t, workspace.data_ptr(), wbytes, logp.data_ptr(),
            lse.data_ptr(), _opt_ptr(lse_lo), _stream(hidden))
        _lib.check("fused_linear_logp_forward", st)
    return (logp, lse, lse_lo) if want_lo else (logp, lse)


def fused_linear_logp_backward_workspace_size(d: int, v: int) -> int:
    """Bytes of device scratch that fused_linear_logp_backward needs."""
    import ctypes

    b = ctypes.c_int64(0)
    _lib.check("fused_linear_logp_backward_workspace_size",
               _lib.load().fused_linear_logp_backward_workspace_size(int(d), int(v), ctypes.byref(b)))
    return int(b.value)


def fused_linear_logp_backward(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                               lse: torch.Tensor, grad: torch.Tensor, ignore_index: int = IGNORE_INDEX,
                               lse_lo: torch.Tensor | None = None, temperature: float = 1.0,
                               active_mask: torch.Tensor | None = None,
                               dhidden: torch.Tensor | None = None, dweight: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None, accumulate_dweight: bool = False):
    """(dhidden [N, D], dweight [V, D]) FP32 of sum_t grad[t] logp[t] for the
    fused LM head, from the forward's lse (and lse_lo); dZ is recomputed on
    the tensor cores in 4096-row chunks and never stored for all rows.  With
    ``accumulate_dweight`` the given ``dweight`` is added to, not overwritten
    (gradient accumulation over micro-batches)."""
    n, d, ld_h = _rows(hidden, "hidden")
    v, d_w, ld_w = _rows(weight, "weight")
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("hidden and weight must be bfloat16")
    if d_w != d:
        raise ValueError(f"hidden has {d} columns but weight has {d_w}")
    inv_t = _inv_temperature(temperature)
    _vec(targets, "targets", n, torch.int64)
    _vec(lse, "lse", n, torch.float32)
    _vec(grad, "grad", n, torch.float32)
    dev = hidden.device
    if lse_lo is not None:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    if dhidden is None:
        dhidden = torch.empty((n, d), dtype=torch.float32, device=dev)
    if dweight is None:
        if accumulate_dweight:
            raise ValueError("accumulate_dweight needs a dweight tensor to add to")
        dweight = torch.empty((v, d), dtype=torch.float32, device=dev)
    if dhidden.dtype != torch.float32 or tuple(dhidden.shape) != (n, d):
        raise ValueError("dhidden must be float32 [N, D]")
    if dweight.dtype != torch.float32 or tuple(dweight.shape) != (v, d):
        raise ValueError("dweight must be float32 [V, D]")
    _, _, ld_dh = _rows(dhidden, "dhidden")
    _, _, ld_dw = _rows(dweight, "dweight")
    _cuda(hidden, weight, targets, lse, grad, dhidden, dweight)
    mp = _mask(active_mask, n)
    if workspace is None and n > 0:
        workspace = torch.empty(fused_linear_logp_backward_workspace_size(d, v), dtype=torch.uint8, device=dev)
    if workspace is None:
        wptr, wbytes = None, 0
    else:
        _cuda(workspace)
        wptr, wbytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = _lib.load().fused_linear_logp_backward(
        hidden.data_ptr(), n, d, ld_h, weight.data_ptr(), v, ld_w, targets.data_ptr(), int(ignore_index), mp,
        inv_t, lse.data_ptr(), _opt_ptr(lse_lo), grad.data_ptr(), wptr, wbytes, dhidden.data_ptr(), ld_dh,
        dweight.data_ptr(), ld_dw, int(bool(accumulate_dweight)), _stream(hidden))
    _lib.check("fused_linear_logp_backward", st)
    return dhidden, dweight


def fused_linear_logp_forward_noalloc(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                                      logp: torch.Tensor, lse: torch.Tensor,
                                      lse_lo: torch.Tensor | None = None,
                                      ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                                      active_mask: torch.Tensor | None = None):
    """fused_linear_logp_forward for callers that cannot allocate: the caller
    passes the outputs, and the library uses its fixed 16 MiB static scratch
    instead of a workspace (at most 3527 rows per call at V = 151936; calls
    must not overlap on the GPU).  Nothing is allocated here."""
    n, d, ld_h = _rows(hidden, "hidden")
    v, d_w, ld_w = _rows(weight, "weight")
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("hidden and weight must be bfloat16")
    if d_w != d:
        raise ValueError(f"hidden has {d} columns but weight has {d_w}")
    inv_t = _inv_temperature(temperature)
    _vec(targets, "targets", n, torch.int64)
    _vec(logp, "logp", n, torch.float32)
    _vec(lse, "lse", n, torch.float32)
    _cuda(hidden, weight, targets, logp, lse)
    if lse_lo is not None:
        _vec(lse_lo, "lse_lo", n, torch.float32)
        _cuda(lse_lo)
    mp = _mask(active_mask, n)
    st = _lib.load().fused_linear_logp_forward_noalloc(
        hidden.data_ptr(), n, d, ld_h, weight.data_ptr(), v, ld_w, targets.data_ptr(), int(ignore_index),
        mp, inv_t, logp.data_ptr(), lse.data_ptr(), _opt_ptr(lse_lo), _stream(hidden))
    _lib.check("fused_linear_logp_forward_noalloc", st)


class FusedLogp(torch.autograd.Function):
    """logp = FusedLogp.apply(logits, targets, ignore_index); the backward
    writes dlogits straight to BF16 from the saved FP32 LSE (O(N) state)."""

    @staticmethod
    def forward(ctx, logits, targets, ignore_index=IGNORE_INDEX, temperature=1.0,
                active_mask=None):
        logp, lse, lse_lo = fused_logp_forward(logits, targets, ignore_index, with_lse_lo=True,
                                               temperature=temperature, active_mask=active_mask)
        ctx.save_for_backward(logits, targets, lse, lse_lo, active_mask)
        ctx.ignore_index = ignore_index
        ctx.temperature = temperature
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        logits, targets, lse, lse_lo, active_mask = ctx.saved_tensors
        g = grad_logp.to(torch.float32).contiguous()
        d = fused_logp_backward(logits, targets, lse, g, ctx.ignore_index, lse_lo=lse_lo,
                                temperature=ctx.temperature, active_mask=active_mask)
        return d, None, None, None, None


def fused_logp(logits: torch.Tensor, targets: torch.Tensor,
               ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
               active_mask: torch.Tensor | None = None) -> torch.Tensor:
    """Autograd-aware selected-token logp (FP32 [N])."""
    return FusedLogp.apply(logits, targets, ignore_index, temperature, active_mask)


def fused_linear_logp_shard_partials(hidden: torch.Tensor, weight_shard: torch.Tensor, vocab_start: int,
                                     v_total: int, targets: torch.Tensor, workspace: torch.Tensor,
                                     temperature: float = 1.0) -> None:
    """Tile partials of one vocabulary shard of the LM head (global columns
    [vocab_start, vocab_start + weight_shard.shape[0]), vocab_start a multiple
    of 256) into `workspace` (a byte tensor of
    fused_linear_logp_workspace_size(N, v_total) bytes shared by all shards)."""
    n, d, ld_h = _rows(hidden, "hidden")
    w, d_w, ld_w = _rows(weight_shard, "weight_shard")
    if hidden.dtype != torch.bfloat16 or weight_shard.dtype != torch.bfloat16:
        raise TypeError("hidden and weight_shard must be bfloat16")
    if d_w != d:
        raise ValueError(f"hidden has {d} columns but weight_shard has {d_w}")
    _vec(targets, "targets", n, torch.int64)
    _cuda(hidden, weight_shard, targets, workspace)
    st = _lib.load().fused_linear_logp_shard_partials(
        hidden.data_ptr(), n, d, ld_h, weight_shard.data_ptr(), w, ld_w, int(vocab_start), int(v_total),
        targets.data_ptr(), _inv_temperature(temperature), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(hidden))
    _lib.check("fused_linear_logp_shard_partials", st)


def fused_linear_logp_merge(workspace: torch.Tensor, v_total: int, targets: torch.Tensor,
                            ignore_index: int = IGNORE_INDEX, with_lse_lo: bool = False,
                            temperature: float = 1.0, active_mask: torch.Tensor | None = None):
    """(logp, lse[, lse_lo]) FP32 [N] from the shards' partials in `workspace`."""
    n = targets.shape[0]
    _vec(targets, "targets", n, torch.int64)
    dev = targets.device
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    lse_lo = torch.empty(n, dtype=torch.float32, device=dev) if with_lse_lo else None
    _cuda(workspace, targets)
    mp = _mask(active_mask, n)
    st = _lib.load().fused_linear_logp_merge(
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), n, int(v_total), targets.data_ptr(),
        int(ignore_index), mp, _inv_temperature(temperature), logp.data_ptr(), lse.data_ptr(), _opt_ptr(lse_lo),
        _stream(targets))
    _lib.check("fused_linear_logp_merge", st)
    return (logp, lse, lse_lo) if with_lse_lo else (logp, lse)


def fused_linear_logp_merge_gathered(gathered: torch.Tensor, vocab_starts, real_widths, targets: torch.Tensor,
                                     v_total: int, ignore_index: int = IGNORE_INDEX, with_lse_lo: bool = False,
                                     temperature: float = 1.0, active_mask: torch.Tensor | None = None):
    """(logp, lse[, lse_lo]) FP32 [N] of a vocabulary-parallel LM head from
    the ranks' all-gathered workspaces: ``gathered`` FP32 [world, >= block]
    in rank order, rank r having run ``fused_linear_logp_shard_partials`` on
    columns [vocab_starts[r], vocab_starts[r] + real_widths[r]) into its own
    workspace."""
    import ctypes

    if gathered.dtype != torch.float32 or gathered.dim() != 2 or gathered.stride(1) != 1:
        raise ValueError("gathered must be an FP32 [world, L] tensor with unit column stride")
    world = gathered.shape[0]
    if len(vocab_starts) != world or len(real_widths) != world:
        raise ValueError("vocab_starts and real_widths need one entry per rank")
    n = targets.shape[0]
    _vec(targets, "targets", n, torch.int64)
    dev = targets.device
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    lse_lo = torch.empty(n, dtype=torch.float32, device=dev) if with_lse_lo else None
    _cuda(gathered, targets)
    mp = _mask(active_mask, n)
    starts = (ctypes.c_int64 * max(1, world))(*[int(a) for a in vocab_starts])
    widths = (ctypes.c_int64 * max(1, world))(*[int(w) for w in real_widths])
    st = _lib.load().fused_linear_logp_merge_gathered(
        gathered.data_ptr(), gathered.stride(0), world, starts, widths, n, int(v_total), targets.data_ptr(),
        int(ignore_index), mp, _inv_temperature(temperature), logp.data_ptr(), lse.data_ptr(), _opt_ptr(lse_lo),
        _stream(targets))
    _lib.check("fused_linear_logp_merge_gathered", st)
    return (logp, lse, lse_lo) if with_lse_lo else (logp, lse)


def sum_blocks(blocks: torch.Tensor) -> torch.Tensor:
    """((b_0 + b_1) + b_2) + ... of FP32 blocks [world, rows, cols], one
    rounding per addition in block order (``flp_sum_blocks``)."""
    if blocks.dtype != torch.float32 or blocks.dim() != 3 or not blocks[0].is_contiguous():
        raise ValueError("blocks must be FP32 [world, rows, cols] with contiguous blocks")
    _cuda(blocks)
    world, rows, cols = blocks.shape
    out = torch.empty((rows, cols), dtype=torch.float32, device=blocks.device)
    st = _lib.load().flp_sum_blocks(blocks.data_ptr(), blocks.stride(0), world, rows, cols, out.data_ptr(), cols,
                                    _stream(blocks))
    _lib.check("flp_sum_blocks", st)
    return out


def fused_linear_logp_shard_backward(hidden: torch.Tensor, weight_shard: torch.Tensor, vocab_start: int,
                                     v_total: int, targets: torch.Tensor, lse: torch.Tensor, grad: torch.Tensor,
                                     dhidden: torch.Tensor, accumulate_dhidden: bool,
                                     ignore_index: int = IGNORE_INDEX, lse_lo: torch.Tensor | None = None,
                                     temperature: float = 1.0, active_mask: torch.Tensor | None = None,
                                     dweight_shard: torch.Tensor | None = None, accumulate_dweight: bool = False,
                                     workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One vocabulary shard's backward: writes (or, with accumulate_dhidden,
    adds) its term of dhidden [N, D] FP32 and returns its dweight rows
    [real_width, D] FP32.  lse / lse_lo are the merged forward's."""
    n, d, ld_h = _rows(hidden, "hidden")
    w, d_w, ld_w = _rows(weight_shard, "weight_shard")
    if hidden.dtype != torch.bfloat16 or weight_shard.dtype != torch.bfloat16:
        raise TypeError("hidden and weight_shard must be bfloat16")
    if d_w != d:
        raise ValueError(f"hidden has {d} columns but weight_shard has {d_w}")
    _vec(targets, "targets", n, torch.int64)
    _vec(lse, "lse", n, torch.float32)
    _vec(grad, "grad", n, torch.float32)
    if lse_lo is not None:
        _vec(lse_lo, "lse_lo", n, torch.float32)
    dev = hidden.device
    if dweight_shard is None:
        if accumulate_dweight:
            raise ValueError("accumulate_dweight needs a dweight_shard tensor to add to")
        dweight_shard = torch.empty((w, d), dtype=torch.float32, device=dev)
    if dhidden.dtype != torch.float32 or tuple(dhidden.shape) != (n, d):
        raise ValueError("dhidden must be float32 [N, D]")
    if dweight_shard.dtype != torch.float32 or tuple(dweight_shard.shape) != (w, d):
        raise ValueError("dweight_shard must be float32 [real_width, D]")
    _, _, ld_dh = _rows(dhidden, "dhidden")
    _, _, ld_dw = _rows(dweight_shard, "dweight_shard")
    _cuda(hidden, weight_shard, targets, lse, grad, dhidden, dweight_shard)
    mp = _mask(active_mask, n)
    if workspace is None and n > 0:
        workspace = torch.empty(fused_linear_logp_backward_workspace_size(d, w), dtype=torch.uint8, device=dev)
    wptr, wbytes = (None, 0) if workspace is None else (workspace.data_ptr(),
                                                        workspace.numel() * workspace.element_size())
    st = _lib.load().fused_linear_logp_shard_backward(
        hidden.data_ptr(), n, d, ld_h, weight_shard.data_ptr(), w, ld_w, int(vocab_start), int(v_total),
        targets.data_ptr(), int(ignore_index), mp, _inv_temperature(temperature), lse.data_ptr(), _opt_ptr(lse_lo),
        grad.data_ptr(), wptr, wbytes, dhidden.data_ptr(), ld_dh, int(bool(accumulate_dhidden)),
        dweight_shard.data_ptr(), ld_dw, int(bool(accumulate_dweight)), _stream(hidden))
    _lib.check("fused_linear_logp_shard_backward", st)
    return dweight_shard


class FusedLinearLogp(torch.autograd.Function):
    """logp = FusedLinearLogp.apply(hidden, weight, targets, ...): the fused
    LM head + logp; the logits never exist.  The backward recomputes dZ on the
    tensor cores from the saved LSE (O(N) state) and returns dhidden and
    dweight in the dtypes of hidden and weight."""

    @staticmethod
    def forward(ctx, hidden, weight, targets, ignore_index=IGNORE_INDEX, temperature=1.0,
                active_mask=None):
        logp, lse, lse_lo = fused_linear_logp_forward(hidden, weight, targets, ignore_index,
                                                      with_lse_lo=True, temperature=temperature,
                                                      active_mask=active_mask)
        ctx.save_for_backward(hidden, weight, targets, lse, lse_lo, active_mask)
        ctx.ignore_index = ignore_index
        ctx.temperature = temperature
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        hidden, weight, targets, lse, lse_lo, active_mask = ctx.saved_tensors
        g = grad_logp.to(torch.float32).contiguous()
        dh, dw = fused_linear_logp_backward(hidden, weight, targets, lse, g, ctx.ignore_index,
                                            lse_lo=lse_lo, temperature=ctx.temperature,
                                            active_mask=active_mask)
        dh = dh if hidden.dtype == torch.float32 else dh.to(hidden.dtype)
        dw = dw if weight.dtype == torch.float32 else dw.to(weight.dtype)
        return dh, dw, None, None, None, None


def fused_linear_logp(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                      ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                      active_mask: torch.Tensor | None = None) -> torch.Tensor:
    """Autograd-aware fused LM head + selected-token logp (FP32 [N]) of
    hidden [N, D] @ weight[V, D].T, both BF16."""
    return FusedLinearLogp.apply(hidden, weight, targets, ignore_index, temperature, active_mask)


def flp_device_error(device: int | torch.device = 0) -> int:
    """Read and clear the library's sticky device error word (0 = healthy;
    1 = a bounded wait of a kernel ran out).  Synchronises with the device."""
    import ctypes

    dev = torch.device(device).index if not isinstance(device, int) else device
    code = ctypes.c_int(-1)
    _lib.check("flp_device_error", _lib.load().flp_device_error(int(dev or 0), ctypes.byref(code)))
    return code.value


def flp_selftest_wait_timeout(device: int = 0, limit_cycles: int = 200000) -> int:
    """Run the bounded-wait self-test (a wait nothing completes); returns 1 if
    the wait gave up as it must."""
    import ctypes

    out = ctypes.c_int(-1)
    _lib.check("flp_selftest_wait_timeout",
               _lib.load().flp_selftest_wait_timeout(int(device), int(limit_cycles), ctypes.byref(out)))
    return out.value


def flp_selftest_ex2_bias(device: int = 0):
    """(measured mean relative error of the hardware exp2 approximation, the
    compiled-in compensation); the compensation is right when they cancel."""
    import ctypes

    m, c = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _lib.check("flp_selftest_ex2_bias",
               _lib.load().flp_selftest_ex2_bias(int(device), ctypes.byref(m), ctypes.byref(c)))
    return m.value, c.value
