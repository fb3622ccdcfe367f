"""Seeded synthetic inputs for the selected-token log-probability path.

This module only draws random inputs; it holds none of the method's
arithmetic.  It serves both the FP64 oracle (tests, CPU baseline) and the GPU
path (tests, bench, smoke), so that both see the same bytes.

The workloads stand in for the RL-Kernel pages' benchmark (PR #495, "Benchmark
script": randn BF16 logits, randint targets, V = 151936, the Qwen3 vocabulary
named in issue #241 Background).  No dataset or trained weights are used.

Recipe (all draws in FP32, then ONE round-to-nearest-even cast to BF16):
  tiny     N=64,    V=1024,   x ~ N(0,1); 10% of rows (floor) ignore_index;
           g ~ N(0,1).
  mid      N=2048,  V=151936, x ~ N(0,2^2) plus +8 at one uniform column per
           row; 5% ignore; g ~ N(0,1).
  long     N=32768, V=151936, x as mid; 5% ignore; g = +-1/N random sign.
  sweep    V=151936, x ~ N(0,3^2); probe and filler rows from separate
           streams.
  sharded  N=8192,  V=151936, x ~ N(0,2^2); targets uniform; no ignore rows.
  linear   fused LM head: hidden H [N, D] ~ N(0,1), weight W [V, D] ~
           N(0, (2/sqrt(D))^2) (so the logits H W^T have standard deviation
           about 2, like the logits workloads), both drawn like the logits
           (FP32, one cast to BF16) from their own seeds; targets as above
           with 5% ignore.  Long: N=32768, D=4096 (a Qwen3-8B-sized hidden
           state; the pages name no hidden size), V=151936.
Targets are uniform in [0, V); exactly floor(p*N) rows, chosen by a seeded
permutation, get the ignore index -100.  Each random stream has its own
generator seeded from (seed, stream id), so changing one never shifts another.
Logits are generated in row blocks to bound the FP32 temporaries.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

IGNORE_INDEX = -100
QWEN3_VOCAB = 151936


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    v: int
    sigma: float
    spike: float          # added at one uniform column per row (0: none)
    ignore_frac: float
    grad: str             # "normal" | "sign_over_n" | "none"
    seed: int = 0


WORKLOADS = {
    "tiny": Workload("tiny", 64, 1024, 1.0, 0.0, 0.10, "normal"),
    "mid": Workload("mid", 2048, QWEN3_VOCAB, 2.0, 8.0, 0.05, "normal"),
    "long": Workload("long", 32768, QWEN3_VOCAB, 2.0, 8.0, 0.05, "sign_over_n"),
    "sweep": Workload("sweep", 2048, QWEN3_VOCAB, 3.0, 0.0, 0.0, "normal"),
    "sharded": Workload("sharded", 8192, QWEN3_VOCAB, 2.0, 0.0, 0.0, "none"),
}

# stream ids
_S_LOGITS, _S_SPIKE, _S_TARGET, _S_IGNORE, _S_GRAD = 1, 2, 3, 4, 5


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + stream * 7919 + 17)
    return g


def logits(n: int, v: int, sigma: float, spike: float, seed: int, device="cpu",
           ld: int | None = None, block_rows: int = 1024,
           dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """[n, ld] (ld >= v; padding columns are 0) ~ N(0, sigma^2) + spike, drawn in
    FP32 and cast once (round to nearest even) to `dtype`."""
    ld = v if ld is None else ld
    out = torch.zeros((n, ld), dtype=dtype, device=device)
    gl = _gen(device, seed, _S_LOGITS)
    gs = _gen(device, seed, _S_SPIKE)
    for r0 in range(0, n, block_rows):
        r1 = min(n, r0 + block_rows)
        blk = torch.randn((r1 - r0, v), generator=gl, device=device, dtype=torch.float32)
        if sigma != 1.0:
            blk.mul_(sigma)
        if spike:
            cols = torch.randint(0, v, (r1 - r0,), generator=gs, device=device)
            blk[torch.arange(r1 - r0, device=device), cols] += spike
        out[r0:r1, :v] = blk.to(dtype)
        del blk
    return out


def targets(n: int, v: int, ignore_frac: float, seed: int, device="cpu") -> torch.Tensor:
    y = torch.randint(0, v, (n,), generator=_gen(device, seed, _S_TARGET), device=device,
                      dtype=torch.int64)
    k = int(ignore_frac * n)
    if k:
        perm = torch.randperm(n, generator=_gen(device, seed, _S_IGNORE), device=device)
        y[perm[:k]] = IGNORE_INDEX
    return y


def grads(n: int, kind: str, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, seed, _S_GRAD)
    if kind == "normal":
        return torch.randn((n,), generator=g, device=device, dtype=torch.float32)
    if kind == "sign_over_n":
        sign = torch.randint(0, 2, (n,), generator=g, device=device).to(torch.float32) * 2 - 1
        return sign * (1.0 / n)
    if kind == "none":
        return torch.zeros((n,), dtype=torch.float32, device=device)
    raise ValueError(kind)


def make(name_or_wl, device="cpu", n: int | None = None, seed: int | None = None,
         ld: int | None = None, dtype: torch.dtype = torch.bfloat16):
    """(logits [n, ld] in `dtype`, targets int64 [n], grad fp32 [n]) of a workload."""
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    n = wl.n if n is None else n
    seed = wl.seed if seed is None else seed
    x = logits(n, wl.v, wl.sigma, wl.spike, seed, device=device, ld=ld, dtype=dtype)
    y = targets(n, wl.v, wl.ignore_frac, seed, device=device)
    g = grads(n, wl.grad, seed, device=device)
    return x, y, g


LINEAR_LONG = (32768, 4096, QWEN3_VOCAB)   # (N, D, V) of the fused LM-head workload


def linear(n: int, d: int, v: int, seed: int = 0, device="cpu", ld_h: int | None = None,
           ld_w: int | None = None, ignore_frac: float = 0.05):
    """(hidden [n, ld_h] BF16, weight [v, ld_w] BF16, targets int64 [n]) of the
    fused LM-head workload; padding columns are 0."""
    base = 1_000 + 3 * int(seed)
    h = logits(n, d, 1.0, 0.0, base, device=device, ld=ld_h)
    w = logits(v, d, 2.0 / d ** 0.5, 0.0, base + 1, device=device, ld=ld_w, block_rows=4096)
    y = targets(n, v, ignore_frac, base + 2, device=device)
    return h, w, y


def sweep_rows(count: int, v: int, sigma: float, seed: int, stream: int, device="cpu"):
    """Rows for the batch-invariance sweep: (x [count, v], y [count], g [count]).

    stream 0 = probe rows, stream 1 = filler rows; each (seed, stream) pair is
    its own generator family."""
    base = seed * 2 + stream + 1000
    x = logits(count, v, sigma, 0.0, base, device=device)
    y = targets(count, v, 0.0, base, device=device)
    g = grads(count, "normal", base, device=device)
    return x, y, g


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a BF16 (or FP16) tensor (for the oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def host_array(t: torch.Tensor):
    """(numpy array, dtype name) of a logits/gradient tensor for the oracle:
    uint16 bit patterns for bf16/f16, float32 values for f32."""
    if t.dtype == torch.float32:
        return t.detach().cpu().contiguous().numpy(), "f32"
    name = {torch.bfloat16: "bf16", torch.float16: "f16"}[t.dtype]
    return bf16_bits(t), name
