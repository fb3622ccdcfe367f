"""The no-allocation variant of the fused LM head + logp forward.

Some callers cannot allocate device memory (a plugin handed only its input
and output buffers, code under an application memory pool that forbids
direct cudaMalloc, a loop where cudaMalloc/cudaFree would synchronise the
device).  fused_linear_logp_forward_noalloc serves them from a fixed static
scratch array instead of a caller workspace.  This file checks, through the
C ABI, that two calls in a row (different shapes, the second reusing the
scratch the first left behind) give what the workspace entry point gives,
and that a call beyond the fixed size is refused.  It is named so that
pytest collects it last."""

import numpy as np
import pytest
import torch

import selected_token_logprob_gb300 as flp
from selected_token_logprob_gb300 import _lib
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-4   # the logp / LSE tolerance of the other GPU tests


def _call_noalloc(lib, h, w, y, outs, temperature, mask=None):
    n, d = h.shape
    v = w.shape[0]
    logp, lse, lo = outs
    return lib.fused_linear_logp_forward_noalloc(
        h.data_ptr(), n, d, h.stride(0), w.data_ptr(), v, w.stride(0), y.data_ptr(), -100,
        None if mask is None else mask.data_ptr(), float(np.float32(1.0 / temperature)),
        logp.data_ptr(), lse.data_ptr(), lo.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = _lib.load(build_if_missing=True)
    cases = [(2048, 1024, workloads.QWEN3_VOCAB, 0.7, 11), (333, 520, 5000, 1.0, 12)]
    for n, d, v, temperature, seed in cases:
        h, w, y = workloads.linear(n, d, v, seed=seed, device=DEV)
        mask = (torch.arange(n, device=DEV) % 9 != 4).to(torch.uint8)
        outs = [torch.full((n,), float("nan"), device=DEV) for _ in range(3)]
        st = _call_noalloc(lib, h, w, y, outs, temperature, mask)
        assert st == 0, lib.flp_last_error()
        ref = flp.fused_linear_logp_forward(h, w, y, with_lse_lo=True, temperature=temperature,
                                            active_mask=mask)
        torch.cuda.synchronize()
        for got, want in zip(outs, ref):
            assert torch.isfinite(got).all()
            assert torch.max(torch.abs(got - want)).item() <= TOL
            assert torch.equal(got.view(torch.int32), want.view(torch.int32))   # same kernel, same bits
    assert flp.flp_device_error(0) == 0


def test_noalloc_refuses_more_than_its_scratch():
    lib = _lib.load(build_if_missing=True)
    n, d, v = 3528, 64, workloads.QWEN3_VOCAB
    h = torch.zeros((n, d), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((v, d), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros(n, dtype=torch.int64, device=DEV)
    outs = [torch.empty(n, device=DEV) for _ in range(3)]
    assert _call_noalloc(lib, h, w, y, outs, 1.0) == _lib.FLP_EUNSUPPORTED
    assert b"16777216" in lib.flp_last_error()
    with pytest.raises(flp.FusedLogpError, match="scratch"):
        flp.fused_linear_logp_forward_noalloc(h, w, y, outs[0], outs[1])


def test_noalloc_largest_accepted_call_matches_workspace_entry_point():
    """3527 rows at V = 151936 need 16,774,656 of the array's 16,777,216
    bytes, so the last rows' partials sit at its end; two calls in a row give
    the workspace entry point's bits."""
    lib = _lib.load(build_if_missing=True)
    n, d, v = 3527, 256, workloads.QWEN3_VOCAB
    assert flp.fused_linear_logp_workspace_size(n, v) <= 16 << 20 < flp.fused_linear_logp_workspace_size(n + 1, v)
    h, w, y = workloads.linear(n, d, v, seed=13, device=DEV)
    for _ in range(2):
        outs = [torch.full((n,), float("nan"), device=DEV) for _ in range(3)]
        assert _call_noalloc(lib, h, w, y, outs, 1.0) == 0, lib.flp_last_error()
        ref = flp.fused_linear_logp_forward(h, w, y, with_lse_lo=True)
        torch.cuda.synchronize()
        for got, want in zip(outs, ref):
            assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    assert flp.flp_device_error(0) == 0


def test_noalloc_calls_leave_device_memory_unchanged():
    """After one warm-up call per shape (which loads the kernels), further
    calls of several shapes change neither the device's free memory nor
    torch's allocated bytes."""
    lib = _lib.load(build_if_missing=True)
    shapes = [(1000, 512, workloads.QWEN3_VOCAB), (77, 64, 3000), (2048, 128, 20000)]
    cases = []
    for k, (n, d, v) in enumerate(shapes):
        h, w, y = workloads.linear(n, d, v, seed=40 + k, device=DEV)
        outs = [torch.empty(n, device=DEV) for _ in range(3)]
        cases.append((h, w, y, outs))
    for h, w, y, outs in cases:
        assert _call_noalloc(lib, h, w, y, outs, 1.0) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        for h, w, y, outs in cases:
            assert _call_noalloc(lib, h, w, y, outs, 0.8) == 0
            flp.fused_linear_logp_forward_noalloc(h, w, y, outs[0], outs[1], lse_lo=outs[2])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
