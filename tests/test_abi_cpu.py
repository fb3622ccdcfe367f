"""The C ABI library builds, loads and exports every symbol its header
declares, and rejects bad arguments on the host before touching any device.
These run without a GPU: every call here either returns before its first CUDA
runtime call or fails that call's pointer check."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import selected_token_logprob_gb300 as flp
from selected_token_logprob_gb300 import _lib
from selected_token_logprob_gb300 import build as flp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EINVAL, EUNSUP = _lib.FLP_EINVAL, _lib.FLP_EUNSUPPORTED


@pytest.fixture(scope="module")
def lib():
    flp_build.build()
    return _lib.load()


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(inc, fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                            src, flags=re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"fused_logp_forward", "fused_logp_backward", "logp_shard_partials",
            "logp_merge_partials", "flp_last_error", "flp_tile_width"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


def test_version_and_tile_width(lib):
    assert b"sm_103a" in lib.flp_version()
    for v, w in [(151936, 9496), (1024, 64), (1, 8), (0, 0), (255, 16), (1031, 72), (128, 8),
                 (129, 16), (2**40, 2**40 // 16)]:
        assert lib.flp_tile_width(v) == w, (v, w)
    assert flp.flp_tile_width(151936) == 9496


def test_empty_input_is_ok_without_device(lib):
    assert lib.fused_logp_forward(None, 0, 10, 10, None, -100, None, None, None, None) == 0
    assert lib.flp_last_error() == b""
    assert lib.fused_logp_backward(None, 0, 10, 10, None, -100, None, None, None, None, 10,
                                   None) == 0
    assert lib.logp_merge_partials(None, None, None, None, -100, 0, 10, None, None, None,
                                   None) == 0


def test_forward_argument_errors(lib):
    buf = (ctypes.c_char * 64)()
    p = ctypes.addressof(buf)
    cases = [
        dict(n=-1, v=10, ld=10),
        dict(n=4, v=0, ld=10),
        dict(n=4, v=10, ld=9),
        dict(n=2**62, v=2**20, ld=2**20),   # extent overflows int64
    ]
    for c in cases:
        st = lib.fused_logp_forward(p, c["n"], c["v"], c["ld"], p, -100, p, p, None, None)
        assert st == EINVAL, c
        assert lib.flp_last_error()
    # null pointers
    assert lib.fused_logp_forward(None, 4, 10, 10, p, -100, p, p, None, None) == EINVAL
    assert b"logits" in lib.flp_last_error()
    # host memory is not accepted as device memory
    assert lib.fused_logp_forward(p, 4, 10, 10, p, -100, p, p, None, None) == EINVAL


def test_backward_argument_errors(lib):
    buf = (ctypes.c_char * 64)()
    p = ctypes.addressof(buf)
    assert lib.fused_logp_backward(p, 4, 10, 10, p, -100, p, None, p, p, 9, None) == EINVAL  # ld_out < v
    assert lib.fused_logp_backward(p, -2, 10, 10, p, -100, p, None, p, p, 10, None) == EINVAL
    assert lib.fused_logp_backward(p, 4, 10, 10, p, -100, None, None, p, p, 10, None) == EINVAL


def test_shard_gate(lib):
    buf = (ctypes.c_char * 64)()
    p = ctypes.addressof(buf)
    V, W = 151936, 9496
    # bounds off the tile grid are refused before any device work
    assert lib.logp_shard_partials(p, 8, 76032, 100, 75968, V, p, p, p, p, None) == EUNSUP
    assert lib.logp_shard_partials(p, 8, 76032, 0, 75000, V, p, p, p, p, None) == EUNSUP
    assert b"tile width" in lib.flp_last_error()
    # outside the vocabulary / bad widths
    assert lib.logp_shard_partials(p, 8, 76032, 2 * W, V, V, p, p, p, p, None) == EINVAL
    assert lib.logp_shard_partials(p, 8, 10, 0, 9496, V, p, p, p, p, None) == EINVAL
    assert lib.logp_shard_partials(p, 8, 10, 0, 0, V, p, p, p, p, None) == EINVAL
    # a last shard may be ragged: passes the gate, then fails on host memory
    assert lib.logp_shard_partials(p, 8, 76032, 15 * W, V - 15 * W, V, p, p, p, p, None) == EINVAL
    assert b"device memory" in lib.flp_last_error() or b"cudaPointer" in lib.flp_last_error()


def test_ex_entry_points_reject_bad_dtype_and_temperature(lib):
    buf = (ctypes.c_char * 64)()
    p = ctypes.addressof(buf)
    assert lib.fused_logp_forward_ex(p, 3, 4, 10, 10, p, -100, None, 1.0, p, p, None, None) == EINVAL
    assert b"dtype" in lib.flp_last_error()
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.fused_logp_forward_ex(p, 0, 4, 10, 10, p, -100, None, bad, p, p, None, None) == EINVAL
        assert lib.fused_logp_backward_ex(p, 0, 4, 10, 10, p, -100, None, bad, p, None, p, p, 10,
                                          None) == EINVAL
        assert lib.logp_merge_partials_ex(p, p, p, p, -100, None, 4, 10, bad, p, p, None, None) == EINVAL
    assert lib.logp_shard_partials_ex(p, 7, 4, 10, 0, 10, 10, 1.0, p, p, p, p, None) == EINVAL
    # FP32 shard bounds are checked on the same tile grid
    assert lib.logp_shard_partials_ex(p, 2, 8, 76032, 100, 75968, 151936, 1.0, p, p, p, p,
                                      None) == EUNSUP


def test_device_entry_points_reject_null_outputs(lib):
    assert lib.flp_device_error(0, None) == EINVAL
    assert lib.flp_selftest_wait_timeout(0, 1000, None) == EINVAL
    import ctypes as C
    out = C.c_int(0)
    assert lib.flp_selftest_wait_timeout(0, -1, C.byref(out)) == EINVAL
    assert lib.flp_selftest_wait_timeout(0, 10**9, C.byref(out)) == EINVAL


def test_python_binding_checks_before_calling():
    x = torch.zeros((4, 10), dtype=torch.float64)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(TypeError):
        flp.fused_logp_forward(x, y)
    xb = x.to(torch.bfloat16)
    with pytest.raises(ValueError):
        flp.fused_logp_forward(xb, y, temperature=0.0)
    with pytest.raises(ValueError):
        flp.fused_logp_forward(xb, y, temperature=float("inf"))
    with pytest.raises(TypeError):
        flp.fused_logp_forward(xb, y.to(torch.int32))
    with pytest.raises(ValueError):
        flp.fused_logp_forward(xb, torch.zeros(3, dtype=torch.int64))
    with pytest.raises(ValueError):
        flp.fused_logp_forward(xb.t(), torch.zeros(10, dtype=torch.int64))
    with pytest.raises(ValueError):
        flp.fused_logp_forward(xb, y)  # CPU tensors are refused, no CPU fallback
    lse = torch.zeros(4)
    with pytest.raises(TypeError):
        flp.fused_logp_backward(xb, y, lse, torch.zeros(4, dtype=torch.float64))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(flp_build, "LIB", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load()


def test_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "selected_token_logprob_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in src.lower(), fn


def test_linear_logp_host_checks(lib):
    b = ctypes.c_int64(0)
    assert lib.fused_linear_logp_workspace_size(2048, 151936, ctypes.byref(b)) == 0
    nvt = -(-151936 // 256)
    assert b.value == -(-(2 * nvt * 2048 + 2048) * 4 // 256) * 256
    assert lib.fused_linear_logp_workspace_size(-1, 10, ctypes.byref(b)) == EINVAL
    assert lib.fused_linear_logp_workspace_size(4, 0, ctypes.byref(b)) == EINVAL
    assert lib.fused_linear_logp_workspace_size(4, 10, None) == EINVAL
    assert flp.fused_linear_logp_workspace_size(0, 7) == 0

    def call(n=256, d=512, ld_h=512, ptr_h=1 << 20, v=5000, ld_w=512, ptr_w=1 << 21, s=1.0,
             ws=1 << 22, ws_bytes=1 << 30):
        return lib.fused_linear_logp_forward(ptr_h, n, d, ld_h, ptr_w, v, ld_w, 1 << 23, -100, None, s,
                                             ws, ws_bytes, 1 << 24, 1 << 25, None, None)

    assert call(n=0) == 0                                   # empty: no device touched
    assert call(n=-1) == EINVAL
    assert call(d=0) == EINVAL
    assert call(v=0) == EINVAL
    assert call(ld_h=500) == EINVAL and b"ld_h" in lib.flp_last_error()
    assert call(ld_w=256) == EINVAL
    assert call(s=0.0) == EINVAL
    assert call(s=float("inf")) == EINVAL
    assert call(ld_h=516) == EUNSUP                         # row stride not 16-byte
    assert call(ptr_h=(1 << 20) + 8) == EUNSUP              # base not 16-byte aligned
    assert call(ptr_w=(1 << 21) + 2) == EUNSUP
    assert call(n=1 << 31) == EUNSUP
    assert call(ws_bytes=1000) == EINVAL and b"workspace" in lib.flp_last_error()
    assert call(ws=(1 << 22) + 4) == EINVAL
    # pointer checks come last: host pointers are not device memory
    assert call() == EINVAL


def test_linear_logp_binding_checks_before_calling():
    h = torch.zeros(4, 64, dtype=torch.bfloat16)
    w = torch.zeros(10, 64, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(TypeError):
        flp.fused_linear_logp_forward(h.float(), w, y)
    with pytest.raises(ValueError):
        flp.fused_linear_logp_forward(h, w[:, :32], y)
    with pytest.raises(ValueError):
        flp.fused_linear_logp_forward(h, w, y, temperature=0.0)
    with pytest.raises(ValueError):
        flp.fused_linear_logp_forward(h, w, y)               # CPU tensors


def test_linear_logp_noalloc_host_checks(lib):
    """The no-allocation variant refuses, before touching any device, a call
    whose scratch would exceed its fixed 16 MiB, and names the sizes."""
    def call(n, v=151936, d=4096):
        return lib.fused_linear_logp_forward_noalloc(1 << 20, n, d, d, 1 << 21, v, d, 1 << 22, -100, None,
                                                     1.0, 1 << 23, 1 << 24, None, None)

    assert call(0) == 0
    assert call(-1) == EINVAL
    assert call(3528) == EUNSUP
    msg = lib.flp_last_error()
    assert b"3528 rows" in msg and b"16777216" in msg
    assert call(3527) == EINVAL          # within the limit: reaches the pointer checks
    assert b"hidden" in lib.flp_last_error()


def test_linear_backward_host_checks(lib):
    b = ctypes.c_int64(0)
    assert lib.fused_linear_logp_backward_workspace_size(4096, 151936, ctypes.byref(b)) == 0
    assert b.value >= 2048 * 151936 * 2 + 2048 * 4096 * 4
    assert lib.fused_linear_logp_backward_workspace_size(0, 10, ctypes.byref(b)) == EINVAL

    def call(n=16, d=64, ld_h=64, v=100, ld_w=64, ws=1 << 20, ws_bytes=1 << 40, ld_dh=64, ld_dw=64, s=1.0):
        return lib.fused_linear_logp_backward(1 << 20, n, d, ld_h, 1 << 21, v, ld_w, 1 << 22, -100, None, s,
                                              1 << 23, None, 1 << 24, ws, ws_bytes, 1 << 25, ld_dh, 1 << 26,
                                              ld_dw, 0, None)

    assert call(n=-1) == EINVAL
    assert call(ld_dh=32) == EINVAL and call(ld_dw=8) == EINVAL
    assert call(ld_h=68) == EUNSUP
    assert call(ws_bytes=100) == EINVAL
    assert call(ws=(1 << 20) + 16) == EINVAL          # not 256-byte aligned
    assert call(s=-1.0) == EINVAL
    assert call() == EINVAL                            # host pointers are not device memory


def test_linear_shard_host_checks(lib):
    def call(n=16, w=512, start=256, v_total=2000, ld=64):
        return lib.fused_linear_logp_shard_partials(1 << 20, n, 64, ld, 1 << 21, w, ld, start, v_total,
                                                    1 << 22, 1.0, 1 << 23, 1 << 30, None)

    assert call(start=100) == EUNSUP and b"multiple" in lib.flp_last_error()
    assert call(start=1792) == EINVAL                 # [1792, 2304) is not inside [0, 2000)
    assert call(start=-256) == EINVAL
    assert call(n=0) == 0
    assert call() == EINVAL                           # host pointers are not device memory
    assert lib.fused_linear_logp_merge(None, 0, 0, 10, None, -100, None, 1.0, None, None, None, None) == 0
    assert lib.fused_linear_logp_merge(1 << 20, 10, 16, 2000, 1 << 21, -100, None, 1.0, 1 << 22, 1 << 23,
                                       None, None) == EINVAL   # workspace too small


def test_grpo_binding_rejects_an_unknown_mode():
    import selected_token_logprob_gb300 as flp

    t = torch.zeros(4)
    with pytest.raises(ValueError, match="mode must be one of"):
        flp.logp_grpo_loss(t, t, t, mode="seq_sum_token_mean")


def test_grpo_host_checks(lib):
    b = ctypes.c_int64(0)
    # 32 bytes of count and ticket, two 8-byte sums per CTA of the token pass
    # (608), 8 bytes per CTA of the sequences' counts (1024) and per count
    # range (1024), and with S sequences 8 per sequence and 4 per 16 tokens;
    # rounded up to 256; without sequences n does not enter:
    # 32 + 9728 + 8192 + 8192 = 26144 -> 26368;  + 8*100 + 4*2048 = 35136 -> 35328
    assert lib.logp_grpo_loss_workspace_size(32768, 0, ctypes.byref(b)) == 0 and b.value == 26368
    assert lib.logp_grpo_loss_workspace_size(32768, 100, ctypes.byref(b)) == 0 and b.value == 35328
    assert lib.logp_grpo_loss_workspace_size(0, 0, ctypes.byref(b)) == 0 and b.value == 26368
    assert lib.logp_grpo_loss_workspace_size(1 << 31, 0, ctypes.byref(b)) == 0 and b.value == 26368
    assert lib.logp_grpo_loss_workspace_size(-1, 0, ctypes.byref(b)) == EINVAL

    def call(mode=0, ws=1 << 20, ws_bytes=1 << 20, n=1000, eps_lo=0.2):
        return lib.logp_grpo_loss(1 << 21, 1 << 22, None, 1 << 23, None, None, 0, n, mode, eps_lo, 0.2, 0.0,
                                  0.0, ws, ws_bytes, 1 << 24, 1 << 25, None, None)

    assert call(mode=3) == EINVAL and b"mode" in lib.flp_last_error()
    assert call(eps_lo=1.5) == EINVAL
    assert call(ws_bytes=8) == EINVAL and b"workspace" in lib.flp_last_error()
    assert call(ws=(1 << 20) + 8) == EINVAL
    assert call() == EINVAL                            # host pointers are not device memory

    # the two-part form checks the same things before any device access
    def counts(mode=0, ws=1 << 20, ws_bytes=1 << 20, n=1000, normalizer=0.0):
        return lib.logp_grpo_loss_counts(None, None, 0, n, mode, normalizer, ws, ws_bytes, None)

    assert counts(mode=-1) == EINVAL and b"mode" in lib.flp_last_error()
    assert counts(n=-5) == EINVAL
    assert counts(normalizer=-1.0) == EINVAL
    assert counts(ws_bytes=64) == EINVAL and b"workspace" in lib.flp_last_error()
    assert counts(ws=(1 << 20) + 4) == EINVAL
    assert counts() == EINVAL                          # a host address is not device memory
    assert lib.logp_grpo_loss_counted(1 << 21, 1 << 22, None, 1 << 23, None, None, 0, 1000, 2, 0.2, 0.2, 0.0,
                                      0.0, 1 << 20, 1 << 20, 1 << 24, 1 << 25, None, None) == EINVAL


def test_gathered_merge_validates_the_rank_layout_on_the_host(lib):
    """The tile -> rank table of a vocabulary-parallel merge is checked before
    any device access: shards off the tile grid, a gap, an overlap, too many
    ranks, a short rank stride."""
    v, w = 151936, 9496
    I64 = ctypes.c_int64

    def call(starts, widths, n=4, stride=None, world=None):
        k = len(starts)
        a = (I64 * max(1, k))(*starts)
        b = (I64 * max(1, k))(*widths)
        return lib.logp_merge_gathered_partials_ex(None, 33 * n if stride is None else stride,
                                                   k if world is None else world, a, b, None, -100, None, n, v,
                                                   1.0, None, None, None, None)

    assert call([0, 8 * w + 8], [8 * w + 8, v - 8 * w - 8]) == EUNSUP
    assert b"tile grid" in lib.flp_last_error()
    assert call([0, 9 * w], [8 * w, v - 9 * w]) == EINVAL
    assert b"held by no rank" in lib.flp_last_error()
    assert call([0, 7 * w], [8 * w, v - 7 * w]) == EINVAL
    assert b"held by rank 0 and rank 1" in lib.flp_last_error()
    assert call([k * w for k in range(16)] + [0], [w] * 17) == EINVAL
    assert call([0, 8 * w], [8 * w, v - 8 * w], stride=33 * 4 - 1) == EINVAL
    assert b"rank_stride" in lib.flp_last_error()
    # a correct layout with n == 0 returns before touching the device
    assert call([0, 8 * w], [8 * w, v - 8 * w], n=0) == 0


def test_shard_backward_validates_the_shard_on_the_host(lib):
    st = lib.logp_shard_backward(None, 4, 100, 151900, 100, 151936, None, -100, None, None, None, None, 100,
                                 None)
    assert st == EINVAL and b"inside the vocabulary" in lib.flp_last_error()
    assert lib.logp_shard_backward(None, 0, 100, 0, 100, 151936, None, -100, None, None, None, None, 100,
                                   None) == 0


def test_vocab_parallel_lm_head_host_checks(lib):
    """The gathered LM-head merge and the ordered block sum validate the rank
    layout and the extents on the host, before any device access."""
    I64 = ctypes.c_int64
    v, n = 20000, 16
    block = (2 * ((v + 255) // 256) + 1) * n

    def merge(starts, widths, stride=block, world=None):
        k = len(starts)
        a = (I64 * max(1, k))(*starts)
        b = (I64 * max(1, k))(*widths)
        return lib.fused_linear_logp_merge_gathered(None, stride, k if world is None else world, a, b, n, v, None,
                                                    -100, None, 1.0, None, None, None, None)

    assert merge([0, 10240], [10240, 9760], world=0) == EINVAL
    assert merge([0, 10240], [10240, 9760], world=17) == EINVAL
    assert merge([0, 10240], [10240, 9760], stride=block - 1) == EINVAL and b"rank_stride" in lib.flp_last_error()
    assert merge([0, 10000], [10000, 10000]) == EUNSUP and b"tile grid" in lib.flp_last_error()
    assert merge([0, 10496], [10240, 9504]) == EINVAL and b"held by no rank" in lib.flp_last_error()
    assert merge([0, 9984], [10240, 10016]) == EINVAL and b"held by two ranks" in lib.flp_last_error()
    assert merge([0, 10240], [10240, 9800]) == EINVAL and b"not inside" in lib.flp_last_error()
    assert merge([0, 10240], [10240, 9760]) == EINVAL              # the layout is fine; host pointers are not
    assert lib.flp_sum_blocks(None, 10, 0, 2, 5, None, 5, None) == EINVAL
    assert lib.flp_sum_blocks(None, 10, 2, 2, 5, None, 4, None) == EINVAL and b"ld_out" in lib.flp_last_error()
    assert lib.flp_sum_blocks(None, 9, 2, 2, 5, None, 5, None) == EINVAL and b"block_stride" in lib.flp_last_error()
    assert lib.flp_sum_blocks(None, 10, 2, 0, 5, None, 5, None) == 0   # nothing to sum
