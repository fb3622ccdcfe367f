"""FP64 CPU oracle for the selected-token log-probability path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``selected_token_logprob_gb300``) never imports it, and the two share no code:
the oracle is plain C in IEEE double (``logp_oracle.c``), built with gcc, plus
this ctypes loader that marshals numpy arrays.

What each function computes, and the passage it follows, is stated in the C
file.  BF16 arrays are passed as ``numpy.uint16`` bit patterns.

Parity status: every oracle function is pinned by CPU tests against closed
forms, brute force, finite differences or a library routine (see
``tests/test_oracle_pins.py``); none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "logp_oracle.c")
_LIB = os.path.join(_HERE, "liblogp_oracle.so")
_lock = threading.Lock()
_lib = None

_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_U16P = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_I64P = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction) if stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_f16.restype = ctypes.c_uint16
        lib.oracle_round_f16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16_array.argtypes = [_F64P, _U16P, _I64]
        lib.oracle_bf16_to_double_array.argtypes = [_U16P, _F64P, _I64]
        lib.oracle_round_f16_array.argtypes = [_F64P, _U16P, _I64]
        lib.oracle_f16_to_double_array.argtypes = [_U16P, _F64P, _I64]
        V = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_forward.argtypes = [V, I, _I64, _I64, _I64, _I64P, _I64, V, D, _F64P, _F64P]
        lib.oracle_backward.argtypes = [V, I, _I64, _I64, _I64, _I64P, _I64, V, D, _F32P, _F64P, _I64]
        lib.oracle_backward_compare.argtypes = [V, I, _I64, _I64, _I64, _I64P, _I64, V, D, _F32P,
                                                V, I, _I64, _F64P, _I64P]
        lib.oracle_range_partials.argtypes = [V, I, _I64, _I64, _I64, _I64, _I64, D, _F64P, _F64P]
        lib.oracle_merge_partials.argtypes = [_F64P, _F64P, _I64, _I64, _F64P]
        lib.oracle_grpo_loss.argtypes = [_F64P, _F64P, V, _F64P, V, V, _I64, _I64, I, D, D, D, D,
                                         _F64P, _F64P]
        lib.oracle_linear_logp.argtypes = [_U16P, _I64, _U16P, _I64, _I64, _I64, _I64, _I64P, _I64,
                                           V, D, _F64P, _F64P, V]
        lib.oracle_linear_backward.argtypes = [_U16P, _I64, _U16P, _I64, _I64, _I64, _I64, _I64P, _I64,
                                               V, D, _F32P, I, V, _F64P, _F64P]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


DTYPES = {"bf16": 0, "f16": 1, "f32": 2}


def _logits(x, dtype: str | None):
    """Contiguous array and dtype code: uint16 bits for bf16/f16, float32 for f32."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        if dtype not in (None, "f32"):
            raise TypeError("float32 logits are dtype f32")
        return x, DTYPES["f32"]
    if x.dtype != np.uint16:
        raise TypeError("logits are uint16 bit patterns (bf16/f16) or float32")
    dtype = dtype or "bf16"
    if dtype not in ("bf16", "f16"):
        raise TypeError("uint16 logits are bf16 or f16 bit patterns")
    return x, DTYPES[dtype]


def _mask(mask, n):
    if mask is None:
        return None, None
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    if m.shape != (n,):
        raise ValueError("mask must have shape [n]")
    return m, m.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("BF16 arrays are passed as uint16 bit patterns")
    return a


def _shape(x: np.ndarray, v: int | None):
    """(n, v, ld) of a 2-D BF16 bit array whose first v columns are the row."""
    if x.ndim != 2:
        raise ValueError("logits must be 2-D")
    n, ld = x.shape
    return n, (ld if v is None else v), ld


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def round_bf16(d) -> np.ndarray:
    """Nearest BF16 (ties to even) of each double, as uint16 bit patterns."""
    d = np.asarray(d, dtype=np.float64)
    flat = np.ascontiguousarray(d.reshape(-1))
    out = np.empty(flat.shape, dtype=np.uint16)
    _load().oracle_round_bf16_array(flat, out, flat.size)
    return out.reshape(d.shape)


def bf16_to_f64(b) -> np.ndarray:
    b = np.asarray(b)
    flat = _u16(b.reshape(-1))
    out = np.empty(flat.shape, dtype=np.float64)
    _load().oracle_bf16_to_double_array(flat, out, flat.size)
    return out.reshape(b.shape)


def round_f16(d) -> np.ndarray:
    """Nearest binary16 (ties to even) of each double, as uint16 bit patterns."""
    d = np.asarray(d, dtype=np.float64)
    flat = np.ascontiguousarray(d.reshape(-1))
    out = np.empty(flat.shape, dtype=np.uint16)
    _load().oracle_round_f16_array(flat, out, flat.size)
    return out.reshape(d.shape)


def f16_to_f64(b) -> np.ndarray:
    b = np.asarray(b)
    flat = _u16(b.reshape(-1))
    out = np.empty(flat.shape, dtype=np.float64)
    _load().oracle_f16_to_double_array(flat, out, flat.size)
    return out.reshape(b.shape)


def forward(x, y, ignore_index: int = -100, v: int | None = None, dtype: str | None = None,
            scale: float = 1.0, mask=None):
    """FP64 (logp[n], lse[n]) of logits x[n, ld] (first v columns), with the
    logits scaled by `scale` (1/temperature) and an optional active mask."""
    x, dt = _logits(x, dtype)
    n, v, ld = _shape(x, v)
    y = np.ascontiguousarray(y, dtype=np.int64)
    mk, mp = _mask(mask, n)
    logp = np.empty(n, dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    _load().oracle_forward(x.ctypes.data, dt, n, v, ld, y, ignore_index, mp, float(scale), logp, lse)
    return logp, lse


def backward(x, y, g, ignore_index: int = -100, v: int | None = None, dtype: str | None = None,
             scale: float = 1.0, mask=None) -> np.ndarray:
    """Dense FP64 gradient d[n, v] with respect to the unscaled logits (small
    shapes only)."""
    x, dt = _logits(x, dtype)
    n, v, ld = _shape(x, v)
    y = np.ascontiguousarray(y, dtype=np.int64)
    g = np.ascontiguousarray(g, dtype=np.float32)
    mk, mp = _mask(mask, n)
    d = np.empty((n, v), dtype=np.float64)
    _load().oracle_backward(x.ctypes.data, dt, n, v, ld, y, ignore_index, mp, float(scale), g, d, v)
    return d


def backward_compare(x, y, g, dl, ignore_index: int = -100, v: int | None = None,
                     dtype: str | None = None, scale: float = 1.0, mask=None,
                     out_dtype: str | None = None) -> dict:
    """Stream-compare a gradient dl[n, ld_out] (uint16 bits of bf16/f16, or
    float32) with the FP64 gradient; "correctly rounded" = equal to the nearest
    value of the output dtype (that of the logits unless out_dtype is given)."""
    x, dt = _logits(x, dtype)
    n, v, ld = _shape(x, v)
    dl, odt = _logits(dl, out_dtype if out_dtype is not None else
                      (None if x.dtype == np.float32 else (dtype or "bf16")))
    if dl.ndim != 2 or dl.shape[0] != n or dl.shape[1] < v:
        raise ValueError("dlogits shape mismatch")
    y = np.ascontiguousarray(y, dtype=np.int64)
    g = np.ascontiguousarray(g, dtype=np.float32)
    mk, mp = _mask(mask, n)
    stats = np.zeros(3, dtype=np.float64)
    counts = np.zeros(3, dtype=np.int64)
    _load().oracle_backward_compare(x.ctypes.data, dt, n, v, ld, y, ignore_index, mp, float(scale),
                                    g, dl.ctypes.data, odt, dl.shape[1], stats, counts)
    return {
        "max_abs_diff": float(stats[0]),
        "max_abs_d": float(stats[1]),
        "max_rounding_gap": float(stats[2]),
        "n_compared": int(counts[0]),
        "n_not_correctly_rounded": int(counts[1]),
        "n_nonfinite": int(counts[2]),
    }


def linear_logp(h, w, y, ignore_index: int = -100, d: int | None = None, scale: float = 1.0,
                mask=None, with_bound: bool = False):
    """FP64 (logp[n], lse[n]) of the logits z = h[:, :d] @ w[:, :d].T (h [n, ldh]
    and w [v, ldw] as BF16 bit patterns), scaled by `scale` (1/temperature);
    with `with_bound`, also max_j sum_k |h_k w_jk| per row."""
    h, w = _u16(h), _u16(w)
    if h.ndim != 2 or w.ndim != 2:
        raise ValueError("hidden and weight must be 2-D")
    n, ldh = h.shape
    v, ldw = w.shape
    d = min(ldh, ldw) if d is None else int(d)
    if d > ldh or d > ldw:
        raise ValueError("d exceeds a row stride")
    y = np.ascontiguousarray(y, dtype=np.int64)
    if y.shape != (n,):
        raise ValueError("targets must have shape [n]")
    mk, mp = _mask(mask, n)
    logp = np.empty(n, dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    bound = np.empty(n, dtype=np.float64) if with_bound else None
    _load().oracle_linear_logp(h, ldh, w, ldw, n, d, v, y, ignore_index, mp, float(scale), logp, lse,
                               bound.ctypes.data if with_bound else None)
    return (logp, lse, bound) if with_bound else (logp, lse)


def linear_backward(h, w, y, g, ignore_index: int = -100, d: int | None = None, scale: float = 1.0,
                    mask=None, round_dz: bool = True, with_dz: bool = False):
    """FP64 (dH [n, d], dW [v, d]) of sum_t g_t logp_t of the fused LM head,
    through dZ rounded to BF16 when `round_dz` (as the method writes dlogits);
    with `with_dz`, also dZ [n, v]."""
    h, w = _u16(h), _u16(w)
    n, ldh = h.shape
    v, ldw = w.shape
    d = min(ldh, ldw) if d is None else int(d)
    y = np.ascontiguousarray(y, dtype=np.int64)
    g = np.ascontiguousarray(g, dtype=np.float32)
    if y.shape != (n,) or g.shape != (n,):
        raise ValueError("targets and grad must have shape [n]")
    mk, mp = _mask(mask, n)
    dh = np.empty((n, d), dtype=np.float64)
    dw = np.empty((v, d), dtype=np.float64)
    dz = np.empty((n, v), dtype=np.float64) if with_dz else None
    _load().oracle_linear_backward(h, ldh, w, ldw, n, d, v, y, ignore_index, mp, float(scale), g,
                                   int(bool(round_dz)), dz.ctypes.data if with_dz else None, dh, dw)
    return (dh, dw, dz) if with_dz else (dh, dw)


def range_partials(x, w: int, k: int, v: int | None = None, dtype: str | None = None,
                   scale: float = 1.0):
    """FP64 (m, s) partials [n, k] of the scaled logits over consecutive column
    ranges of width w."""
    x, dt = _logits(x, dtype)
    n, v, ld = _shape(x, v)
    pm = np.empty((n, k), dtype=np.float64)
    ps = np.empty((n, k), dtype=np.float64)
    _load().oracle_range_partials(x.ctypes.data, dt, n, v, ld, w, k, float(scale), pm, ps)
    return pm, ps


def merge_partials(pm, ps) -> np.ndarray:
    """FP64 LSE[n] from partials [n, k] merged in index order."""
    pm = np.ascontiguousarray(pm, dtype=np.float64)
    ps = np.ascontiguousarray(ps, dtype=np.float64)
    n, k = pm.shape
    lse = np.empty(n, dtype=np.float64)
    _load().oracle_merge_partials(pm, ps, n, k, lse)
    return lse


GRPO_MODES = {"token_mean": 0, "seq_mean_token_mean": 1, "seq_mean_token_sum": 2}


def grpo_loss(logp, old_logp, advantages, ref_logp=None, mask=None, cu_seqlens=None,
              mode: str = "token_mean", eps_lo: float = 0.2, eps_hi: float = 0.2,
              beta: float = 0.0, normalizer: float = 0.0):
    """FP64 (loss, g[n]) of the clipped-surrogate GRPO loss on per-token logp
    (definitions in logp_oracle.c, oracle_grpo_loss)."""
    lp = np.ascontiguousarray(logp, dtype=np.float64)
    n = lp.shape[0]
    old = np.ascontiguousarray(old_logp, dtype=np.float64)
    adv = np.ascontiguousarray(advantages, dtype=np.float64)
    ref = None if ref_logp is None else np.ascontiguousarray(ref_logp, dtype=np.float64)
    mk, mp = _mask(mask, n)
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    loss = np.zeros(1, dtype=np.float64)
    g = np.empty(n, dtype=np.float64)
    _load().oracle_grpo_loss(lp, old, None if ref is None else ref.ctypes.data, adv, mp,
                             None if cu is None else cu.ctypes.data,
                             0 if cu is None else cu.shape[0] - 1, n, GRPO_MODES[mode],
                             float(eps_lo), float(eps_hi), float(beta), float(normalizer), loss, g)
    return float(loss[0]), g
