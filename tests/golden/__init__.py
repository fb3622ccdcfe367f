"""Loader for the text fixtures in this folder (no arithmetic of the method)."""

import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def _floats(spec: str, v: int):
    kind, _, body = spec.partition(":")
    if kind == "fill":
        return [float(body)] * v
    if kind == "list":
        vals = [float(t) for t in body.split(",")]
        if len(vals) != v:
            raise ValueError(f"expected {v} values, got {len(vals)}")
        return vals
    raise ValueError(spec)


def closed_forms():
    """Cases of closed_forms.txt as dicts; logits as float64 arrays whose
    values are exact BF16 numbers."""
    cases = []
    with open(os.path.join(HERE, "closed_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, v, lg, y, g, logp, lse, d = [t.strip() for t in line.split(";")]
            v = int(v)
            cases.append({
                "name": name,
                "v": v,
                "logits": np.array(_floats(lg, v), dtype=np.float64),
                "target": int(y),
                "grad": None if g == "-" else float(g),
                "logp": float(logp),
                "lse": float(lse),
                "dlogits": None if d == "-" else np.array(_floats(d, v), dtype=np.float64),
            })
    return cases


def temperature_forms():
    """Cases of temperature_forms.txt (as closed_forms, plus "scale")."""
    cases = []
    with open(os.path.join(HERE, "temperature_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, v, lg, y, sc, g, logp, lse, d = [t.strip() for t in line.split(";")]
            v = int(v)
            cases.append({
                "name": name,
                "v": v,
                "logits": np.array(_floats(lg, v), dtype=np.float64),
                "target": int(y),
                "scale": float(sc),
                "grad": None if g == "-" else float(g),
                "logp": float(logp),
                "lse": float(lse),
                "dlogits": None if d == "-" else np.array(_floats(d, v), dtype=np.float64),
            })
    return cases


def to_bf16_bits_exact(vals) -> np.ndarray:
    """BF16 bit patterns of values that are exactly representable in BF16
    (raises otherwise): the top half of their binary32 encoding."""
    a = np.asarray(vals, dtype=np.float64)
    f = a.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), a, equal_nan=True):
        raise ValueError("not a binary32 value")
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("not a BF16 value")
    return (u >> 16).astype(np.uint16)


__all__ = ["closed_forms", "temperature_forms", "to_bf16_bits_exact"]
