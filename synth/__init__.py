"""Seeded synthetic inputs for the tensor-parallel MLP workloads.

This module is shared by the CUDA path's tests and bench and by the oracle's
tests.  It holds none of the method's arithmetic: only random draws, the
float32 -> bfloat16 encoding of those draws (round to nearest, ties to even,
applied once to each drawn value), and the workload shapes.

Recipe (one ``numpy.random.default_rng(seed)`` per workload, seed 0 unless a
test says otherwise; draws in this fixed order, float32 samples):

* MLP workloads: X [M x H] ~ N(0, 1); W1 [H x F] ~ N(0, 1/H) (for SwiGLU: Wg
  then Wu, each [H x F], stored side by side as W1 = [Wg | Wu], [H x 2F]);
  W2 [F x H] ~ N(0, 1/F); then, if asked for, round(outlier_frac * M)
  distinct outlier rows of X chosen with ``rng.choice`` and scaled by
  ``outlier_scale`` in float32.  For bf16 workloads every array is then cast
  to bfloat16 once.
* Decode workloads draw X with 16 rows and use its first M rows, so M in
  {1, 4, 16} shares one set of weights.
* Attention projections: X [M x H] ~ N(0, 1); Wqkv [H x 3H] = [Wq | Wk | Wv]
  ~ N(0, 1/H); Wo [H x H] ~ N(0, 1/H); A [M x H] ~ N(0, 1) (the attention
  output that feeds the output projection; heads side by side).
* Partial sums for the standalone shard-sum: P [T x n] float32 ~ N(0, 1).
* Attention core: Q, K, V head-major [n_heads x M x head_dim] ~ N(0, 1),
  drawn in that order; Q is then scaled by ``q_scale`` (score spread: 1 gives
  scores of about unit variance, larger values peakier softmax rows) and key
  row j by 1 + ``key_ramp`` * j / M (later keys score higher, so a row's
  running maximum keeps moving); bfloat16.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "WORKLOADS",
    "f32_to_bf16_bits",
    "mlp_inputs",
    "attn_inputs",
    "partials_inputs",
    "attention_inputs",
]

# Workload shapes.  Names say what each one is; the sizes are those of the
# tensor-parallel MLP on the pages (prefill, decode, attention projections).
WORKLOADS = {
    "tiny_fp32_gelu": dict(kind="mlp", M=8, H=64, F=256, T=2, act="gelu", dtype="f32"),
    "prefill_gelu_m2048_h4096_f16384_t4": dict(
        kind="mlp", M=2048, H=4096, F=16384, T=4, act="gelu", dtype="bf16"),
    "decode_swiglu_h8192_f28672_t8": dict(
        kind="mlp", M=16, H=8192, F=28672, T=8, act="swiglu", dtype="bf16",
        decode_m=(1, 4, 16)),
    "attn_proj_m4096_h4096_32x128_t8": dict(
        kind="attn", M=4096, H=4096, n_heads=32, head_dim=128, T=8, dtype="bf16"),
    "prefill_swiglu_m8192_h8192_f28672_t8_outliers": dict(
        kind="mlp", M=8192, H=8192, F=28672, T=8, act="swiglu", dtype="bf16",
        outlier_frac=0.01, outlier_scale=20.0),
}

_CHUNK = 1 << 24


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Encode float32 values as bfloat16 bit patterns (uint16), rounding to
    nearest with ties to even.  Inputs are finite draws; no NaN handling."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    flat = a.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for s in range(0, flat.size, _CHUNK):
        u = flat[s:s + _CHUNK].view(np.uint32)
        bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        out[s:s + _CHUNK] = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    return out.reshape(a.shape)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _encode(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    raise ValueError(f"unknown dtype {dtype!r}")


def mlp_inputs(M: int, H: int, F: int, act: str, dtype: str, seed: int = 0,
               outlier_frac: float = 0.0, outlier_scale: float = 20.0,
               x_rows: int | None = None) -> dict:
    """Draw X, W1, W2 for one MLP workload.

    Returns a dict with ``X`` [M x H], ``W1`` [H x F] (or [H x 2F] = [Wg | Wu]
    for ``act == "swiglu"``), ``W2`` [F x H], each float32 (``dtype="f32"``)
    or bfloat16 bit patterns as uint16 (``dtype="bf16"``), plus
    ``outlier_rows`` (sorted indices, possibly empty).  ``x_rows`` draws X
    with that many rows and keeps the first M (decode workloads).
    """
    rng = np.random.default_rng(seed)
    xr = M if x_rows is None else x_rows
    if xr < M:
        raise ValueError("x_rows must be >= M")
    X = _normal(rng, (xr, H), 1.0)
    w_std = 1.0 / math.sqrt(H)
    if act == "swiglu":
        Wg = _normal(rng, (H, F), w_std)
        Wu = _normal(rng, (H, F), w_std)
        W1 = np.concatenate([Wg, Wu], axis=1)
        del Wg, Wu
    else:
        W1 = _normal(rng, (H, F), w_std)
    W2 = _normal(rng, (F, H), 1.0 / math.sqrt(F))
    rows = np.zeros(0, dtype=np.int64)
    if outlier_frac > 0.0:
        k = int(round(outlier_frac * xr))
        rows = np.sort(rng.choice(xr, size=k, replace=False)).astype(np.int64)
        X[rows] *= np.float32(outlier_scale)
    X = X[:M]
    rows = rows[rows < M]
    return dict(X=_encode(X, dtype), W1=_encode(W1, dtype), W2=_encode(W2, dtype),
                outlier_rows=rows)


def attn_inputs(M: int, H: int, n_heads: int, head_dim: int, seed: int = 0) -> dict:
    """Draw X [M x H], Wqkv [H x 3H] = [Wq | Wk | Wv], Wo [H x H] and the
    attention output A [M x H] (bfloat16 bit patterns)."""
    if n_heads * head_dim != H:
        raise ValueError("n_heads * head_dim must equal H")
    rng = np.random.default_rng(seed)
    X = _normal(rng, (M, H), 1.0)
    Wqkv = _normal(rng, (H, 3 * H), 1.0 / math.sqrt(H))
    Wo = _normal(rng, (H, H), 1.0 / math.sqrt(H))
    A = _normal(rng, (M, H), 1.0)
    return dict(X=f32_to_bf16_bits(X), Wqkv=f32_to_bf16_bits(Wqkv),
                Wo=f32_to_bf16_bits(Wo), A=f32_to_bf16_bits(A))


def partials_inputs(T: int, n: int, seed: int = 0) -> np.ndarray:
    """Draw T partial products of n float32 values each, [T x n] ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    return _normal(rng, (T, n), 1.0)


def attention_inputs(M: int, n_heads: int, head_dim: int = 128, seed: int = 0, q_scale: float = 1.0,
                     key_ramp: float = 0.0) -> dict:
    """Draw head-major Q, K, V [n_heads x M x head_dim] (bfloat16 bit patterns)."""
    rng = np.random.default_rng(seed)
    shape = (n_heads, M, head_dim)
    Q, K, V = _normal(rng, shape, 1.0), _normal(rng, shape, 1.0), _normal(rng, shape, 1.0)
    if q_scale != 1.0:
        Q *= np.float32(q_scale)
    if key_ramp != 0.0:
        K *= (1.0 + np.float32(key_ramp) * np.arange(M, dtype=np.float32) / np.float32(M))[None, :, None]
    return dict(Q=f32_to_bf16_bits(Q), K=f32_to_bf16_bits(K), V=f32_to_bf16_bits(V))
