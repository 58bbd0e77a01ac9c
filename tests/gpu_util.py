"""Helpers for the GPU parity tests: moving seeded inputs to the device and
the error measures the tolerances are stated in."""
import numpy as np


def to_device(a: np.ndarray):
    """numpy float32 or bfloat16 bits (uint16) -> CUDA tensor of that type."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def bf16_bits(t) -> np.ndarray:
    """bfloat16 CUDA tensor -> uint16 bit patterns on the host."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rowwise_rms_error(Z: np.ndarray, Zref: np.ndarray) -> float:
    """max over (r, c) of |Z - Zref| / RMS(Zref[r, :]): the bf16 tolerance
    measure, normalised per output row (token)."""
    rms = np.sqrt(np.mean(np.asarray(Zref, np.float64) ** 2, axis=1, keepdims=True))
    return float(np.max(np.abs(np.asarray(Z, np.float64) - Zref) / np.maximum(rms, 1e-300)))


def global_rms_error(Z: np.ndarray, Zref: np.ndarray, rms: float | None = None) -> float:
    """max |Z - Zref| / RMS: the tolerance normalised by one RMS for the
    whole output.  `rms` is the whole output's RMS when only sampled rows are
    compared (see stratified_rms); default: the RMS of Zref itself."""
    if rms is None:
        rms = float(np.sqrt(np.mean(np.asarray(Zref, np.float64) ** 2)))
    return float(np.max(np.abs(np.asarray(Z, np.float64) - Zref)) / max(rms, 1e-300))


def stratified_rms(Zref_rows: np.ndarray, is_outlier: np.ndarray, n_outliers: int, M: int) -> float:
    """RMS of a whole [M x H] output from sampled rows, one stratum for the
    `n_outliers` outlier rows and one for the rest: the mean square of each
    stratum is taken from its sampled rows and weighted by its share of M."""
    ms = np.mean(np.asarray(Zref_rows, np.float64) ** 2, axis=1)
    is_outlier = np.asarray(is_outlier, bool)
    total = 0.0
    if n_outliers:
        if not is_outlier.any():
            raise ValueError("no outlier row among the samples")
        total += n_outliers / M * float(np.mean(ms[is_outlier]))
    if n_outliers < M:
        total += (M - n_outliers) / M * float(np.mean(ms[~is_outlier]))
    return float(np.sqrt(total))


def normwise_error(Z: np.ndarray, Zref: np.ndarray) -> float:
    """max |Z - Zref| / max |Zref|: the float32 tolerance measure."""
    return float(np.max(np.abs(np.asarray(Z, np.float64) - Zref)) / max(np.max(np.abs(Zref)), 1e-300))


# Tolerances (stated for the path): bf16 inputs with float32 accumulation,
# bf16 intermediate Y: max-abs error over the output row's RMS <= 2e-2;
# float32 inputs: normwise relative error <= 1e-4.
TOL_BF16_ROW_RMS = 2e-2
TOL_F32_NORMWISE = 1e-4

# The diagnostic against the oracle that also rounds the first layer's output
# h to bfloat16 as the workloads store it (oracle.mlp_unsharded_hbf16).  A
# kernel that rounds its float32 h to nearest differs from that oracle only
# in the h whose float32 value (float32 sums of K products, some of which
# nearly cancel) lies across a bfloat16 midpoint from the exact value, one
# bfloat16 step each.  If a fraction p of the h do, its error against that
# oracle is about sqrt(3 p) times its error against the fp64-h oracle (which
# every h's rounding makes, uniformly distributed over the step), and p is a
# few percent at most: a ratio below about 0.4 (0.14-0.26 for an exact
# float32 emulation of the kernels on small shapes; on the GPU at the full
# workload sizes 0.13 prefill GeLU, 0.30 large SwiGLU, 0.12-0.21 decode).
# A kernel that skipped the rounding, or truncated h instead, has the ratio
# above 1 (tests/test_planted_mistakes.py).  Bound on the ratio: 0.75.
BF16H_ERROR_RATIO = 0.75

# The same measure normalised by the RMS of the whole output (the literal
# reading), on a workload with 1 % of its token rows scaled x20.  SwiGLU is
# quadratic in x, so an outlier row's output RMS is about 10x the whole
# output's RMS, and the ordinary bf16 rounding of its h (the same share of
# that row's own RMS as in every row) reads 10x larger here.  Emulating only
# that rounding in numpy on the large SwiGLU workload's sampled rows (fp64
# otherwise) gives 7.2e-3 of an outlier row's own RMS, 0.069 of the whole
# output's.  Held to 0.1: on the outlier rows this is a per-row bound of about
# 1e-2, half the row-RMS tolerance, so a regression confined to the outlier
# rows cannot hide inside their own (large) normalisation.
TOL_BF16_GLOBAL_RMS_OUTLIERS = 0.1

# Gradients of the training path: the chain to dW1 and dX passes three bf16
# roundings (the saved pre-activation, dP = dH * act'(P) and, for dW, the
# transposed operands are exact copies) against the forward's one (Y); the
# forward's measured row-RMS error is about 8e-3 per rounding, so the
# gradients are held to 3e-2.  That assumes the weight gradients sum over
# enough tokens for those roundings (2^-9 relative each) to average: an exact
# float32 emulation of the same rounding chain (SwiGLU, H = 384, F = 512)
# puts dW1 at 1.3e-2 with 512 or 2048 tokens, 2.0e-2 with 128 and 2.5-3.2e-2
# with 44, where a few tokens' terms dominate each dW1 element.  The bound
# is asserted for sums over at least 64 tokens (GRAD_MIN_TOKENS), as all
# the backward tests run.
TOL_BF16_GRAD_ROW_RMS = 3e-2
GRAD_MIN_TOKENS = 64

# The attention output passes through two bf16 roundings: the probabilities P
# (each weight relative 2^-9, rounded once before the P V product) and the
# stored output O.  Checked elementwise like any stored bf16 tensor, as
# |O - ref| <= 2^-8 |ref| + TOL_ATTN_ELEMENT * RMS(ref row): the first term
# holds O's own rounding (<= 2^-9 |ref|); the second the probability rounding,
# whose error is a weighted sum of (v_j - o) with independent relative errors
# of at most 2^-9 (measured <= 1.03e-2 of the row RMS alone and <= 8.1e-3 on
# top of the first term, on the parity inputs, by emulating the kernel's
# arithmetic in numpy).  The row-RMS measure is held to the multi-rounding
# bound TOL_BF16_GRAD_ROW_RMS.
TOL_ATTN_ELEMENT = 1.5e-2


def attention_elementwise_ok(got: np.ndarray, ref: np.ndarray) -> float:
    """Largest (|got - ref| - 2^-8 |ref|) / RMS(ref row); the check passes
    when it is <= TOL_ATTN_ELEMENT."""
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    slack = (np.abs(np.asarray(got, np.float64) - ref) - 2.0 ** -8 * np.abs(ref)) / np.maximum(rms, 1e-300)
    return float(np.max(slack))
