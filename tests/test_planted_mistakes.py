"""Planted mistakes (CPU only): each test builds a plausible wrong result from
the oracle's own pieces, as a slip in the computation would, and shows that the
comparison its pin (or the GPU parity test) uses rejects it.  This checks that
the checks can fail: a pin that accepts a dropped shard, swapped SwiGLU halves,
a missing attention scale or a one-ulp change of a bit-exact sum would be no
pin.  Mistakes are planted on the host, in computations built from the oracle;
the CUDA path is not involved."""
import math

import numpy as np
import pytest

import oracle
from synth import attention_inputs, mlp_inputs, partials_inputs
from tests.gpu_util import TOL_BF16_ROW_RMS, BF16H_ERROR_RATIO, attention_elementwise_ok, rowwise_rms_error


def _normwise(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _sharded_from_pieces(d, T, act, drop=None):
    """Sum over shards of act(X W1_i) W2_i, built from the oracle's first-layer
    shard outputs and a plain matmul with the oracle's W2 row blocks; `drop`
    leaves one shard out."""
    X = d["X"]
    F = d["W2"].shape[0]
    Z = 0.0
    for i in range(T):
        if i == drop:
            continue
        Y = oracle.colpar_shard(X, d["W1"], F, T, act, i)
        W2i = oracle.shard_w2(d["W2"], T, i)
        W2f = (W2i.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if W2i.dtype == np.uint16 else W2i
        Z = Z + Y @ W2f
    return Z


def test_dropped_shard_is_caught():
    d = mlp_inputs(M=7, H=32, F=64, act="gelu", dtype="f32", seed=3)
    ref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")
    good = _sharded_from_pieces(d, 4, "gelu")
    bad = _sharded_from_pieces(d, 4, "gelu", drop=2)
    assert _normwise(good, ref) <= 1e-12          # the construction itself is right
    assert _normwise(bad, ref) > 1e-3             # the sharded = unsharded pin rejects it
    assert rowwise_rms_error(bad, ref) > TOL_BF16_ROW_RMS  # and so does the GPU parity bound


def test_swapped_swiglu_halves_are_caught():
    """Gate and up exchanged: SiLU(u) g instead of SiLU(g) u."""
    d = mlp_inputs(M=9, H=32, F=64, act="swiglu", dtype="f32", seed=4)
    W1 = d["W1"]
    F = d["W2"].shape[0]
    swapped = np.concatenate([W1[:, F:], W1[:, :F]], axis=1)
    ref = oracle.mlp_unsharded(d["X"], W1, d["W2"], "swiglu")
    bad = oracle.mlp_unsharded(d["X"], swapped, d["W2"], "swiglu")
    assert rowwise_rms_error(bad, ref) > TOL_BF16_ROW_RMS


def test_tanh_gelu_is_caught():
    """The tanh approximation of GeLU differs from the erf form by about 1e-4
    to 1e-3 near |x| = 2, far outside the golden GeLU pin's relative 2e-15."""
    for x in (-2.0, 1.5, 2.0):
        tanh_gelu = 0.5 * x * (1 + math.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))
        assert abs(tanh_gelu - oracle.gelu(x)) > 1e-6 * abs(oracle.gelu(x))


def test_one_ulp_in_a_bit_exact_sum_is_caught():
    """The shard-sum is checked bit for bit: changing one element by one unit
    in the last place is a failure."""
    P = partials_inputs(4, 1000, seed=5)
    Z = oracle.partial_sum_f32(P)
    bad = Z.copy()
    bad.view(np.uint32)[123] += 1
    assert not np.array_equal(bad, Z)
    assert np.array_equal(oracle.partial_sum_f32(P), Z)


def test_attention_scale_and_mask_mistakes_are_caught():
    """Attention without the 1/sqrt(head_dim) scale, or with the causal mask off
    by one key, is rejected by the attention parity bound."""
    from scipy.special import softmax
    d = attention_inputs(64, 2, seed=6)
    Q, K, V = ((d[k].astype(np.uint32) << 16).view(np.float32).astype(np.float64) for k in ("Q", "K", "V"))
    ref = oracle.attention(d["Q"], d["K"], d["V"], causal=True)

    def attn(scale, shift):
        nh, M, hd = Q.shape
        mask = np.tril(np.ones((M, M), dtype=bool), k=shift)
        with np.errstate(invalid="ignore"):  # a row with no key at all (shift -1, token 0) is NaN
            return np.concatenate([softmax(np.where(mask, Q[h] @ K[h].T * scale, -np.inf), axis=1) @ V[h]
                                   for h in range(nh)], axis=1)

    assert attention_elementwise_ok(attn(1 / math.sqrt(128), 0), ref) <= 1e-10  # the construction is right
    # no scale; one key too many; one key too few (token 0 then has none, so rows from 1)
    for wrong, rows in ((attn(1.0, 0), slice(None)), (attn(1 / math.sqrt(128), 1), slice(None)),
                        (attn(1 / math.sqrt(128), -1), slice(1, None))):
        assert rowwise_rms_error(wrong[rows], ref[rows]) > 3e-2
        assert attention_elementwise_ok(wrong[rows], ref[rows]) > 1.5e-2


@pytest.mark.parametrize("T", [2, 4])
def test_misplaced_shard_column_is_caught(T):
    """Shard i taking the columns of shard i + 1 (an off-by-one in the
    partition) breaks the brute-force layout pin."""
    rng = np.random.default_rng(7)
    H, F = 4, 8 * T
    W1 = rng.standard_normal((H, F)).astype(np.float32)
    good = oracle.shard_w1(W1, F, T, "gelu", 0)
    shifted = W1[:, F // T: 2 * F // T]
    assert np.array_equal(good, W1[:, : F // T])
    assert not np.array_equal(good, shifted)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_unrounded_or_truncated_h_is_caught(act):
    """The diagnostic against the oracle that rounds h to bfloat16 (to
    nearest even): a computation that kept h unrounded, or truncated it to
    bfloat16, is not closer to that oracle than to the fp64-h one by the
    required ratio."""
    d = mlp_inputs(M=16, H=512, F=2048, act=act, dtype="bf16", seed=5)
    F = d["W2"].shape[0]
    ref = oracle.mlp_unsharded_hbf16(d["X"], d["W1"], d["W2"], act)
    unrounded = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    h = oracle.colpar_full(d["X"], d["W1"], F, act)
    W2 = (d["W2"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    truncated = (h.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64) @ W2
    exact = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    for bad in (unrounded, truncated):
        assert rowwise_rms_error(bad, ref) > BF16H_ERROR_RATIO * rowwise_rms_error(bad, exact)
