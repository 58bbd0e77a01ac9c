"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code (CPU only).

Each test names the fact it pins.  Together they are chosen so that a
plausible slip in the oracle (a dropped term of GeLU, the gate and up halves
swapped, a transposed operand, an off-by-one shard index, a dropped partial)
fails at least one of them.
"""
import math
from pathlib import Path

import numpy as np
import pytest
from scipy import special

import oracle
from synth import attn_inputs, f32_to_bf16_bits, mlp_inputs

GOLDEN = Path(__file__).parent / "golden"


def _kv(name):
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        out[k] = float(v)
    return out


def _table(name):
    rows = []
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(float(t) for t in line.split()))
    return rows


def _decode(a):
    """Exact values of float32 / bfloat16-bit arrays, decoded here without the oracle."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _normwise(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --- element decoding --------------------------------------------------------

@pytest.mark.parametrize("bits,val", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x3FC0, 1.5), (0x4049, 3.140625),
    (0x0001, 2.0 ** -133), (0x8000, -0.0), (0x7F7F, 3.3895313892515355e38),
    (0x3E80, 0.25),
])
def test_bf16_values_exact(bits, val):
    """bfloat16 is the upper half of an IEEE float32: known bit patterns."""
    a = np.array([bits], dtype=np.uint16)
    assert oracle.value(a, 0) == val
    assert math.copysign(1.0, oracle.value(a, 0)) == math.copysign(1.0, val)


# --- activations --------------------------------------------------------------

@pytest.mark.parametrize("x,phi", _table("gelu_normal_cdf.txt"))
def test_gelu_is_x_times_normal_cdf(x, phi):
    """GeLU(x) = x Phi(x) at tabulated Phi values (a dropped 0.5, a missing
    1/sqrt(2) or the tanh approximation all fail here).  In the left tail
    1 + erf(x/sqrt 2) cancels, so the bound there is absolute: |x| times a
    few units of fp64 rounding."""
    assert oracle.gelu(x) == pytest.approx(x * phi, rel=2e-15, abs=4e-16 * abs(x))


def test_silu_closed_forms():
    """SiLU(g) = g sigmoid(g): SiLU(1) = 1/(1+e^-1), SiLU(-1) = -1/(1+e), SiLU(0) = 0."""
    assert oracle.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert oracle.silu(-1.0) == pytest.approx(-0.2689414213699951, rel=1e-15)
    assert oracle.silu(0.0) == 0.0
    for g in np.linspace(-30, 30, 61):
        assert oracle.silu(g) == pytest.approx(g * special.expit(g), rel=1e-14, abs=1e-300)


# --- the hand-worked example --------------------------------------------------

def test_one_sigma_two_shard_mlp():
    """Two shards, X = [1, -1], W1 = I, W2 = [[1, 0], [1, 0]]:
    Z = [GeLU(1) + GeLU(-1), 0] = [erf(1/sqrt 2), 0]."""
    g = _kv("one_sigma_mlp.txt")
    X = np.array([[1.0, -1.0]], dtype=np.float32)
    W1 = np.eye(2, dtype=np.float32)
    W2 = np.array([[1.0, 0.0], [1.0, 0.0]], dtype=np.float32)
    for Z in (oracle.mlp_unsharded(X, W1, W2, "gelu"), oracle.mlp_sharded(X, W1, W2, 2, "gelu")):
        assert Z[0, 0] == pytest.approx(g["Z0"], rel=1e-15)
        assert Z[0, 1] == g["Z1"]


def test_shape_mismatch_rejected():
    X = np.zeros((1, 2), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.mlp_unsharded(X, np.eye(2, dtype=np.float32), np.ones((2, 1), np.float32), "gelu")


# --- the column-parallel identity (act per shard) ----------------------------

@pytest.mark.parametrize("act", ["gelu", "swiglu", "identity"])
@pytest.mark.parametrize("T", [1, 2, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_activation_concatenation_identity(act, T, dtype):
    """act([y_1 | ... | y_T]) = [act(y_1) | ... | act(y_T)] exactly: the
    per-shard first layer, concatenated, equals the unsharded one bit for bit."""
    d = mlp_inputs(M=5, H=24, F=32, act=act, dtype=dtype, seed=3)
    full = oracle.colpar_full(d["X"], d["W1"], 32, act)
    parts = [oracle.colpar_shard(d["X"], d["W1"], 32, T, act, i) for i in range(T)]
    assert np.array_equal(np.concatenate(parts, axis=1), full)


# --- sharded == unsharded -----------------------------------------------------

@pytest.mark.parametrize("act", ["gelu", "swiglu", "identity"])
@pytest.mark.parametrize("T", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sharded_equals_unsharded(act, T, dtype):
    """Sum over shards of act(X W1_i) W2_i equals act(X W1) W2 (the all-reduce
    reconstructs the dense output) to fp64 rounding."""
    d = mlp_inputs(M=7, H=32, F=64, act=act, dtype=dtype, seed=11)
    zu = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    zs = oracle.mlp_sharded(d["X"], d["W1"], d["W2"], T, act)
    assert _normwise(zs, zu) <= 1e-12


def test_sharded_equals_unsharded_with_outlier_rows():
    d = mlp_inputs(M=64, H=32, F=64, act="swiglu", dtype="bf16", seed=0,
                   outlier_frac=0.05, outlier_scale=20.0)
    assert d["outlier_rows"].size == 3
    zu = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "swiglu")
    zs = oracle.mlp_sharded(d["X"], d["W1"], d["W2"], 8, "swiglu")
    assert _normwise(zs, zu) <= 1e-12


# --- special cases that reduce to library routines ---------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identity_activation_is_associative_product(dtype):
    """With no activation, Z = X (W1 W2): checks operand order and transposes
    of both GEMMs against a library matmul on the exact input values."""
    d = mlp_inputs(M=6, H=16, F=40, act="identity", dtype=dtype, seed=5)
    X, W1, W2 = (_decode(d[k]) for k in ("X", "W1", "W2"))
    ref = X @ (W1 @ W2)
    for T in (1, 2, 4, 8):
        assert _normwise(oracle.mlp_sharded(d["X"], d["W1"], d["W2"], T, "identity"), ref) <= 1e-13
    assert _normwise(oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "identity"), ref) <= 1e-13


def test_permutation_weights_give_gelu_of_input():
    """W1 = P, W2 = P^T (P a permutation): Z = GeLU(X) elementwise, checked
    against x * Phi(x) from scipy's normal CDF."""
    rng = np.random.default_rng(1)
    n = 16
    perm = rng.permutation(n)
    P = np.zeros((n, n), dtype=np.float32)
    P[np.arange(n), perm] = 1.0
    X = rng.standard_normal((4, n)).astype(np.float32) * 2
    ref = X.astype(np.float64) * special.ndtr(X.astype(np.float64))
    # erf-form cancellation in the left tail: absolute bound |x| * 4 ulp(1)
    bound = 1e-14 * np.abs(ref) + 4e-16 * np.abs(X.astype(np.float64))
    for T in (1, 2, 4):
        Z = oracle.mlp_sharded(X, P, np.ascontiguousarray(P.T), T, "gelu")
        assert np.all(np.abs(Z - ref) <= bound)
    Zi = oracle.mlp_unsharded(X, P, np.ascontiguousarray(P.T), "identity")
    assert np.array_equal(Zi, X.astype(np.float64))


def test_swiglu_gate_is_first_half():
    """W1 = [Wg | Wu] with Wg = I, Wu = diag(d), W2 = I: Z = SiLU(x) * d * x.
    Swapping the halves gives SiLU(d x) * x instead, which differs."""
    rng = np.random.default_rng(2)
    n = 8
    d = rng.uniform(0.5, 2.0, n).astype(np.float32)
    X = rng.standard_normal((3, n)).astype(np.float32)
    I = np.eye(n, dtype=np.float32)
    W1 = np.concatenate([I, np.diag(d)], axis=1)
    Xd = X.astype(np.float64)
    ref = Xd * special.expit(Xd) * d * Xd
    for T in (1, 2, 4):
        np.testing.assert_allclose(oracle.mlp_sharded(X, W1, I, T, "swiglu"), ref, rtol=1e-14)
    swapped = np.concatenate([np.diag(d), I], axis=1)
    assert not np.allclose(oracle.mlp_unsharded(X, swapped, I, "swiglu"), ref, rtol=1e-6)


# --- the partition layout (bit exact, brute force) ---------------------------

def _ids(shape):
    return np.arange(int(np.prod(shape)), dtype=np.uint32).astype(np.uint16).reshape(shape)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_w1_column_blocks(act, T):
    """Element (k, c) of W1 (of Wg, Wu for SwiGLU) lands in shard c // (F/T)
    at local column c % (F/T), and every element lands exactly once."""
    H, F = 12, 64
    ncols = 2 * F if act == "swiglu" else F
    W1 = _ids((H, ncols))
    Fs = F // T
    seen = np.zeros(W1.size, dtype=np.int64)
    for i in range(T):
        for which in ((0, 1) if act == "swiglu" else (0,)):
            s = oracle.shard_w1(W1, F, T, act, i, which)
            assert s.shape == (H, Fs)
            for k in range(H):
                for c in range(Fs):
                    src = which * F + i * Fs + c
                    assert s[k, c] == W1[k, src]
                    seen[k * ncols + src] += 1
    assert np.all(seen == 1)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_w2_row_blocks(T):
    """Row r of W2 lands in shard r // (F/T) at local row r % (F/T), once."""
    F, H = 64, 12
    W2 = _ids((F, H))
    Fs = F // T
    seen = np.zeros(W2.size, dtype=np.int64)
    for i in range(T):
        s = oracle.shard_w2(W2, T, i)
        assert s.shape == (Fs, H)
        for r in range(Fs):
            assert np.array_equal(s[r], W2[i * Fs + r])
            seen[(i * Fs + r) * H:(i * Fs + r + 1) * H] += 1
    assert np.all(seen == 1)


@pytest.mark.parametrize("T", [1, 2, 4])
def test_qkv_head_aligned_shards(T):
    """Shard i holds heads [i*nh/T, (i+1)*nh/T) of each of Wq, Wk, Wv; Wo's
    rows of those heads; every column / row exactly once."""
    nh, hd = 8, 4
    H = nh * hd
    Wqkv = _ids((H, 3 * H))
    Wo = _ids((H, H))
    hps = nh // T
    W = hps * hd
    seen = np.zeros(3 * H, dtype=np.int64)
    for i in range(T):
        s = oracle.shard_wqkv(Wqkv, nh, hd, T, i)
        assert s.shape == (H, 3 * W)
        for p in range(3):
            for c in range(W):
                head = i * hps + c // hd
                src = p * H + head * hd + c % hd
                assert np.array_equal(s[:, p * W + c], Wqkv[:, src])
                seen[src] += 1
        o = oracle.shard_wo(Wo, nh, hd, T, i)
        assert np.array_equal(o, Wo[i * W:(i + 1) * W])
    assert np.all(seen == 1)


def test_indivisible_shards_rejected():
    W1 = np.zeros((4, 10), dtype=np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.shard_w1(W1, 10, 4, "gelu", 0)
    assert e.value.code == oracle.ERR_INDIVISIBLE
    X = np.zeros((2, 4), dtype=np.float32)
    W2 = np.zeros((10, 4), dtype=np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.mlp_sharded(X, W1, W2, 3, "gelu")


# --- attention projections ----------------------------------------------------

def test_qkv_shards_are_dense_columns_and_oproj_sum_is_dense():
    """Head-sharded QKV equals the matching columns of the dense X Wqkv bit
    for bit; the row-parallel output projection summed over shards equals
    the dense A Wo."""
    nh, hd, T, M = 8, 8, 4, 5
    d = attn_inputs(M=M, H=nh * hd, n_heads=nh, head_dim=hd, seed=4)
    H = nh * hd
    dense = oracle.linear(d["X"], d["Wqkv"])
    W = nh // T * hd
    for i in range(T):
        s = oracle.qkv_shard(d["X"], d["Wqkv"], nh, hd, T, i)
        cols = np.concatenate([np.arange(p * H + i * W, p * H + (i + 1) * W) for p in range(3)])
        assert np.array_equal(s, dense[:, cols])
    ref = _decode(d["A"]) @ _decode(d["Wo"])
    assert _normwise(oracle.oproj_sharded(d["A"], d["Wo"], nh, hd, T), ref) <= 1e-13


# --- row sampling -------------------------------------------------------------

def test_row_subset_matches_full_rows():
    """A row of Z depends only on that row of X: the sampled-row oracle (used at
    full sizes) returns exactly the rows of the full computation."""
    d = mlp_inputs(M=20, H=16, F=32, act="swiglu", dtype="bf16", seed=9)
    full = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "swiglu")
    rows = np.array([19, 0, 7, 7])
    sub = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "swiglu", rows=rows)
    assert np.array_equal(sub, full[rows])


# --- the all-reduce-sum arithmetic -------------------------------------------

def test_partial_sum_integers_exact():
    """Integer-valued partials sum exactly in float32: each shard counted once."""
    rng = np.random.default_rng(0)
    P = rng.integers(-1000, 1000, size=(8, 257)).astype(np.float32)
    assert np.array_equal(oracle.partial_sum_f32(P), P.astype(np.int64).sum(0).astype(np.float32))


def test_partial_sum_order_is_ascending_left_to_right():
    """(a + b) + c in float32 with a = 1, b = 2^-24, c = 2^-24 gives 1, while
    a + (b + c) gives 1 + 2^-23: the order is ascending shard index, left to right."""
    P = np.array([[1.0], [2.0 ** -24], [2.0 ** -24]], dtype=np.float32)
    assert oracle.partial_sum_f32(P)[0] == np.float32(1.0)
    P2 = P[::-1].copy()
    assert oracle.partial_sum_f32(P2)[0] == np.float32(1.0 + 2.0 ** -23)


def test_partial_sum_within_float32_bound():
    rng = np.random.default_rng(1)
    P = rng.standard_normal((8, 4096)).astype(np.float32)
    exact = P.astype(np.float64).sum(0)
    bound = 8 * 2.0 ** -24 * np.abs(P.astype(np.float64)).sum(0)
    assert np.all(np.abs(oracle.partial_sum_f32(P) - exact) <= bound)


def test_synth_bf16_encoding_round_to_nearest_even():
    """The shared input encoder: ties go to the even bfloat16, others to nearest."""
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -2.5], dtype=np.float32)
    bits = f32_to_bf16_bits(v)
    assert list(bits) == [0x3F80, 0x3F82, 0x3F80, 0xC020]


# --- the other collectives: reduce-scatter, all-gather, bf16 all-reduce -------

@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_reduce_scatter_then_all_gather_is_the_all_reduce(T):
    """The ring all-reduce is a reduce-scatter followed by an all-gather (the
    2 (T-1)/T byte count of the ring): the composition equals the all-reduce
    bit for bit, and each block is the sum of that block over ranks."""
    rng = np.random.default_rng(T)
    n = 64 * T
    P = rng.standard_normal((T, n)).astype(np.float32)
    rs = oracle.reduce_scatter_f32(P)
    assert rs.shape == (T, n // T)
    assert np.array_equal(oracle.all_gather(rs), oracle.partial_sum_f32(P))
    Pi = rng.integers(-50, 50, size=(T, n)).astype(np.float32)
    exact = Pi.astype(np.int64).sum(0).reshape(T, n // T).astype(np.float32)
    assert np.array_equal(oracle.reduce_scatter_f32(Pi), exact)


def test_all_gather_is_concatenation():
    parts = np.arange(24, dtype=np.uint16).reshape(4, 6)
    assert np.array_equal(oracle.all_gather(parts), np.arange(24, dtype=np.uint16))


def test_reduce_scatter_rejects_uneven_blocks():
    with pytest.raises(oracle.OracleError):
        oracle.reduce_scatter_f32(np.zeros((3, 10), dtype=np.float32))


def test_bf16_rounding_matches_the_input_encoder_and_ties_to_even():
    """Two independent implementations of round-to-nearest-even agree; ties
    go to the even neighbour."""
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 100,
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0,
                                  3.3895314e38], dtype=np.float32)])
    assert [oracle.f32_to_bf16(x) for x in v] == list(f32_to_bf16_bits(v))
    assert oracle.f32_to_bf16(1 + 2 ** -8) == 0x3F80
    assert oracle.f32_to_bf16(1 + 3 * 2 ** -8) == 0x3F82
    P = rng.standard_normal((4, 999)).astype(np.float32)
    assert np.array_equal(oracle.partial_sum_bf16(P), f32_to_bf16_bits(oracle.partial_sum_f32(P)))


# --- backward of the MLP ------------------------------------------------------

def _loss(X, W1, W2, G, act):
    """L = sum(Z * G) with the oracle's forward; dL/dZ = G."""
    return float(np.sum(oracle.mlp_unsharded(X, W1, W2, act) * G))


@pytest.mark.parametrize("act", ["gelu", "swiglu", "identity"])
def test_backward_matches_central_differences(act):
    """Every gradient (dX, dW1, dW2) equals the central difference of the
    forward loss sum(Z * dZ) on fp64 inputs: a pin independent of the
    backward's own formulas."""
    rng = np.random.default_rng(12)
    M, H, F = 3, 4, 6
    ncols = 2 * F if act == "swiglu" else F
    X = rng.standard_normal((M, H))
    W1 = rng.standard_normal((H, ncols)) * 0.7
    W2 = rng.standard_normal((F, H)) * 0.7
    G = rng.standard_normal((M, H))
    eps = 1e-6
    dX = oracle.mlp_backward_dx(X, W1, W2, G, act)
    dW1, dW2 = oracle.mlp_backward_dw(X, W1, W2, G, act)
    nparts = 2 if act == "swiglu" else 1

    def fd(arr, idx):
        a, b = arr.copy(), arr.copy()
        a[idx] += eps
        b[idx] -= eps
        if arr is X:
            return (_loss(a, W1, W2, G, act) - _loss(b, W1, W2, G, act)) / (2 * eps)
        if arr is W1:
            return (_loss(X, a, W2, G, act) - _loss(X, b, W2, G, act)) / (2 * eps)
        return (_loss(X, W1, a, G, act) - _loss(X, W1, b, G, act)) / (2 * eps)

    for idx in np.ndindex(X.shape):
        assert dX[idx] == pytest.approx(fd(X, idx), rel=1e-6, abs=1e-8)
    for k, c in np.ndindex(W1.shape):
        part, f = divmod(c, F)
        got = dW1[k, part * F + f] if nparts == 2 else dW1[k, c]
        assert got == pytest.approx(fd(W1, (k, c)), rel=1e-6, abs=1e-8)
    for idx in np.ndindex(W2.shape):
        assert dW2[idx] == pytest.approx(fd(W2, idx), rel=1e-6, abs=1e-8)


def test_activation_derivatives_closed_forms():
    """GeLU'(0) = 1/2, GeLU'(1) = Phi(1) + phi(1); SiLU'(0) = 1/2."""
    from math import exp, pi, sqrt
    assert oracle.gelu_grad(0.0) == pytest.approx(0.5, rel=1e-15)
    assert oracle.gelu_grad(1.0) == pytest.approx(0.8413447460685429 + exp(-0.5) / sqrt(2 * pi), rel=1e-14)
    assert oracle.silu_grad(0.0) == pytest.approx(0.5, rel=1e-15)
    for g in (-3.0, -0.5, 0.7, 4.0):
        h = 1e-6
        assert oracle.silu_grad(g) == pytest.approx((oracle.silu(g + h) - oracle.silu(g - h)) / (2 * h), rel=1e-8)
        assert oracle.gelu_grad(g) == pytest.approx((oracle.gelu(g + h) - oracle.gelu(g - h)) / (2 * h), rel=1e-8)


def test_identity_backward_is_transposed_products():
    """act = identity: dX = dZ W2^T W1^T, dW1 = X^T dZ W2^T, dW2 = (X W1)^T dZ."""
    d = mlp_inputs(M=5, H=8, F=16, act="identity", dtype="f32", seed=6)
    rng = np.random.default_rng(7)
    G = rng.standard_normal((5, 8)).astype(np.float32)
    X, W1, W2 = (_decode(d[k]) for k in ("X", "W1", "W2"))
    Gd = G.astype(np.float64)
    assert _normwise(oracle.mlp_backward_dx(d["X"], d["W1"], d["W2"], G, "identity"), Gd @ W2.T @ W1.T) <= 1e-13
    dW1, dW2 = oracle.mlp_backward_dw(d["X"], d["W1"], d["W2"], G, "identity")
    assert _normwise(dW1, X.T @ (Gd @ W2.T)) <= 1e-13
    assert _normwise(dW2, (X @ W1).T @ Gd) <= 1e-13


def test_backward_column_subset_matches_full():
    d = mlp_inputs(M=6, H=8, F=16, act="swiglu", dtype="bf16", seed=2)
    G = f32_to_bf16_bits(np.random.default_rng(1).standard_normal((6, 8)).astype(np.float32))
    full1, full2 = oracle.mlp_backward_dw(d["X"], d["W1"], d["W2"], G, "swiglu")
    cols = np.array([3, 11, 0])
    s1, s2 = oracle.mlp_backward_dw(d["X"], d["W1"], d["W2"], G, "swiglu", fcols=cols)
    assert np.array_equal(s1[:, :3], full1[:, cols]) and np.array_equal(s1[:, 3:], full1[:, 16 + cols])
    assert np.array_equal(s2, full2[cols])


# --- one transformer block --------------------------------------------------------

def _block_weights(H, F, act, seed):
    rng = np.random.default_rng(seed)
    ncols = 2 * F if act == "swiglu" else F
    return (rng.standard_normal((H, 3 * H)) / np.sqrt(H), rng.standard_normal((H, H)) / np.sqrt(H),
            rng.standard_normal((H, ncols)) / np.sqrt(H), rng.standard_normal((F, H)) / np.sqrt(F))


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("causal", [True, False])
def test_block_sharded_equals_unsharded(act, causal):
    """Both all-reduces reconstruct the dense block: per-shard heads and MLP
    columns summed over shards equal the dense computation."""
    rng = np.random.default_rng(0)
    M, nh, hd, F = 6, 4, 4, 16
    H = nh * hd
    X = rng.standard_normal((M, H))
    Wqkv, Wo, W1, W2 = _block_weights(H, F, act, 1)
    dense, hd_ = oracle.block_forward(X, Wqkv, Wo, W1, W2, nh, hd, 1, act, causal, sharded=False)
    for T in (1, 2, 4):
        out, h = oracle.block_forward(X, Wqkv, Wo, W1, W2, nh, hd, T, act, causal, sharded=True)
        assert _normwise(out, dense) <= 1e-12 and _normwise(h, hd_) <= 1e-12


def test_block_attention_closed_forms():
    """With Wq = 0 every score is 0, so causal attention at token r is the mean
    of v_0..v_r, and the first token attends only to itself."""
    rng = np.random.default_rng(3)
    M, nh, hd, F = 5, 2, 4, 8
    H = nh * hd
    X = rng.standard_normal((M, H))
    Wqkv, Wo, W1, W2 = _block_weights(H, F, "gelu", 2)
    Wqkv[:, :H] = 0.0
    Wo = np.eye(H)
    W1 = np.zeros_like(W1)  # the MLP adds GeLU(0) W2 = 0
    out, h = oracle.block_forward(X, Wqkv, Wo, W1, W2, nh, hd, 2, "gelu", causal=True)
    V = X @ Wqkv[:, 2 * H:]
    for r in range(M):
        expect = X[r] + V[: r + 1].mean(axis=0)
        assert np.allclose(h[r], expect, rtol=1e-13, atol=1e-13)
        assert np.allclose(out[r], expect, rtol=1e-13, atol=1e-13)
    noncausal, _ = oracle.block_forward(X, Wqkv, Wo, W1, W2, nh, hd, 2, "gelu", causal=False)
    assert np.allclose(noncausal, X + V.mean(axis=0), rtol=1e-13, atol=1e-13)


def test_block_matches_a_library_attention():
    """Causal softmax attention written with library routines (scipy softmax,
    numpy matmuls) on the same fp64 inputs."""
    from scipy.special import softmax
    rng = np.random.default_rng(4)
    M, nh, hd, F = 7, 2, 4, 8
    H = nh * hd
    X = rng.standard_normal((M, H))
    Wqkv, Wo, W1, W2 = _block_weights(H, F, "swiglu", 5)
    out, h = oracle.block_forward(X, Wqkv, Wo, W1, W2, nh, hd, 2, "swiglu", causal=True)
    Q, K, V = X @ Wqkv[:, :H], X @ Wqkv[:, H:2 * H], X @ Wqkv[:, 2 * H:]
    O = np.zeros((M, H))
    mask = np.tril(np.ones((M, M), dtype=bool))
    for g in range(nh):
        sl = slice(g * hd, (g + 1) * hd)
        S = np.where(mask, Q[:, sl] @ K[:, sl].T / np.sqrt(hd), -np.inf)
        O[:, sl] = softmax(S, axis=1) @ V[:, sl]
    href = X + O @ Wo
    G, U = href @ W1[:, :F], href @ W1[:, F:]
    ref = href + (G * special.expit(G) * U) @ W2
    assert _normwise(h, href) <= 1e-13 and _normwise(out, ref) <= 1e-13


# --- attention core (per head) ------------------------------------------------

def _library_attention(Q, K, V, causal):
    """Scaled dot-product attention per head from library routines (scipy
    softmax, numpy matmuls): [nh, M, hd] -> [M, nh*hd]."""
    from scipy.special import softmax
    nh, M, hd = Q.shape
    mask = np.tril(np.ones((M, M), dtype=bool)) if causal else np.ones((M, M), dtype=bool)
    return np.concatenate([softmax(np.where(mask, Q[h] @ K[h].T / np.sqrt(hd), -np.inf), axis=1) @ V[h]
                           for h in range(nh)], axis=1)


@pytest.mark.parametrize("causal", [True, False])
def test_attention_matches_a_library_attention(causal):
    """Softmax attention written with library routines on the same fp64
    inputs; 3 heads so that a head offset slip shows."""
    rng = np.random.default_rng(11)
    Q, K, V = (rng.standard_normal((3, 9, 8)) for _ in range(3))
    got = oracle.attention(Q, K, V, causal=causal)
    assert _normwise(got, _library_attention(Q, K, V, causal)) <= 1e-13


def test_attention_closed_forms():
    """Q = 0 makes every score 0: causal attention at token r is the mean of
    v_0..v_r (non-causal: of all v), and token 0 attends only to itself."""
    rng = np.random.default_rng(12)
    K, V = rng.standard_normal((2, 6, 4)), rng.standard_normal((2, 6, 4))
    Q = np.zeros_like(K)
    got = oracle.attention(Q, K, V, causal=True)
    for r in range(6):
        expect = np.concatenate([V[h, : r + 1].mean(axis=0) for h in range(2)])
        assert np.allclose(got[r], expect, rtol=1e-14, atol=1e-14)
    full = oracle.attention(Q, K, V, causal=False)
    assert np.allclose(full, np.concatenate([V[h].mean(axis=0) for h in range(2)])[None, :].repeat(6, 0),
                       rtol=1e-14, atol=1e-14)
    Qr = rng.standard_normal((2, 6, 4))
    assert np.array_equal(oracle.attention(Qr, K, V, causal=True, rows=[0]), V[:, 0].reshape(1, -1))


def test_attention_key_shift_invariance_and_scale():
    """Adding one vector e to every key adds q.e/sqrt(hd) to all scores of a
    row, which the softmax removes; a score gap of d log 2 between two keys
    weighs them 2^-d : 1 (the 1/sqrt(hd) scale, checked with hd = 4)."""
    rng = np.random.default_rng(13)
    Q, K, V = (rng.standard_normal((2, 7, 4)) for _ in range(3))
    e = rng.standard_normal(4) * 3.0
    base = oracle.attention(Q, K, V, causal=True)
    assert _normwise(oracle.attention(Q, K + e, V, causal=True), base) <= 1e-12
    # two keys, q . (k1 - k0) / 2 = 3 log 2: weights 1/9 and 8/9
    q = np.array([[[1.0, 0.0, 0.0, 0.0]] * 2])
    k = np.array([[[0.0, 0.0, 0.0, 0.0], [6 * math.log(2), 0.0, 0.0, 0.0]]])
    v = np.array([[[1.0, 0.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0]]])
    got = oracle.attention(q, k, v, causal=False, rows=[0])
    assert np.allclose(got[0], [1 / 9, 8 / 9, 0.0, 0.0], rtol=1e-14, atol=1e-15)


def test_attention_bf16_inputs_widen_exactly():
    """bfloat16 inputs are the same numbers as their fp64 widening."""
    rng = np.random.default_rng(14)
    Qf, Kf, Vf = (rng.standard_normal((2, 5, 8)).astype(np.float32) for _ in range(3))
    Qb, Kb, Vb = (f32_to_bf16_bits(a) for a in (Qf, Kf, Vf))
    wide = [(b.astype(np.uint32) << 16).view(np.float32).astype(np.float64) for b in (Qb, Kb, Vb)]
    assert np.array_equal(oracle.attention(Qb, Kb, Vb), oracle.attention(*wide))


def test_block_attention_is_the_attention_core():
    """The block's attention contribution (Wo = I, MLP zero, T = 1) equals
    the attention of its projections, so the GPU block and the GPU attention
    core are checked against one definition."""
    rng = np.random.default_rng(15)
    M, nh, hd, F = 6, 2, 4, 8
    H = nh * hd
    X = rng.standard_normal((M, H))
    Wqkv, _, W1, W2 = _block_weights(H, F, "gelu", 16)
    _, h = oracle.block_forward(X, Wqkv, np.eye(H), np.zeros_like(W1), W2, nh, hd, 1, "gelu", causal=True)
    heads = lambda A: A.reshape(M, nh, hd).transpose(1, 0, 2).copy()  # noqa: E731
    Q, K, V = (heads(X @ Wqkv[:, i * H:(i + 1) * H]) for i in range(3))
    assert _normwise(h - X, oracle.attention(Q, K, V, causal=True)) <= 1e-13


# ---- the MLP with its first-layer output in bfloat16 ---------------------------------

def test_mlp_hbf16_rounds_each_h_to_nearest_even():
    """mlp_unsharded_hbf16 rounds every first-layer output h (not Z) to
    bfloat16, to nearest with ties to even.  Identity activation, X = [1],
    W2 = ones: Z is the sum of the rounded h values, known in closed form."""
    h = [1 + 2 ** -8 + 2 ** -10,     # above the midpoint of 1 and 1 + 2^-7: up
         1 + 2 ** -8,                # the midpoint: to even, 1
         1 + 3 * 2 ** -8,            # the midpoint of 1 + 2^-7 and 1 + 2^-6: to even, 1 + 2^-6
         -(1 + 2 ** -8 + 2 ** -10)]  # negative: -(1 + 2^-7)
    X = np.array([[1.0]], dtype=np.float32)
    W1 = np.array([h], dtype=np.float32)
    W2 = np.ones((4, 1), dtype=np.float32)
    Z = oracle.mlp_unsharded_hbf16(X, W1, W2, "identity")
    assert Z[0, 0] == (1 + 2 ** -7) + 1 + (1 + 2 ** -6) - (1 + 2 ** -7)
    # only h is rounded: with one h the rounded Z is that h's rounding
    Z1 = oracle.mlp_unsharded_hbf16(X, W1[:, :1], np.array([[3.0]], dtype=np.float32), "identity")
    assert Z1[0, 0] == 3 * (1 + 2 ** -7)


def test_mlp_hbf16_equals_fp64_h_when_h_is_bf16_exact():
    """Small integer inputs make every h an integer below 256, exact in
    bfloat16: then the two oracles agree exactly, for any W2."""
    rng = np.random.default_rng(4)
    X = rng.integers(-3, 4, size=(6, 8)).astype(np.float32)
    W1 = rng.integers(-3, 4, size=(8, 12)).astype(np.float32)
    W2 = rng.standard_normal((12, 8)).astype(np.float32)
    assert np.array_equal(oracle.mlp_unsharded_hbf16(X, W1, W2, "identity"),
                          oracle.mlp_unsharded(X, W1, W2, "identity"))


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_mlp_hbf16_within_the_rounding_bound(act):
    """Rounding h to bfloat16 moves each h by at most 2^-8 of itself (2^-9
    to float32 and then bfloat16, with a float32 step below that), so the two
    oracles differ by at most 2^-8 (|h| |W2|) elementwise, and do differ."""
    d = mlp_inputs(M=5, H=64, F=256, act=act, dtype="bf16", seed=11)
    Za = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    Zb = oracle.mlp_unsharded_hbf16(d["X"], d["W1"], d["W2"], act)
    h = oracle.colpar_full(d["X"], d["W1"], d["W2"].shape[0], act)
    W2 = (d["W2"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bound = 2.0 ** -8 * (np.abs(h) @ np.abs(W2))
    assert np.all(np.abs(Zb - Za) <= bound)
    assert np.any(Zb != Za)
