"""Parity of the training path (forward that keeps its activations, and the
backward pass) with the fp64 oracle.  The backward oracle is pinned by
central differences of the forward (tests/test_oracle_pins.py).  Tolerance:
the bf16 row-RMS measure of the forward (bf16 operands, float32
accumulation, bf16 dP between the GEMMs)."""
import numpy as np
import pytest

import oracle
from synth import f32_to_bf16_bits, mlp_inputs
from tests.gpu_util import (TOL_BF16_GRAD_ROW_RMS, TOL_BF16_ROW_RMS, bf16_bits, rowwise_rms_error,
                            to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import linear_sharding_gb300 as tp
    tp.load_library()
    return tp


def _bits_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _within_bf16_rounding(got, ref):
    """A stored bf16 tensor: each element within one bf16 rounding (2^-8
    relative) of the fp64 reference, plus 2e-3 of its row's RMS for the float32
    accumulation before the rounding."""
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    return bool(np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-3 * rms))


def _dz(M, H, seed):
    return f32_to_bf16_bits(np.random.default_rng(seed).standard_normal((M, H)).astype(np.float32))


def _run(tp, d, dZ, T, act, variant):
    import torch
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    tp.tp_shards_enable_backward(s, to_device(d["W1"]), to_device(d["W2"]))
    X = to_device(d["X"])
    Z, Hs, Ps = tp.tp_mlp_forward_train(s, X, variant)
    dX, dW1, dW2 = tp.tp_mlp_backward(s, X, Hs, Ps, to_device(dZ), variant)
    torch.cuda.synchronize()
    assert tp.tp_last_device_status() == 0
    return s, Z, Hs, Ps, dX, dW1, dW2


@pytest.mark.parametrize("variant", ["auto", "partials"])
@pytest.mark.parametrize("act,M,H,F,T", [
    ("gelu", 200, 512, 2048, 4),      # CTA-pair tiles, ragged M, 256-wide dH tiles
    ("swiglu", 130, 512, 2048, 4),
    ("identity", 64, 256, 1024, 2),   # single-CTA tiles
    ("gelu", 300, 384, 1152, 3),      # 128-wide tiles everywhere, T = 3
    ("gelu", 96, 256, 768, 2),        # 256-wide weight-gradient tiles that span two shards of 384
    ("swiglu", 160, 256, 1024, 1),    # T = 1: the backward all-reduce sums a single term
])
def test_training_forward_and_backward_small(tp, variant, act, M, H, F, T):
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=M + T)
    dZ = _dz(M, H, seed=M)
    s, Z, Hs, Ps, dX, dW1, dW2 = _run(tp, d, dZ, T, act, variant)
    Fs = F // T
    # forward output and the saved activations
    assert rowwise_rms_error(Z.cpu().numpy(), oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)) <= TOL_BF16_ROW_RMS
    hfull = oracle.colpar_full(d["X"], d["W1"], F, act)
    h = _bits_to_f64(bf16_bits(Hs)).transpose(1, 0, 2).reshape(M, F)
    assert _within_bf16_rounding(h, hfull)
    if act != "identity":
        pre = oracle.linear(d["X"], d["W1"])          # [M x F] or [M x 2F] = [g | u]
        p = _bits_to_f64(bf16_bits(Ps))                 # [parts, T, M, Fs]
        p = np.concatenate([p[k].transpose(1, 0, 2).reshape(M, F) for k in range(p.shape[0])], axis=1)
        assert _within_bf16_rounding(p, pre)
    # gradients
    dx_ref = oracle.mlp_backward_dx(d["X"], d["W1"], d["W2"], dZ, act)
    dw1_ref, dw2_ref = oracle.mlp_backward_dw(d["X"], d["W1"], d["W2"], dZ, act)
    e = [rowwise_rms_error(dX.cpu().numpy(), dx_ref), rowwise_rms_error(dW1.cpu().numpy(), dw1_ref),
         rowwise_rms_error(dW2.cpu().numpy(), dw2_ref)]
    print(f"{act} M={M} T={T} {variant}: dX {e[0]:.3e} dW1 {e[1]:.3e} dW2 {e[2]:.3e}")
    assert max(e) <= TOL_BF16_GRAD_ROW_RMS
    s.close()


def test_backward_requires_enable(tp):
    import torch
    d = mlp_inputs(M=64, H=256, F=1024, act="gelu", dtype="bf16", seed=1)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), 2, "gelu")
    X = to_device(d["X"])
    Z, Hs, Ps = tp.tp_mlp_forward_train(s, X)
    with pytest.raises(tp.TPError):
        tp.tp_mlp_backward(s, X, Hs, Ps, torch.zeros_like(X))


@pytest.mark.parametrize("name", ["prefill_gelu_m2048_h4096_f16384_t4",
                                  "prefill_swiglu_m8192_h8192_f28672_t8_outliers"])
def test_backward_full_size_sampled(tp, name):
    """Full workload sizes: dX on sampled token rows, dW1 columns and dW2 rows
    on sampled FFN indices (every token contributes to those)."""
    import torch
    from synth import WORKLOADS
    w = WORKLOADS[name]
    d = mlp_inputs(M=w["M"], H=w["H"], F=w["F"], act=w["act"], dtype="bf16", seed=0,
                   outlier_frac=w.get("outlier_frac", 0.0), outlier_scale=w.get("outlier_scale", 20.0))
    dZ = _dz(w["M"], w["H"], seed=5)
    s, Z, Hs, Ps, dX, dW1, dW2 = _run(tp, d, dZ, w["T"], w["act"], "auto")
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(w["M"], 8, replace=False))
    fcols = np.sort(rng.choice(w["F"], 8, replace=False))
    dx_ref = oracle.mlp_backward_dx(d["X"], d["W1"], d["W2"], dZ, w["act"], rows=rows)
    err = rowwise_rms_error(dX[torch.from_numpy(rows).cuda()].cpu().numpy(), dx_ref)
    print(f"{name}: dX row-RMS err {err:.3e}")
    assert err <= TOL_BF16_GRAD_ROW_RMS
    dw1_ref, dw2_ref = oracle.mlp_backward_dw(d["X"], d["W1"], d["W2"], dZ, w["act"], fcols=fcols)
    cols = fcols if w["act"] != "swiglu" else np.concatenate([fcols, w["F"] + fcols])
    got1 = dW1[:, torch.from_numpy(cols).cuda()].cpu().numpy()
    got2 = dW2[torch.from_numpy(fcols).cuda()].cpu().numpy()
    e1 = rowwise_rms_error(got1.T, dw1_ref.T)   # per sampled column
    e2 = rowwise_rms_error(got2, dw2_ref)
    print(f"{name}: dW1 col-RMS err {e1:.3e}, dW2 row-RMS err {e2:.3e}")
    assert e1 <= TOL_BF16_GRAD_ROW_RMS and e2 <= TOL_BF16_GRAD_ROW_RMS
    s.close()


@pytest.mark.parametrize("M", [256, 100])   # CTA-pair tiles; single-CTA tiles with a ragged M
def test_activation_gradient_elementwise(tp, M):
    """The dP epilogue element by element.  With H = F, T = 1 and W1 = W2 = I the
    pre-activation is X itself, dH = dZ and dX = dP = bf16(dZ * GeLU'(X)), each a
    single product term, so every element of dX must lie within one bf16 rounding
    of the fp64 oracle's dZ * GeLU'(X).  X spans [-8, 8] on a grid that includes
    0 and -0, where Phi(y) switches between its two forms; dZ is a seeded normal
    draw, so both signs of each factor occur."""
    H = 256
    x = np.linspace(-8.0, 8.0, M * H).astype(np.float32).reshape(M, H)
    x[0, :2] = (0.0, -0.0)
    X = f32_to_bf16_bits(x)
    eye = f32_to_bf16_bits(np.eye(H, dtype=np.float32))
    dZ = _dz(M, H, seed=7 + M)
    d = {"X": X, "W1": eye, "W2": eye}
    s, Z, Hs, Ps, dX, dW1, dW2 = _run(tp, d, dZ, 1, "gelu", "auto")
    ref = oracle.mlp_backward_dx(X, eye, eye, dZ, "gelu")
    got = dX.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(_bits_to_f64(dZ))
    print(f"M={M}: max |dX - ref| / bound = {np.max(err / np.maximum(bound, 1e-30)):.3f}")
    assert np.all(err <= bound)
    s.close()


@pytest.mark.parametrize("M", [256, 100])
def test_swiglu_gradient_elementwise(tp, M):
    """The SwiGLU backward epilogue element by element.  With H = F, T = 1,
    W1 = [I | I] and W2 = I, g = u = X and dH = dZ, so dX = bf16(dZ u SiLU'(g)) +
    bf16(dZ SiLU(g)) summed in float32: each element within one bf16 rounding of
    each of the two terms of the fp64 oracle's dX (the bound takes the terms'
    magnitudes from the logistic function, the oracle gives their sum)."""
    from scipy.special import expit
    H = 256
    x = np.linspace(-12.0, 12.0, M * H).astype(np.float32).reshape(M, H)
    x[0, :2] = (0.0, -0.0)
    X = f32_to_bf16_bits(x)
    eye = np.eye(H, dtype=np.float32)
    W1 = f32_to_bf16_bits(np.concatenate([eye, eye], axis=1))
    W2 = f32_to_bf16_bits(eye)
    dZ = _dz(M, H, seed=11 + M)
    d = {"X": X, "W1": W1, "W2": W2}
    s, Z, Hs, Ps, dX, dW1, dW2 = _run(tp, d, dZ, 1, "swiglu", "auto")
    ref = oracle.mlp_backward_dx(X, W1, W2, dZ, "swiglu")
    got = dX.cpu().numpy().astype(np.float64)
    xv, dz = _bits_to_f64(X), _bits_to_f64(dZ)
    sg = expit(xv)
    terms = np.abs(dz) * (np.abs(xv * sg * (1.0 + xv * (1.0 - sg))) + np.abs(xv * sg))
    bound = 2.0 ** -8 * terms + 1e-6 * np.abs(dz)
    err = np.abs(got - ref)
    print(f"M={M}: max |dX - ref| / bound = {np.max(err / np.maximum(bound, 1e-30)):.3f}")
    assert np.all(err <= bound)
    s.close()
