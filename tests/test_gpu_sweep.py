"""Seeded random sweeps over the shapes the API accepts: the fused attention
core and the MLP forward, each case against the fp64 oracle on a few sampled
rows (always the first and the last).  The fixed parity cases pin chosen
tile boundaries; these cover the combinations between them (ragged M of
every size class, shard counts, head counts, causal or not, every all-reduce
variant, score scales that make the online softmax raise its shift), and
would show a barrier-phase or work-split slip that only some shapes reach.
Same tolerances as the fixed cases."""
import numpy as np
import pytest

import oracle
from synth import attention_inputs, mlp_inputs
from tests.gpu_util import (GRAD_MIN_TOKENS, TOL_ATTN_ELEMENT, TOL_BF16_GRAD_ROW_RMS, TOL_BF16_ROW_RMS,
                            attention_elementwise_ok, rowwise_rms_error, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import linear_sharding_gb300 as tp
    tp.load_library()
    return tp


def _rows(rng, M, k=4):
    rows = {0, M - 1}
    rows.update(int(r) for r in rng.integers(0, M, size=k))
    return np.array(sorted(rows), dtype=np.int64)


def test_attention_random_shapes(tp):
    import torch
    rng = np.random.default_rng(2024)
    for case in range(200):
        M = int(rng.integers(1, 2049))
        nh = int(rng.integers(1, 9))
        causal = bool(rng.integers(0, 2))
        q_scale = float(rng.choice([0.5, 1.0, 2.0, 3.0]))
        d = attention_inputs(M, nh, seed=case, q_scale=q_scale)
        O = tp.tp_attention_forward(to_device(d["Q"]), to_device(d["K"]), to_device(d["V"]), causal)
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0, (M, nh, causal)
        rows = _rows(rng, M)
        got = (O[torch.from_numpy(rows).cuda()].cpu().view(torch.int16).numpy().view(np.uint16)
               .astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ref = oracle.attention(d["Q"], d["K"], d["V"], causal, rows=rows)
        e, el = rowwise_rms_error(got, ref), attention_elementwise_ok(got, ref)
        assert e <= TOL_BF16_GRAD_ROW_RMS and el <= TOL_ATTN_ELEMENT, (case, M, nh, causal, q_scale, e, el)


def test_mlp_random_shapes(tp):
    import torch
    rng = np.random.default_rng(2025)
    for case in range(120):
        act = str(rng.choice(["gelu", "swiglu", "identity"]))
        T = int(rng.choice([1, 2, 3, 4, 8]))
        Fs = 128 * int(rng.integers(1, 5))
        H = 128 * int(rng.integers(2, 9))
        M = int(rng.choice([int(rng.integers(1, 17)), int(rng.integers(17, 1200))]))
        variant = str(rng.choice(["auto", "partials", "tmem_acc"]))
        d = mlp_inputs(M=M, H=H, F=Fs * T, act=act, dtype="bf16", seed=case, x_rows=max(M, 16))
        s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
        Z = tp.tp_mlp_forward(s, to_device(d["X"][:M]), variant=variant)
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0, (act, M, H, Fs, T, variant)
        rows = _rows(rng, M)
        got = Z[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
        ref = oracle.mlp_unsharded(d["X"][:M], d["W1"], d["W2"], act, rows=rows)
        e = rowwise_rms_error(got, ref)
        assert e <= TOL_BF16_ROW_RMS, (case, act, M, H, Fs, T, variant, e)
        s.close()


def test_training_backward_random_shapes(tp):
    """The training forward and the backward (dX, dW1, dW2) on random shapes,
    every element against the fp64 backward oracle (token counts from
    GRAD_MIN_TOKENS up, the domain of the gradient bound)."""
    import torch
    from synth import f32_to_bf16_bits
    rng = np.random.default_rng(2026)
    for case in range(30):
        act = str(rng.choice(["gelu", "swiglu", "identity"]))
        T = int(rng.choice([1, 2, 3, 4]))
        Fs = 128 * int(rng.integers(1, 4))
        H = 128 * int(rng.integers(2, 5))
        M = int(rng.integers(GRAD_MIN_TOKENS, 401))
        variant = str(rng.choice(["auto", "partials"]))
        d = mlp_inputs(M=M, H=H, F=Fs * T, act=act, dtype="bf16", seed=100 + case)
        dZ = f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
        s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
        tp.tp_shards_enable_backward(s, to_device(d["W1"]), to_device(d["W2"]))
        X = to_device(d["X"])
        Z, Hs, Ps = tp.tp_mlp_forward_train(s, X, variant)
        dX, dW1, dW2 = tp.tp_mlp_backward(s, X, Hs, Ps, to_device(dZ), variant)
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0, (act, M, H, Fs, T, variant)
        dx_ref = oracle.mlp_backward_dx(d["X"], d["W1"], d["W2"], dZ, act)
        dw1_ref, dw2_ref = oracle.mlp_backward_dw(d["X"], d["W1"], d["W2"], dZ, act)
        e = max(rowwise_rms_error(dX.cpu().numpy(), dx_ref), rowwise_rms_error(dW1.cpu().numpy(), dw1_ref),
                rowwise_rms_error(dW2.cpu().numpy(), dw2_ref))
        assert e <= TOL_BF16_GRAD_ROW_RMS, (case, act, M, H, Fs, T, variant, e)
        s.close()


def test_block_random_shapes(tp):
    """One transformer block (QKV, attention, O-projection with its residual,
    the MLP with its residual) on random shapes, sampled rows against the
    block oracle."""
    from tests.test_gpu_block import _check, _weights
    rng = np.random.default_rng(2027)
    for case in range(16):
        nh = int(rng.choice([1, 2, 3, 4, 6, 8]))
        T = int(rng.choice([t for t in (1, 2, 3, 4, 8) if nh % t == 0]))
        H = nh * 128
        F = 128 * int(rng.integers(1, 5)) * T
        M = int(rng.integers(2, 701))
        act = str(rng.choice(["gelu", "swiglu", "identity"]))
        causal = bool(rng.integers(0, 2))
        variant = str(rng.choice(["auto", "partials", "tmem_acc"]))
        d = _weights(M, H, F, act, seed=300 + case)
        _check(tp, d, M, H, F, nh, 128, T, act, causal, variant, _rows(rng, M, k=6))
