"""Parity of one tensor-parallel transformer block (head-sharded causal
attention + MLP, two all-reduce-sums, residuals) with the fp64 oracle, on
sampled token rows.  Tolerance: row-RMS of the residual stream h and of the
output (2e-2), and of the attention and MLP contributions alone (h - X,
out - h), which pass through more bf16 roundings (Q, K, V, the
probabilities, O; h and Y), held to the training bound 3e-2."""
import numpy as np
import pytest

import oracle
from synth import f32_to_bf16_bits
from tests.gpu_util import (TOL_BF16_GRAD_ROW_RMS, TOL_BF16_ROW_RMS, rowwise_rms_error, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import linear_sharding_gb300 as tp
    tp.load_library()
    return tp


def _weights(M, H, F, act, seed):
    rng = np.random.default_rng(seed)
    ncols = 2 * F if act == "swiglu" else F
    draw = lambda shape, std: f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))  # noqa: E731
    return dict(X=draw((M, H), 1.0), Wqkv=draw((H, 3 * H), H ** -0.5), Wo=draw((H, H), H ** -0.5),
                W1=draw((H, ncols), H ** -0.5), W2=draw((F, H), F ** -0.5))


def _check(tp, d, M, H, F, nh, hd, T, act, causal, variant, rows):
    import torch
    a = tp.tp_shard_weights_qkv(to_device(d["Wqkv"]), to_device(d["Wo"]), nh, hd, T)
    m = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    X = to_device(d["X"])
    out, h = tp.tp_block_forward(a, m, X, causal=causal, variant=variant, h_out=True)
    torch.cuda.synchronize()
    assert tp.tp_last_device_status() == 0
    ref_out, ref_h = oracle.block_forward(d["X"], d["Wqkv"], d["Wo"], d["W1"], d["W2"], nh, hd, T, act,
                                          causal=causal, sharded=True, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    o, hh = out[idx].cpu().numpy(), h[idx].cpu().numpy()
    x = (d["X"][rows].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    e = dict(h=rowwise_rms_error(hh, ref_h), out=rowwise_rms_error(o, ref_out),
             attn=rowwise_rms_error(hh - x, ref_h - x), mlp=rowwise_rms_error(o - hh, ref_out - ref_h))
    print(f"block M={M} H={H} T={T} {act} causal={causal} {variant}: " +
          " ".join(f"{k} {v:.3e}" for k, v in e.items()))
    assert e["h"] <= TOL_BF16_ROW_RMS and e["out"] <= TOL_BF16_ROW_RMS
    assert e["attn"] <= TOL_BF16_GRAD_ROW_RMS and e["mlp"] <= TOL_BF16_GRAD_ROW_RMS
    a.close()
    m.close()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("act,M,nh,T,variant", [
    ("gelu", 300, 4, 2, "auto"),      # ragged M: 300 keys, scores padded to 512
    ("swiglu", 256, 4, 4, "partials"),
    ("gelu", 100, 2, 2, "tmem_acc"),  # single-CTA tiles everywhere
    ("swiglu", 200, 2, 1, "auto"),    # T = 1: one shard, both all-reduces sum a single term
])
def test_block_small(tp, causal, act, M, nh, T, variant):
    hd = 128
    H, F = nh * hd, 4 * nh * hd
    d = _weights(M, H, F, act, seed=M + nh)
    rows = np.unique(np.concatenate([[0, 1, M - 1], np.random.default_rng(1).choice(M, 10, replace=False)]))
    _check(tp, d, M, H, F, nh, hd, T, act, causal, variant, rows)


def test_block_attention_projection_workload(tp):
    """The attention-projection workload's shapes (M = 4096 tokens, 32 heads
    of 128, T = 8) with a SwiGLU MLP of F = 4H, rows sampled across all 4096
    tokens, the last one included: late queries attend over up to 4096 keys
    (the oracle then needs K and V of every token)."""
    M, nh, hd, T = 4096, 32, 128, 8
    H, F = nh * hd, 4 * nh * hd
    d = _weights(M, H, F, "swiglu", seed=7)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, 127, 128, 511, 2047, 2048, 4094, 4095],
                                     rng.choice(M, 8, replace=False)]))
    _check(tp, d, M, H, F, nh, hd, T, "swiglu", True, "auto", rows)
