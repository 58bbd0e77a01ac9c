"""The forward pass can be captured into a CUDA graph and replayed: with a
caller-provided workspace, tp_mlp_forward only enqueues kernels on the
current stream (no allocation, no synchronisation), so a decode loop can
replay one captured step.  The replay must give the same bits as the eager
call, also after the input buffer is refilled in place."""
import numpy as np
import pytest

from synth import mlp_inputs
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import linear_sharding_gb300 as tp
    tp.load_library()
    return tp


@pytest.mark.parametrize("M,H,F,T,act,variant", [
    (16, 1024, 4096, 4, "swiglu", "auto"),      # decode kernels (split-K, weights as the MMA's A)
    (256, 1024, 4096, 4, "gelu", "tmem_acc"),   # CTA-pair prefill tiles
    (256, 1024, 4096, 4, "gelu", "partials"),   # partials + shard-sum
    (700, 8192, 1024, 1, "identity", "tmem_acc"),  # wide row-parallel tiles (tensor maps made per call)
])
def test_forward_replays_from_a_cuda_graph(tp, M, H, F, T, act, variant):
    import torch
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=31, x_rows=max(M, 16))
    d2 = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=32, x_rows=max(M, 16))
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    X, X2 = to_device(d["X"]), to_device(d2["X"])
    ws = torch.empty(max(tp.tp_mlp_workspace_bytes(s, M, variant), 16), dtype=torch.uint8, device="cuda")
    eager1 = tp.tp_mlp_forward(s, X, variant, None, ws).clone()
    eager2 = tp.tp_mlp_forward(s, X2, variant, None, ws).clone()
    torch.cuda.synchronize()
    Xin = X.clone()
    Z = torch.empty((M, H), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tp.tp_mlp_forward(s, Xin, variant, Z, ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Z, eager1)
    Xin.copy_(X2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Z, eager2)
    assert tp.tp_last_device_status() == 0
    s.close()


def test_attention_replays_from_a_cuda_graph(tp):
    """The fused attention core allocates nothing: captured once, replayed
    with Q, K and V refilled in place."""
    import torch
    from synth import attention_inputs
    a1, a2 = attention_inputs(700, 3, seed=51), attention_inputs(700, 3, seed=52)
    Q, K, V = (to_device(a1[k]) for k in "QKV")
    eager1 = tp.tp_attention_forward(Q, K, V, True).clone()
    Q2, K2, V2 = (to_device(a2[k]) for k in "QKV")
    eager2 = tp.tp_attention_forward(Q2, K2, V2, True).clone()
    torch.cuda.synchronize()
    O = torch.empty_like(eager1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tp.tp_attention_forward(Q, K, V, True, O)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(O, eager1)
    Q.copy_(Q2)
    K.copy_(K2)
    V.copy_(V2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(O, eager2)
    assert tp.tp_last_device_status() == 0


def test_block_replays_from_a_cuda_graph(tp):
    """One transformer block with a caller-provided workspace, captured once
    and replayed with the input refilled in place."""
    import torch
    from tests.test_gpu_block import _weights
    M, nh, T, act = 300, 4, 2, "swiglu"
    H, F = nh * 128, 4 * nh * 128
    d = _weights(M, H, F, act, seed=61)
    d2 = _weights(M, H, F, act, seed=62)
    a = tp.tp_shard_weights_qkv(to_device(d["Wqkv"]), to_device(d["Wo"]), nh, 128, T)
    m = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    ws = torch.empty(max(tp.tp_block_workspace_bytes(a, m, M), 16), dtype=torch.uint8, device="cuda")
    X, X2 = to_device(d["X"]), to_device(d2["X"])
    e1, _ = tp.tp_block_forward(a, m, X, workspace=ws)
    e1 = e1.clone()
    e2, _ = tp.tp_block_forward(a, m, X2, workspace=ws)
    e2 = e2.clone()
    torch.cuda.synchronize()
    Xin = X.clone()
    out = torch.empty((M, H), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tp.tp_block_forward(a, m, Xin, out=out, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, e1)
    Xin.copy_(X2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, e2)
    assert tp.tp_last_device_status() == 0
    a.close()
    m.close()


def test_training_step_replays_from_a_cuda_graph(tp):
    """A training step (the forward that keeps its activations, then the
    backward) captured once: the binding's buffers come from the graph's
    memory pool and the library allocates nothing.  Replayed with X and dZ
    refilled in place, each gradient is bit-identical to the eager step."""
    import torch
    from synth import f32_to_bf16_bits
    M, H, F, T, act = 256, 512, 2048, 4, "swiglu"
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=81)
    d2 = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=82)
    rng = np.random.default_rng(83)
    dz1 = to_device(f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32)))
    dz2 = to_device(f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32)))
    sh = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    tp.tp_shards_enable_backward(sh, to_device(d["W1"]), to_device(d["W2"]))
    X1, X2 = to_device(d["X"]), to_device(d2["X"])

    def step(X, dZ):
        Z, Hs, Ps = tp.tp_mlp_forward_train(sh, X)
        return (Z,) + tuple(tp.tp_mlp_backward(sh, X, Hs, Ps, dZ))

    eager1 = [t.clone() for t in step(X1, dz1)]
    eager2 = [t.clone() for t in step(X2, dz2)]
    torch.cuda.synchronize()
    Xin, dZin = X1.clone(), dz1.clone()
    step(Xin, dZin)  # warm the allocator outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = step(Xin, dZin)
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(o, e) for o, e in zip(outs, eager1))
    Xin.copy_(X2)
    dZin.copy_(dz2)
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(o, e) for o, e in zip(outs, eager2))
    assert tp.tp_last_device_status() == 0
    sh.close()
