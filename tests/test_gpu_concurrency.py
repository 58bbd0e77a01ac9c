"""Calls from several host threads at once, each on its own CUDA stream: the
MLP forward on two handles (a prefill and a decode shape) and the attention
core, each call bit-identical to the same call made alone.  The library's
host side (per-device state, plans, tensor maps, the launch configuration it
caches on first use) must be safe to enter concurrently; the foreign calls
release the interpreter lock, so the threads do run the host code together."""
import threading

import numpy as np
import pytest

from synth import attention_inputs, mlp_inputs
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu


def test_threads_on_their_own_streams_match_single_calls():
    import torch
    import linear_sharding_gb300 as tp
    tp.load_library()
    d1 = mlp_inputs(M=300, H=512, F=2048, act="gelu", dtype="bf16", seed=41)
    d2 = mlp_inputs(M=16, H=512, F=2048, act="swiglu", dtype="bf16", seed=42, x_rows=16)
    da = attention_inputs(700, 3, seed=43)
    s1 = tp.tp_shard_weights(to_device(d1["W1"]), to_device(d1["W2"]), 4, "gelu")
    s2 = tp.tp_shard_weights(to_device(d2["W1"]), to_device(d2["W2"]), 4, "swiglu")
    X1, X2 = to_device(d1["X"]), to_device(d2["X"])
    Q, K, V = to_device(da["Q"]), to_device(da["K"]), to_device(da["V"])
    jobs = {
        "prefill": lambda: tp.tp_mlp_forward(s1, X1, variant="auto"),
        "decode": lambda: tp.tp_mlp_forward(s2, X2, variant="auto"),
        "attention": lambda: tp.tp_attention_forward(Q, K, V, True),
    }
    ref = {}
    for name, fn in jobs.items():
        out = fn()
        torch.cuda.synchronize()
        ref[name] = out.cpu().clone()
    assert tp.tp_last_device_status() == 0
    errors = []

    def worker(name):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(25):
                    out = jobs[name]()
                    st.synchronize()
                    if not torch.equal(out.cpu(), ref[name]):
                        errors.append(f"{name}: differs from the single call")
                        return
        except Exception as e:  # reported below, on the main thread
            errors.append(f"{name}: {e!r}")

    threads = [threading.Thread(target=worker, args=(n,)) for n in jobs for _ in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    torch.cuda.synchronize()
    assert not errors, errors
    assert tp.tp_last_device_status() == 0
    s1.close()
    s2.close()
