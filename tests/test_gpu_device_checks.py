"""The debug library (libtpmlp_debug.so: the kernels' device-side index
checks compiled in with -DTP_DEVICE_CHECKS=1) runs every main path on small
ragged shapes with no check firing (the status word stays clear), and gives
the same bits as the normal library: the checks observe, they do not change
the arithmetic.  This stands in for a memory checker, which this pool does
not offer: a check that fails is reported, and its access skipped, instead of
faulting."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import linear_sharding_gb300 as tp
from synth import attention_inputs, f32_to_bf16_bits, mlp_inputs, partials_inputs
from tests.gpu_util import bf16_bits, to_device

tp.load_library(sys.argv[2])
out, status = {}, {}

def done(name, *tensors):
    torch.cuda.synchronize()
    status[name] = tp.tp_last_device_status()
    for i, t in enumerate(tensors):
        out[f"{name}_{i}"] = (bf16_bits(t) if t.dtype == torch.bfloat16 else t.detach().cpu().numpy())

d = mlp_inputs(M=300, H=512, F=2048, act="gelu", dtype="bf16", seed=1, x_rows=300)
s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), 4, "gelu")
X = to_device(d["X"])
for v in ("tmem_acc", "partials", "auto"):
    done("mlp_" + v, tp.tp_mlp_forward(s, X, v))
W1, W2 = to_device(d["W1"]), to_device(d["W2"])
tp.tp_shards_enable_backward(s, W1, W2)
Z, Hs, Ps = tp.tp_mlp_forward_train(s, X)
dZ = to_device(mlp_inputs(M=300, H=512, F=2048, act="gelu", dtype="bf16", seed=2, x_rows=300)["X"])
done("train", Z, Hs, Ps, *tp.tp_mlp_backward(s, X, Hs, Ps, dZ))
s.close()

# the row-parallel GEMM on wide tiles (three 256-row blocks, H = 8192: 352- and 320-column tiles)
d = mlp_inputs(M=700, H=8192, F=1024, act="identity", dtype="bf16", seed=8, x_rows=700)
s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), 1, "identity")
done("mlp_wide", tp.tp_mlp_forward(s, to_device(d["X"]), "tmem_acc"))
s.close()

d = mlp_inputs(M=3, H=512, F=2048, act="swiglu", dtype="bf16", seed=3, x_rows=16)
s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), 4, "swiglu")
done("decode", tp.tp_mlp_forward(s, to_device(d["X"])))
s.close()

d = mlp_inputs(M=37, H=96, F=240, act="gelu", dtype="f32", seed=4, x_rows=37)
s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), 3, "gelu")
done("f32", tp.tp_mlp_forward(s, to_device(d["X"])))
s.close()

a = attention_inputs(300, 3, seed=5)
Q, K, V = (to_device(a[k]) for k in ("Q", "K", "V"))
done("attn_causal", tp.tp_attention_forward(Q, K, V, True))
done("attn_full", tp.tp_attention_forward(Q, K, V, False))

rng = np.random.default_rng(6)
H, nh, F = 512, 4, 2048
draw = lambda shape, std: to_device(f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32)))
qa = tp.tp_shard_weights_qkv(draw((H, 3 * H), H ** -0.5), draw((H, H), H ** -0.5), nh, 128, 2)
mm = tp.tp_shard_weights(draw((H, 2 * F), H ** -0.5), draw((F, H), F ** -0.5), 2, "swiglu")
Xb = draw((300, H), 1.0)
done("block", *tp.tp_block_forward(qa, mm, Xb, causal=True, h_out=True))
qa.close()
mm.close()

P = [torch.from_numpy(p).cuda() for p in partials_inputs(3, 1001, seed=7)]
done("partial_sum", tp.tp_partial_sum(P))
np.savez(sys.argv[3], **out)
print("STATUS", " ".join(f"{k}={v}" for k, v in status.items()))
sys.exit(0 if all(v == 0 for v in status.values()) else 3)
"""


def _run(lib, path):
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT, lib, path], capture_output=True, text=True,
                       cwd=ROOT, timeout=900)
    print(r.stdout[-2000:], r.stderr[-2000:])
    return r.returncode


def test_debug_library_runs_clean_and_matches(tmp_path):
    from linear_sharding_gb300 import build as b
    debug_lib = b.build(debug=True)
    normal_lib = b.LIB
    assert os.path.exists(normal_lib)
    assert _run(debug_lib, str(tmp_path / "debug.npz")) == 0, "a device-side check fired (or a call failed)"
    assert _run(normal_lib, str(tmp_path / "normal.npz")) == 0
    dbg, ref = np.load(tmp_path / "debug.npz"), np.load(tmp_path / "normal.npz")
    assert sorted(dbg.files) == sorted(ref.files)
    for k in ref.files:
        assert np.array_equal(dbg[k], ref[k], equal_nan=True), f"{k} differs between the debug and normal builds"
