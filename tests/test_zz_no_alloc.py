"""tp_mlp_forward_noalloc: the forward pass for callers that cannot allocate
device memory during a call (a decode loop under CUDA graph capture or a
real-time scheduler, a runtime that owns all device memory).  Its scratch is
a fixed array inside the library; the output must match tp_mlp_forward's on
the same inputs, call after call.  This file is collected last so that a run
stopping at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

from synth import mlp_inputs
from tests.gpu_util import TOL_BF16_ROW_RMS, rowwise_rms_error, to_device

pytestmark = pytest.mark.gpu


def _noalloc(lib, s, X, Z, act):
    import torch
    return lib.tp_mlp_forward_noalloc(s.handle, ctypes.c_void_p(X.data_ptr()), X.shape[0],
                                      {"gelu": 0, "swiglu": 1, "identity": 2}[act],
                                      ctypes.c_void_p(Z.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("act,M", [("swiglu", 16), ("swiglu", 1), ("gelu", 4), ("gelu", 200)])
def test_noalloc_matches_forward_twice(act, M):
    import torch
    import linear_sharding_gb300 as tp
    lib = tp.load_library()
    H, F, T = 2048, 7168, 8
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=31 + M, x_rows=max(M, 16))
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    X = to_device(d["X"])
    ref = tp.tp_mlp_forward(s, X, variant="auto")
    torch.cuda.synchronize()
    ref = ref.cpu().numpy().astype(np.float64)
    for _ in range(2):
        Z = torch.full((M, H), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, s, X, Z, act) == 0
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0
        assert rowwise_rms_error(Z.cpu().numpy(), ref) <= TOL_BF16_ROW_RMS
    s.close()


def test_noalloc_rejects_work_beyond_its_scratch():
    import torch
    import linear_sharding_gb300 as tp
    lib = tp.load_library()
    M, H, F, T = 2048, 1024, 8192, 4  # Y alone is 32 MiB: over the limit
    d = mlp_inputs(M=M, H=H, F=F, act="gelu", dtype="bf16", seed=3)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "gelu")
    X = to_device(d["X"])
    Z = torch.empty((M, H), dtype=torch.float32, device="cuda")
    assert tp.tp_mlp_workspace_bytes(s, M) > 16 << 20
    assert _noalloc(lib, s, X, Z, "gelu") == 10  # TP_ERR_WORKSPACE
    s.close()
