"""tp_mlp_forward_noalloc: the forward pass for callers that cannot allocate
device memory during a call (a decode loop under CUDA graph capture or a
real-time scheduler, a runtime that owns all device memory).  Its scratch is
a fixed array inside the library.  Where the AUTO plan's workspace fits it,
it runs the same plan and kernels as tp_mlp_forward with variant AUTO, so
its output must equal that call's bit for bit, call after call, and match
the fp64 oracle within the bf16 tolerance; where it does not, it runs the
plan refitted to the scratch.  Between the two compared calls another shape and other inputs
run through the same scratch, so bytes a call reads without writing them
first would show up as a difference.  This file is collected last so that a
run stopping at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

import oracle
from synth import mlp_inputs
from tests.gpu_util import TOL_BF16_ROW_RMS, rowwise_rms_error, to_device

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20
ACT = {"gelu": 0, "swiglu": 1, "identity": 2}


def _noalloc(lib, s, X, Z, act):
    import torch
    return lib.tp_mlp_forward_noalloc(s.handle, ctypes.c_void_p(X.data_ptr()), X.shape[0], ACT[act],
                                      ctypes.c_void_p(Z.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _problem(tp, act, M, H, F, T, seed):
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=seed, x_rows=max(M, 16))
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    return d, s, to_device(d["X"])


def _run(lib, tp, s, X, act, H):
    import torch
    Z = torch.full((X.shape[0], H), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, s, X, Z, act) == 0
    torch.cuda.synchronize()
    assert tp.tp_last_device_status() == 0
    return Z.cpu().numpy()


@pytest.mark.parametrize("act,M,other", [("swiglu", 16, ("gelu", 200)), ("swiglu", 1, ("gelu", 4)),
                                         ("gelu", 4, ("swiglu", 16)), ("gelu", 200, ("swiglu", 1))])
def test_noalloc_matches_forward_twice(act, M, other):
    import torch
    import linear_sharding_gb300 as tp
    lib = tp.load_library()
    H, F, T = 2048, 7168, 8
    d, s, X = _problem(tp, act, M, H, F, T, seed=31 + M)
    # a different problem through the same scratch: its bytes are what the
    # next call finds there
    d2, s2, X2 = _problem(tp, other[0], other[1], H, F, T, seed=77 + other[1])
    ref = tp.tp_mlp_forward(s, X, variant="auto")
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    Zref = oracle.mlp_unsharded(d["X"][:M], d["W1"], d["W2"], act)
    for _ in range(2):
        _run(lib, tp, s2, X2, other[0], H)
        Z = _run(lib, tp, s, X, act, H)
        assert np.array_equal(Z, ref), "noalloc output differs from tp_mlp_forward (AUTO)"
        err = rowwise_rms_error(Z, Zref)
        print(f"noalloc {act} M={M}: row-RMS err {err:.3e} vs the oracle")
        assert err <= TOL_BF16_ROW_RMS
    s.close()
    s2.close()


def test_noalloc_decode_shape_fits_and_matches():
    """The decode MLP the entry point is sized for (H = 8192, F = 28672,
    T = 8, SwiGLU): at M in {1, 4, 16} its workspace fits the scratch on this
    GPU, and an M = 16 call equals tp_mlp_forward bit for bit."""
    import torch
    import linear_sharding_gb300 as tp
    lib = tp.load_library()
    H, F, T = 8192, 28672, 8
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    W1 = (torch.randn((H, 2 * F), generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    W2 = (torch.randn((F, H), generator=g, device="cuda") * F ** -0.5).to(torch.bfloat16)
    s = tp.tp_shard_weights(W1, W2, T, "swiglu")
    del W1, W2
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M in (1, 4, 16):
        need = tp.tp_mlp_workspace_bytes(s, M)
        print(f"decode M={M}: AUTO workspace {need} bytes on {sms} SMs")
        assert 0 < need <= SCRATCH_BYTES
    X = (torch.randn((16, H), generator=g, device="cuda")).to(torch.bfloat16)
    ref = tp.tp_mlp_forward(s, X, variant="auto")
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    for _ in range(2):
        assert np.array_equal(_run(lib, tp, s, X, "swiglu", H), ref)
    s.close()


def test_noalloc_on_wide_row_parallel_tiles():
    """A prefill shape whose row-parallel GEMM takes the wide tiles (three 256-row blocks,
    H = 8192): the call equals tp_mlp_forward bit for bit, twice, with another shape run
    through the scratch in between."""
    import torch
    import linear_sharding_gb300 as tp
    lib = tp.load_library()
    d, s, X = _problem(tp, "identity", 700, 8192, 1024, 1, seed=91)
    d2, s2, X2 = _problem(tp, "gelu", 16, 2048, 7168, 8, seed=92)
    ref = tp.tp_mlp_forward(s, X, variant="auto")
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    for _ in range(2):
        _run(lib, tp, s2, X2, "gelu", 2048)
        assert np.array_equal(_run(lib, tp, s, X, "identity", 8192), ref)
    s.close()
    s2.close()


def test_noalloc_refits_a_plan_beyond_its_scratch():
    """Where the AUTO plan's workspace exceeds the scratch, the call runs the
    same pass refitted to it: no float32 partials of the second layer (all
    shards summed in one TMEM accumulator) and as many first-layer split-K
    slots as fit.  H = 16384, F = 57344, T = 8, SwiGLU at M = 16 needs about
    41 MiB under AUTO on a 152-SM GB300 (its second layer splits into 32
    partial slots); the refitted plan is then the TMEM-accumulator plan, so
    the call equals tp_mlp_forward(variant "tmem_acc") bit for bit."""
    import torch
    import linear_sharding_gb300 as tp
    lib = tp.load_library()
    H, F, T, M = 16384, 57344, 8, 16
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    W1 = (torch.randn((H, 2 * F), generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    W2 = (torch.randn((F, H), generator=g, device="cuda") * F ** -0.5).to(torch.bfloat16)
    s = tp.tp_shard_weights(W1, W2, T, "swiglu")
    del W1, W2
    torch.cuda.empty_cache()
    need_auto = tp.tp_mlp_workspace_bytes(s, M)
    need_tmem = tp.tp_mlp_workspace_bytes(s, M, "tmem_acc")
    print(f"refit M={M}: AUTO workspace {need_auto} bytes, TMEM accumulator {need_tmem} bytes")
    if need_auto <= SCRATCH_BYTES:
        s.close()
        pytest.skip("the AUTO plan fits the scratch on this GPU: nothing to refit")
    assert 0 < need_tmem <= SCRATCH_BYTES
    X = (torch.randn((M, H), generator=g, device="cuda")).to(torch.bfloat16)
    ref = tp.tp_mlp_forward(s, X, variant="tmem_acc")
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    assert np.isfinite(ref).all()
    for _ in range(2):
        assert np.array_equal(_run(lib, tp, s, X, "swiglu", H), ref)
    s.close()


def test_noalloc_replays_from_a_cuda_graph():
    """The use it exists for: a decode step captured into a CUDA graph with no
    workspace at all (after a first call on the device, as documented), then
    replayed with the input refilled in place; bit-identical to eager calls."""
    import torch
    import linear_sharding_gb300 as tp
    lib = tp.load_library()
    H, F, T, M = 2048, 7168, 8, 16
    d, s, X = _problem(tp, "swiglu", M, H, F, T, seed=71)
    d2 = mlp_inputs(M=M, H=H, F=F, act="swiglu", dtype="bf16", seed=72, x_rows=16)
    X2 = to_device(d2["X"])
    e1 = _run(lib, tp, s, X, "swiglu", H)
    e2 = _run(lib, tp, s, X2, "swiglu", H)
    Xin = X.clone()
    Z = torch.empty((M, H), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        assert _noalloc(lib, s, Xin, Z, "swiglu") == 0
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(Z.cpu().numpy(), e1)
    Xin.copy_(X2)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(Z.cpu().numpy(), e2)
    assert tp.tp_last_device_status() == 0
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
    assert tp.tp_mlp_workspace_bytes(s, M) > SCRATCH_BYTES
    assert _noalloc(lib, s, X, Z, "gelu") == 10  # TP_ERR_WORKSPACE
    s.close()
