"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases are compared element by element at sizes that span several
128 x 256 tiles and a ragged tail; the full-size workloads are compared on
sampled output rows (each row of Z depends only on that row of X).  The
shard layout and the shard-sum are bit exact; outputs are within the stated
tolerances (tests/gpu_util.py)."""
import numpy as np
import pytest

import oracle
from synth import WORKLOADS, attn_inputs, mlp_inputs, partials_inputs
from tests.gpu_util import (TOL_BF16_ROW_RMS, BF16H_ERROR_RATIO, TOL_F32_NORMWISE, bf16_bits, global_rms_error,
                            normwise_error, rowwise_rms_error, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import torch
    import linear_sharding_gb300 as tp
    tp.load_library()
    assert torch.cuda.is_available()
    return tp


def _sync():
    import torch
    torch.cuda.synchronize()


# ---- shard layout (bit exact) ---------------------------------------------------

@pytest.mark.parametrize("act,dtype,T", [("gelu", "bf16", 4), ("swiglu", "bf16", 2),
                                         ("identity", "f32", 2), ("gelu", "f32", 8),
                                         ("swiglu", "f32", 1)])
def test_shard_layout_bit_exact(tp, act, dtype, T):
    H, F = 256, 128 * T * 2
    d = mlp_inputs(M=1, H=H, F=F, act=act, dtype=dtype, seed=1)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    for i in range(T):
        assert np.array_equal(tp.tp_shard_get(s, i, 0), oracle.shard_w1(d["W1"], F, T, act, i, 0))
        if act == "swiglu":
            assert np.array_equal(tp.tp_shard_get(s, i, 1), oracle.shard_w1(d["W1"], F, T, act, i, 1))
        assert np.array_equal(tp.tp_shard_get(s, i, 2), oracle.shard_w2(d["W2"], T, i))


def test_qkv_shard_layout_bit_exact(tp):
    nh, hd, T, H = 8, 64, 4, 512
    d = attn_inputs(M=1, H=H, n_heads=nh, head_dim=hd, seed=2)
    s = tp.tp_shard_weights_qkv(to_device(d["Wqkv"]), to_device(d["Wo"]), nh, hd, T)
    for i in range(T):
        assert np.array_equal(tp.tp_shard_get(s, i, 0), oracle.shard_wqkv(d["Wqkv"], nh, hd, T, i))
        assert np.array_equal(tp.tp_shard_get(s, i, 2), oracle.shard_wo(d["Wo"], nh, hd, T, i))


# ---- shard-sum (bit exact against the ascending-order float32 sum) -------------

@pytest.mark.parametrize("T,n", [(1, 1000), (2, 4099), (3, 77777), (4, 1 << 20), (5, 12345),
                                 (8, 1000003), (16, 65536), (11, 3)])
def test_partial_sum_bit_exact(tp, T, n):
    P = partials_inputs(T, n, seed=T)
    parts = [to_device(P[t]) for t in range(T)]
    Z = tp.tp_partial_sum(parts)
    _sync()
    assert np.array_equal(Z.cpu().numpy(), oracle.partial_sum_f32(P))
    # in place into the first partial
    tp.tp_partial_sum(parts, Z=parts[0])
    _sync()
    assert np.array_equal(parts[0].cpu().numpy(), oracle.partial_sum_f32(P))


def test_partial_sum_unaligned_scalar_path(tp):
    """Pointers that are 4- but not 16-byte aligned take the scalar path."""
    import torch
    T, n = 4, 5001
    P = partials_inputs(T, n + 1, seed=7)
    parts = [to_device(P[t])[1:] for t in range(T)]
    Z = torch.empty(n + 1, dtype=torch.float32, device="cuda")[1:]
    tp.tp_partial_sum(parts, Z=Z)
    _sync()
    assert np.array_equal(Z.cpu().numpy(), oracle.partial_sum_f32(P[:, 1:]))


def test_partial_sum_empty_is_noop(tp):
    import torch
    z = torch.full((4,), 7.0, device="cuda")
    tp.tp_partial_sum([z[:0], z[:0]], Z=z[:0])
    _sync()
    assert torch.all(z == 7.0)


# ---- MLP parity, small shapes (every element) ------------------------------------

def _run_mlp(tp, d, T, act, variant, M=None):
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    X = to_device(d["X"])
    Z = tp.tp_mlp_forward(s, X, variant=variant)
    _sync()
    assert tp.tp_last_device_status() == 0
    return Z.cpu().numpy()


@pytest.mark.parametrize("variant", ["partials", "tmem_acc", "auto"])
@pytest.mark.parametrize("act,M,H,F,T", [
    ("gelu", 300, 512, 2048, 4),      # ragged M (300 = 2 x 128 + 44), 2 x 2 x 4 tiles
    ("swiglu", 200, 512, 2048, 8),    # Fs = 256: one gate/up tile per shard
    ("identity", 129, 256, 1024, 2),  # one row into the second M tile
    ("gelu", 517, 384, 1152, 3),      # T = 3, 128-wide tiles in both GEMMs (Fs = H = 384)
    ("swiglu", 260, 512, 1024, 1),    # T = 1: one shard, the all-reduce sums a single term
    ("gelu", 12, 256, 1024, 1),       # T = 1 on the decode path
    ("gelu", 200, 256, 2048, 16),     # T = 16 shards of 128 columns
])
def test_mlp_bf16_small(tp, variant, act, M, H, F, T):
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=M)
    Z = _run_mlp(tp, d, T, act, variant)
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    err = rowwise_rms_error(Z, Zref)
    assert err <= TOL_BF16_ROW_RMS
    assert rowwise_rms_error(Z, oracle.mlp_unsharded_hbf16(d["X"], d["W1"], d["W2"], act)) <= BF16H_ERROR_RATIO * err


def _bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bit patterns, rounding the float32 value to nearest even."""
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_gelu_epilogue_is_exact_erf_gelu_to_bf16(tp):
    """With W1 = I the column-parallel GEMM's output is bf16(GeLU(x)) of each input x (x * 1
    accumulates exactly), so this checks the epilogue's erf ("Tensor Parallelism in Action",
    section 1: Y_i = GeLU(X A_i), erf form) against the fp64 oracle's GeLU over [-8, 8]: each
    output within one bfloat16 step of the exact value, or 1e-6 in the far negative tail.
    M = 384 is one and a half 256-row CTA-pair tiles, so the tile stores clip a tail."""
    M, H = 384, 256
    xb = _bf16_round_bits(np.linspace(-8.0, 8.0, M * H)).reshape(M, H)
    eye = np.zeros((H, H), dtype=np.uint16)
    eye[np.arange(H), np.arange(H)] = 0x3F80  # bfloat16 1.0
    s = tp.tp_shard_weights(to_device(eye), to_device(eye), 1, "gelu")
    Y = tp.tp_colpar_forward(s, to_device(xb))
    _sync()
    got = (bf16_bits(Y[0]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = np.array([oracle.gelu(v) for v in x.ravel()]).reshape(M, H)
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    err = np.abs(got - ref)
    assert np.all(err <= step + 1e-6), float(np.max(err - step))


@pytest.mark.parametrize("variant", ["partials", "tmem_acc", "auto"])
@pytest.mark.parametrize("act", ["gelu", "swiglu", "identity"])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_mlp_bf16_decode_small(tp, variant, act, M):
    """M <= 16 takes the decode kernels (weights as the 128-row MMA operand)."""
    H, F, T = 512, 2048, 4
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=100 + M, x_rows=16)
    Z = _run_mlp(tp, d, T, act, variant)
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    err = rowwise_rms_error(Z, Zref)
    assert err <= TOL_BF16_ROW_RMS
    assert rowwise_rms_error(Z, oracle.mlp_unsharded_hbf16(d["X"], d["W1"], d["W2"], act)) <= BF16H_ERROR_RATIO * err


@pytest.mark.parametrize("variant", ["partials", "tmem_acc"])
@pytest.mark.parametrize("act", ["gelu", "swiglu", "identity"])
def test_mlp_f32_tiny(tp, variant, act):
    """The float32 path (CUDA-core FMA) at the tiny workload's shape."""
    w = WORKLOADS["tiny_fp32_gelu"]
    F = w["F"] if act != "swiglu" else 256
    d = mlp_inputs(M=w["M"], H=w["H"], F=F, act=act, dtype="f32", seed=0)
    Z = _run_mlp(tp, d, w["T"], act, variant)
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    assert normwise_error(Z, Zref) <= TOL_F32_NORMWISE


def test_tiny_fp32_workload_exact_recipe(tp):
    """X[8x64], W1[64x256], W2[256x64], T = 2, erf-GeLU, seed 0; also checks
    sharded == unsharded on the oracle side."""
    w = WORKLOADS["tiny_fp32_gelu"]
    d = mlp_inputs(M=w["M"], H=w["H"], F=w["F"], act="gelu", dtype="f32", seed=0)
    Zu = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")
    Zs = oracle.mlp_sharded(d["X"], d["W1"], d["W2"], w["T"], "gelu")
    assert normwise_error(Zs, Zu) <= 1e-12
    for variant in ("partials", "tmem_acc", "auto"):
        Z = _run_mlp(tp, d, w["T"], "gelu", variant)
        assert normwise_error(Z, Zu) <= TOL_F32_NORMWISE


def test_mlp_f32_ragged_general(tp):
    M, H, F, T = 37, 96, 240, 3
    d = mlp_inputs(M=M, H=H, F=F, act="gelu", dtype="f32", seed=5)
    for variant in ("partials", "tmem_acc"):
        Z = _run_mlp(tp, d, T, "gelu", variant)
        assert normwise_error(Z, oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")) <= TOL_F32_NORMWISE


def test_attn_proj_small(tp):
    M, nh, hd, T = 300, 8, 64, 4
    H = nh * hd
    d = attn_inputs(M=M, H=H, n_heads=nh, head_dim=hd, seed=3)
    s = tp.tp_shard_weights_qkv(to_device(d["Wqkv"]), to_device(d["Wo"]), nh, hd, T)
    X, A = to_device(d["X"]), to_device(d["A"])
    Zref = oracle.oproj_sharded(d["A"], d["Wo"], nh, hd, T)
    for variant in ("partials", "tmem_acc", "auto"):
        QKV, Z = tp.tp_attn_proj_forward(s, X=X, A=A, variant=variant)
        _sync()
        assert tp.tp_last_device_status() == 0
        assert rowwise_rms_error(Z.cpu().numpy(), Zref) <= TOL_BF16_ROW_RMS
        q = bf16_bits(QKV)
        for i in range(T):
            ref = oracle.qkv_shard(d["X"], d["Wqkv"], nh, hd, T, i)
            got = (q[i].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            assert rowwise_rms_error(got, ref) <= TOL_BF16_ROW_RMS


# ---- edge cases ---------------------------------------------------------------------

def test_mlp_edge_cases(tp):
    import torch
    H, F, T = 256, 1024, 4
    d = mlp_inputs(M=8, H=H, F=F, act="gelu", dtype="bf16", seed=9)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "gelu")
    # M = 0 is a no-op
    Z0 = tp.tp_mlp_forward(s, to_device(d["X"])[:0])
    assert Z0.shape == (0, H)
    # workspace too small
    X = to_device(d["X"])
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_mlp_forward(s, X, variant="partials", workspace=ws)
    assert e.value.code == 10
    # the activation must match the shards' packing
    with pytest.raises(tp.TPError):
        tp.tp_mlp_forward(s, X, act="swiglu")
    # an explicit workspace of the stated size works and matches
    need = tp.tp_mlp_workspace_bytes(s, X.shape[0], "partials")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    Z = tp.tp_mlp_forward(s, X, variant="partials", workspace=ws)
    _sync()
    assert rowwise_rms_error(Z.cpu().numpy(),
                             oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")) <= TOL_BF16_ROW_RMS
    # indivisible and unsupported shapes
    with pytest.raises(tp.TPError) as e:
        tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), 3, "gelu")
    assert e.value.code == 2


def test_variants_agree_and_are_deterministic(tp):
    """Both all-reduce variants are correct; each is run-to-run bit identical."""
    M, H, F, T = 256, 512, 2048, 4
    d = mlp_inputs(M=M, H=H, F=F, act="gelu", dtype="bf16", seed=21)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "gelu")
    X = to_device(d["X"])
    outs = {}
    for v in ("partials", "tmem_acc"):
        a = tp.tp_mlp_forward(s, X, variant=v).cpu().numpy()
        b = tp.tp_mlp_forward(s, X, variant=v).cpu().numpy()
        assert np.array_equal(a, b)
        outs[v] = a
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")
    for v in outs:
        assert rowwise_rms_error(outs[v], Zref) <= TOL_BF16_ROW_RMS


def test_machine_balance_steers_the_auto_plan(tp):
    """tp_set_machine_balance: with partial traffic nearly free (1e-3 flop per
    byte) AUTO splits the row-parallel GEMM over float32 partials (a larger
    workspace); with it dear (1e5) it keeps one TMEM accumulator.  Either
    plan's output stays within tolerance of the oracle; 0 restores the
    device's own figure."""
    M, H, F, T = 256, 512, 2048, 4  # 4 output tiles of 128 x 256: few waves, long K per tile
    d = mlp_inputs(M=M, H=H, F=F, act="gelu", dtype="bf16", seed=23)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "gelu")
    X = to_device(d["X"])
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")
    y_bytes = T * M * (F // T) * 2
    sizes = {}
    try:
        for bal in (1e-3, 1e5):
            tp.tp_set_machine_balance(bal)
            sizes[bal] = tp.tp_mlp_workspace_bytes(s, M, "auto")
            Z = tp.tp_mlp_forward(s, X, variant="auto").cpu().numpy()
            assert tp.tp_last_device_status() == 0
            assert rowwise_rms_error(Z, Zref) <= TOL_BF16_ROW_RMS
    finally:
        tp.tp_set_machine_balance(0)
    assert sizes[1e-3] >= y_bytes + 2 * M * H * 4  # at least two float32 partial slots
    assert sizes[1e5] == (y_bytes + 255) // 256 * 256  # Y alone: one accumulator
    with pytest.raises(tp.TPError):
        tp.tp_set_machine_balance(-1.0)
    s.close()


def test_host_buffer_forward(tp):
    """tp_mlp_forward_host: pinned host X in, host Z out, same result."""
    import torch
    M, H, F, T = 64, 256, 1024, 2
    d = mlp_inputs(M=M, H=H, F=F, act="swiglu", dtype="bf16", seed=4)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "swiglu")
    Xh = torch.from_numpy(d["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    Zh = torch.empty((M, H), dtype=torch.float32).pin_memory()
    ws = torch.empty(tp.tp_mlp_host_workspace_bytes(s, M), dtype=torch.uint8, device="cuda")
    tp.tp_mlp_forward_host(s, Xh, Zh, ws)
    _sync()
    Zd = tp.tp_mlp_forward(s, to_device(d["X"])).cpu().numpy()
    assert np.array_equal(Zh.numpy(), Zd)


@pytest.mark.parametrize("M", [256, 64, 4])  # CTA-pair tiles, single-CTA tiles, decode
def test_wait_timeout_reports_and_recovers(tp, M):
    """A wait limit of 1 ns makes the GEMM's waits run out: the kernels return
    early, the status says TP_ERR_TIMEOUT, nothing faults, and the next call
    with the default limit is correct."""
    H, F, T = 512, 2048, 4
    d = mlp_inputs(M=M, H=H, F=F, act="gelu", dtype="bf16", seed=8, x_rows=max(M, 16))
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "gelu")
    X = to_device(d["X"])
    assert tp.tp_last_device_status() == 0
    try:
        tp.tp_set_wait_limit_ns(1)
        tp.tp_mlp_forward(s, X, variant="tmem_acc")
        assert tp.tp_last_device_status() == 7
    finally:
        tp.tp_set_wait_limit_ns(0)
    Z = tp.tp_mlp_forward(s, X, variant="tmem_acc")
    _sync()
    assert tp.tp_last_device_status() == 0
    assert rowwise_rms_error(Z.cpu().numpy(),
                             oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")) <= TOL_BF16_ROW_RMS


# ---- guard bands: no write outside the output buffers -----------------------------

@pytest.mark.parametrize("act,M,H,F,T,variant", [
    ("gelu", 300, 512, 2048, 4, "partials"),   # CTA-pair tiles with a ragged last tile
    ("gelu", 300, 512, 2048, 4, "tmem_acc"),
    ("swiglu", 100, 512, 2048, 8, "auto"),     # single-CTA tiles, ragged
    ("swiglu", 3, 512, 2048, 4, "auto"),       # decode kernels
    ("gelu", 37, 96, 240, 3, "partials"),      # float32 path
])
def test_outputs_stay_inside_their_buffers(tp, act, M, H, F, T, variant):
    """Y, Z and the workspace sit between canary bands; after the forward
    pass every canary word is intact and Z is still correct."""
    import torch
    dtype = "f32" if H == 96 else "bf16"
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype=dtype, seed=77, x_rows=max(M, 16))
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    X = to_device(d["X"])
    G = 4096  # canary words on each side
    canary = 0x7F7FDEAD
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def guarded(n_bytes):
        n_words = (n_bytes + 3) // 4
        buf = torch.full((G + n_words + G,), canary, dtype=torch.int32, device="cuda")
        return buf, buf[G:G + n_words]

    zbuf, zwords = guarded(M * H * 4)
    ybuf, ywords = guarded(T * M * (F // T) * (2 if dtype == "bf16" else 4))
    ws_col = tp.tp_colpar_workspace_bytes(s, M)
    ws_row = tp.tp_rowpar_workspace_bytes(s, M, variant)
    cbuf, cwords = guarded(max(ws_col, 16))
    rbuf, rwords = guarded(max(ws_row, 16))
    Z = zwords.view(torch.float32).view(M, H)
    Y = ywords.view(tdt).view(T, M, F // T)
    tp.tp_colpar_forward(s, X, Y, workspace=cwords.view(torch.uint8))
    tp.tp_rowpar_forward(s, Y, variant, Z, workspace=rwords.view(torch.uint8))
    _sync()
    assert tp.tp_last_device_status() == 0
    for buf in (zbuf, ybuf, cbuf, rbuf):
        assert torch.all(buf[:G] == canary) and torch.all(buf[-G:] == canary)
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act)
    if dtype == "bf16":
        assert rowwise_rms_error(Z.cpu().numpy(), Zref) <= TOL_BF16_ROW_RMS
    else:
        assert normwise_error(Z.cpu().numpy(), Zref) <= TOL_F32_NORMWISE


@pytest.mark.parametrize("M,variant", [(64, "tmem_acc"), (64, "partials"), (300, "tmem_acc")])
def test_float32_output_on_16_byte_boundary_matches_32(tp, M, variant):
    """The float32 epilogue stores 32 bytes at a time where the output rows are
    32-byte aligned and 16 at a time otherwise; Z at a 16-byte offset (legal:
    device pointers need 16-byte alignment) gives bit-identical results."""
    import torch
    H, F, T = 256, 1024, 2
    d = mlp_inputs(M=M, H=H, F=F, act="gelu", dtype="bf16", seed=5, x_rows=M)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "gelu")
    Y = tp.tp_colpar_forward(s, to_device(d["X"]))
    za = torch.full((M * H + 8,), float("nan"), dtype=torch.float32, device="cuda")
    zb = torch.full((M * H + 8,), float("nan"), dtype=torch.float32, device="cuda")
    Za = za[:M * H].view(M, H)           # the allocation's start: 32-byte aligned
    Zb = zb[4:4 + M * H].view(M, H)      # 16 bytes further
    assert Za.data_ptr() % 32 == 0 and Zb.data_ptr() % 32 == 16
    tp.tp_rowpar_forward(s, Y, variant, Za)
    tp.tp_rowpar_forward(s, Y, variant, Zb)
    _sync()
    assert tp.tp_last_device_status() == 0
    assert torch.equal(Za, Zb)
    assert torch.isnan(zb[:4]).all() and torch.isnan(zb[4 + M * H:]).all()
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")
    assert rowwise_rms_error(Za.cpu().numpy(), Zref) <= TOL_BF16_ROW_RMS


# ---- reduce-scatter, all-gather, bf16 all-reduce (bit exact) -----------------------

@pytest.mark.parametrize("T,n", [(2, 4096), (4, 1 << 20), (8, 8 * 1001), (3, 3 * 77), (8, 8 * 4096)])
def test_reduce_scatter_all_gather_bit_exact(tp, T, n):
    import torch
    P = partials_inputs(T, n, seed=40 + T)
    parts = [to_device(P[t]) for t in range(T)]
    rs = tp.tp_reduce_scatter(parts)
    _sync()
    ref = oracle.reduce_scatter_f32(P)
    for i in range(T):
        assert np.array_equal(rs[i].cpu().numpy(), ref[i])
    ag = tp.tp_all_gather(rs)
    _sync()
    assert np.array_equal(ag.cpu().numpy(), oracle.partial_sum_f32(P))
    # in-place all-gather: the parts already live in the output
    buf = torch.zeros(n, dtype=torch.float32, device="cuda")
    nb = n // T
    views = [buf[i * nb:(i + 1) * nb] for i in range(T)]
    for i in range(T):
        views[i].copy_(rs[i])
    tp.tp_all_gather(views, out=buf)
    _sync()
    assert np.array_equal(buf.cpu().numpy(), ag.cpu().numpy())
    # bf16 elements, odd sizes (byte path)
    parts16 = [torch.arange(i * 7, i * 7 + 7, device="cuda").to(torch.bfloat16) for i in range(T)]
    g16 = tp.tp_all_gather(parts16)
    _sync()
    assert torch.equal(g16.float().cpu(), torch.arange(7 * T).float())


@pytest.mark.parametrize("T,n", [(4, 1 << 20), (8, 12345), (1, 7)])
def test_partial_sum_bf16_bit_exact(tp, T, n):
    P = partials_inputs(T, n, seed=60 + T)
    Z = tp.tp_partial_sum_bf16([to_device(P[t]) for t in range(T)])
    _sync()
    assert np.array_equal(bf16_bits(Z), oracle.partial_sum_bf16(P))


# ---- failure injection: device allocation failures ---------------------------------

def test_injected_allocation_failures_report_oom_and_recover(tp):
    """With tp_inject_alloc_failures the library's next allocations fail as if
    the device were full: making shards, a self-allocated workspace and
    enabling the backward each return TP_ERR_OOM, nothing stays allocated,
    and the same calls work right after."""
    import torch
    M, H, F, T = 64, 512, 2048, 4
    d = mlp_inputs(M=M, H=H, F=F, act="gelu", dtype="bf16", seed=41, x_rows=M)
    W1, W2, X = to_device(d["W1"]), to_device(d["W2"]), to_device(d["X"])
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    try:
        tp.tp_inject_alloc_failures(1)
        with pytest.raises(tp.TPError) as e:
            tp.tp_shard_weights(W1, W2, T, "gelu")
        assert e.value.code == 5
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] >= free0 - (8 << 20)  # the failed calls freed what they took
        s = tp.tp_shard_weights(W1, W2, T, "gelu")
        tp.tp_inject_alloc_failures(1)
        with pytest.raises(tp.TPError) as e:
            tp.tp_mlp_forward(s, X)  # no workspace given: the library allocates one
        assert e.value.code == 5
        tp.tp_inject_alloc_failures(1)
        with pytest.raises(tp.TPError) as e:
            tp.tp_shards_enable_backward(s, W1, W2)
        assert e.value.code == 5
        Z = tp.tp_mlp_forward(s, X)
        _sync()
        assert tp.tp_last_device_status() == 0
        assert rowwise_rms_error(Z.cpu().numpy(),
                                 oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "gelu")) <= TOL_BF16_ROW_RMS
        tp.tp_shards_enable_backward(s, W1, W2)
        s.close()
    finally:
        tp.tp_inject_alloc_failures(0)
