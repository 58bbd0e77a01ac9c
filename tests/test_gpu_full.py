"""Parity at the full workload sizes, in the launch configuration the
benchmark times, on sampled output rows (a row of Z depends only on that
row of X, so the oracle computes the sampled rows alone).  Tolerance: bf16
row-RMS measure (tests/gpu_util.py), every variant (float32 partials with
the shard-sum, one TMEM accumulator over all shards, and the planner's
choice).  The global-RMS reading of the tolerance is asserted too: against
2e-2 where there are no outlier rows, and against its own bound on the
large SwiGLU workload (tests/gpu_util.py, TOL_BF16_GLOBAL_RMS_OUTLIERS)."""
import numpy as np
import pytest

import oracle
from synth import WORKLOADS, attn_inputs, mlp_inputs
from tests.gpu_util import (TOL_BF16_GLOBAL_RMS_OUTLIERS, TOL_BF16_ROW_RMS, BF16H_ERROR_RATIO, bf16_bits,
                            global_rms_error, rowwise_rms_error, stratified_rms, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import linear_sharding_gb300 as tp
    tp.load_library()
    return tp


def _sample_rows(M, k, seed, must=()):
    rng = np.random.default_rng(seed)
    rows = set(int(r) for r in must) | {0, M - 1}
    rest = [int(r) for r in rng.choice(M, size=min(M, k), replace=False)]
    for r in rest:
        if len(rows) >= k:
            break
        rows.add(r)
    return np.array(sorted(rows), dtype=np.int64)


def _mlp_check(tp, name, variants, k_rows=24, global_tol=TOL_BF16_ROW_RMS):
    import torch
    w = WORKLOADS[name]
    d = mlp_inputs(M=w["M"], H=w["H"], F=w["F"], act=w["act"], dtype=w["dtype"], seed=0,
                   outlier_frac=w.get("outlier_frac", 0.0), outlier_scale=w.get("outlier_scale", 20.0))
    W1, W2 = to_device(d["W1"]), to_device(d["W2"])
    s = tp.tp_shard_weights(W1, W2, w["T"], w["act"])
    del W1, W2
    X = to_device(d["X"])
    out = d["outlier_rows"]
    rows = _sample_rows(w["M"], k_rows, seed=1, must=out[: min(8, out.size)])
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], w["act"], rows=rows)
    Zref_h = oracle.mlp_unsharded_hbf16(d["X"], d["W1"], d["W2"], w["act"], rows=rows)
    # RMS of the whole output, estimated per stratum (outlier rows, other rows)
    # from the oracle's sampled rows
    rms_all = stratified_rms(Zref, np.isin(rows, out), out.size, w["M"])
    for v in variants:
        Z = tp.tp_mlp_forward(s, X, variant=v)
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0
        Zs = Z[torch.from_numpy(rows).cuda()].cpu().numpy()
        err = rowwise_rms_error(Zs, Zref)
        gerr = global_rms_error(Zs, Zref, rms=rms_all)
        herr = rowwise_rms_error(Zs, Zref_h)
        print(f"{name} {v}: row-RMS err {err:.3e}, global-RMS err {gerr:.3e}, against bf16 h {herr:.3e}")
        assert err <= TOL_BF16_ROW_RMS
        assert gerr <= global_tol
        assert herr <= BF16H_ERROR_RATIO * err
        del Z
    return d, s


def test_prefill_gelu_full(tp):
    _mlp_check(tp, "prefill_gelu_m2048_h4096_f16384_t4", ["auto", "partials", "tmem_acc"])


def test_large_prefill_swiglu_full(tp):
    name = "prefill_swiglu_m8192_h8192_f28672_t8_outliers"
    d, s = _mlp_check(tp, name, ["auto", "partials", "tmem_acc"], k_rows=24,
                      global_tol=TOL_BF16_GLOBAL_RMS_OUTLIERS)
    w = WORKLOADS[name]
    assert d["outlier_rows"].size == 82
    # shard layout bit exact at full size, first and last shard
    for i in (0, w["T"] - 1):
        assert np.array_equal(tp.tp_shard_get(s, i, 0), oracle.shard_w1(d["W1"], w["F"], w["T"], "swiglu", i, 0))
        assert np.array_equal(tp.tp_shard_get(s, i, 1), oracle.shard_w1(d["W1"], w["F"], w["T"], "swiglu", i, 1))
        assert np.array_equal(tp.tp_shard_get(s, i, 2), oracle.shard_w2(d["W2"], w["T"], i))


def test_decode_swiglu_full(tp):
    """Every row at M in {1, 4, 16}, one set of weights."""
    import torch
    w = WORKLOADS["decode_swiglu_h8192_f28672_t8"]
    d = mlp_inputs(M=16, H=w["H"], F=w["F"], act="swiglu", dtype="bf16", seed=0, x_rows=16)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), w["T"], "swiglu")
    Zref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], "swiglu")
    Zref_h = oracle.mlp_unsharded_hbf16(d["X"], d["W1"], d["W2"], "swiglu")
    for M in w["decode_m"]:
        X = to_device(d["X"][:M])
        for v in ("auto", "partials", "tmem_acc"):
            Z = tp.tp_mlp_forward(s, X, variant=v)
            torch.cuda.synchronize()
            assert tp.tp_last_device_status() == 0
            err = rowwise_rms_error(Z.cpu().numpy(), Zref[:M])
            gerr = global_rms_error(Z.cpu().numpy(), Zref[:M])
            herr = rowwise_rms_error(Z.cpu().numpy(), Zref_h[:M])
            print(f"decode M={M} {v}: row-RMS err {err:.3e}, global-RMS err {gerr:.3e}, against bf16 h {herr:.3e}")
            assert err <= TOL_BF16_ROW_RMS and gerr <= TOL_BF16_ROW_RMS and herr <= BF16H_ERROR_RATIO * err


def test_attn_proj_full(tp):
    import torch
    w = WORKLOADS["attn_proj_m4096_h4096_32x128_t8"]
    d = attn_inputs(M=w["M"], H=w["H"], n_heads=w["n_heads"], head_dim=w["head_dim"], seed=0)
    s = tp.tp_shard_weights_qkv(to_device(d["Wqkv"]), to_device(d["Wo"]), w["n_heads"], w["head_dim"], w["T"])
    X, A = to_device(d["X"]), to_device(d["A"])
    rows = _sample_rows(w["M"], 24, seed=2)
    Zref = oracle.oproj_sharded(d["A"], d["Wo"], w["n_heads"], w["head_dim"], w["T"], rows=rows)
    ridx = torch.from_numpy(rows).cuda()
    for v in ("auto", "partials", "tmem_acc"):
        QKV, Z = tp.tp_attn_proj_forward(s, X=X, A=A, variant=v)
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0
        err = rowwise_rms_error(Z[ridx].cpu().numpy(), Zref)
        gerr = global_rms_error(Z[ridx].cpu().numpy(), Zref)
        print(f"attn o-proj {v}: row-RMS err {err:.3e}, global-RMS err {gerr:.3e}")
        assert err <= TOL_BF16_ROW_RMS and gerr <= TOL_BF16_ROW_RMS
    q = bf16_bits(QKV[:, ridx])
    for i in range(w["T"]):
        ref = oracle.qkv_shard(d["X"], d["Wqkv"], w["n_heads"], w["head_dim"], w["T"], i, rows=rows)
        got = (q[i].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert rowwise_rms_error(got, ref) <= TOL_BF16_ROW_RMS


def test_more_than_2_31_elements_in_y(tp):
    """Maximum sizes: M = 65636 (a ragged last tile), H = 1024, F = 36864,
    T = 4 makes the first layer's output Y 2.42e9 bf16 elements (4.8 GB),
    past 2^31: element offsets must not wrap.  Rows on both sides of 2^31 / F
    and of the halfway point, and the last rows, every variant."""
    import torch
    M, H, F, T = 65636, 1024, 36864, 4
    assert M * F > 2 ** 31
    g = torch.Generator(device="cuda")
    g.manual_seed(21)
    X = torch.randn((M, H), generator=g, device="cuda").to(torch.bfloat16)
    W1 = (torch.randn((H, F), generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16)
    W2 = (torch.randn((F, H), generator=g, device="cuda") * F ** -0.5).to(torch.bfloat16)
    s = tp.tp_shard_weights(W1, W2, T, "gelu")
    r31 = 2 ** 31 // F  # the first row with Y elements past 2^31 (T F_s = F columns a row)
    rows = np.array([0, 1, M // 2 - 1, M // 2, r31 - 1, r31, r31 + 1, M - 2, M - 1], dtype=np.int64)
    bits = lambda a: a.cpu().view(torch.int16).numpy().view(np.uint16)
    Xs = bits(X[torch.from_numpy(rows).cuda()])
    Zref = oracle.mlp_unsharded(Xs, bits(W1), bits(W2), "gelu")
    Zref_h = oracle.mlp_unsharded_hbf16(Xs, bits(W1), bits(W2), "gelu")
    del W1, W2
    for v in ("auto", "partials", "tmem_acc"):
        Z = tp.tp_mlp_forward(s, X, variant=v)
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0
        Zs = Z[torch.from_numpy(rows).cuda()].cpu().numpy()
        del Z
        err, herr = rowwise_rms_error(Zs, Zref), rowwise_rms_error(Zs, Zref_h)
        print(f"Y of {M * F} elements, {v}: row-RMS err {err:.3e}, against bf16 h {herr:.3e}")
        assert err <= TOL_BF16_ROW_RMS and herr <= BF16H_ERROR_RATIO * err
    s.close()
