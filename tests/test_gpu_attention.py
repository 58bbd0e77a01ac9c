"""Parity of the fused attention core (tp_attention_forward) with the fp64
oracle on the same bfloat16 Q, K, V: every row at small sizes that span
several query and key tiles with a ragged tail, sampled rows at the
4096-token 32-head workload, peaky and drifting score distributions (the
online softmax's shift), and the edge cases.  Tolerance: the probabilities
and O are each rounded to bfloat16 once; elementwise within 2^-8 |ref| +
TOL_ATTN_ELEMENT row-RMS, and row-RMS within TOL_BF16_GRAD_ROW_RMS."""
import numpy as np
import pytest

import oracle
from synth import attention_inputs
from tests.gpu_util import (TOL_ATTN_ELEMENT, TOL_BF16_GRAD_ROW_RMS, attention_elementwise_ok, bf16_bits,
                            rowwise_rms_error, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import linear_sharding_gb300 as tp
    tp.load_library()
    return tp


def _sync():
    import torch
    torch.cuda.synchronize()


def _as_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ok(got, ref, what):
    e, el = rowwise_rms_error(got, ref), attention_elementwise_ok(got, ref)
    print(f"attention {what}: row-RMS {e:.3e}, elementwise slack {el:.3e}")
    return e <= TOL_BF16_GRAD_ROW_RMS and el <= TOL_ATTN_ELEMENT


def _run(tp, d, causal, rows=None, **kw):
    Q, K, V = (to_device(d[k]) for k in ("Q", "K", "V"))
    O = tp.tp_attention_forward(Q, K, V, causal=causal, **kw)
    _sync()
    assert tp.tp_last_device_status() == 0
    nh, M, hd = d["Q"].shape
    r = np.arange(M) if rows is None else np.asarray(rows)
    got = _as_f64(bf16_bits(O)[r])
    ref = oracle.attention(d["Q"], d["K"], d["V"], causal=causal, rows=r)
    return got, ref, O


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("M,nh", [(1, 1), (100, 2), (128, 1), (129, 3), (300, 4), (1000, 2)])
def test_attention_small_all_rows(tp, M, nh, causal):
    d = attention_inputs(M, nh, seed=M + nh)
    got, ref, _ = _run(tp, d, causal)
    assert _ok(got, ref, f"M={M} nh={nh} causal={causal}")


@pytest.mark.parametrize("q_scale,key_ramp", [(4.0, 0.0), (1.0, 3.0), (3.0, 2.0)])
def test_attention_peaky_and_drifting_scores(tp, q_scale, key_ramp):
    """Scores with a spread of 4 (near one-hot rows), and keys that score
    higher the later they come, so the running maximum moves at every key
    tile and the rescaling of the partial output is exercised."""
    M, nh = 700, 2
    d = attention_inputs(M, nh, seed=5, q_scale=q_scale, key_ramp=key_ramp)
    for causal in (True, False):
        got, ref, _ = _run(tp, d, causal)
        assert _ok(got, ref, f"q_scale={q_scale} key_ramp={key_ramp} causal={causal}")


def test_attention_more_units_than_sms(tp):
    """16 heads x 12 pairs of 128-row query tiles = 192 units on at most 152
    CTAs: CTAs take several units each, in snake order, with the pipeline
    carried across unit boundaries; 3000 tokens leave a ragged last tile
    (rows 2944..2999)."""
    M, nh = 3000, 16
    d = attention_inputs(M, nh, seed=21)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, 1023, 2815, 2816, 2943, 2944, 2998, 2999],
                                     rng.choice(M, 120, replace=False)]))
    for causal in (True, False):
        got, ref, _ = _run(tp, d, causal, rows=rows)
        assert _ok(got, ref, f"M=3000 nh=16 causal={causal}")


def test_attention_full_workload_sampled_rows(tp):
    """The block's attention at its full size (4096 tokens, 32 heads of 128),
    in the launch configuration the benchmark times; rows sampled across all
    query tiles, including the heaviest (last) tiles."""
    M, nh = 4096, 32
    d = attention_inputs(M, nh, seed=9)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 2047, 4094, 4095], rng.choice(M, 57, replace=False)]))
    got, ref, _ = _run(tp, d, True, rows=rows)
    assert _ok(got, ref, f"M=4096 nh=32 causal, {rows.size} rows")


def test_attention_deterministic_and_strided_output(tp):
    """Two calls give identical bits; with ldo > width the columns past the
    heads are left untouched."""
    import torch
    M, nh = 300, 2
    d = attention_inputs(M, nh, seed=2)
    Q, K, V = (to_device(d[k]) for k in ("Q", "K", "V"))
    a = tp.tp_attention_forward(Q, K, V)
    b = tp.tp_attention_forward(Q, K, V)
    wide = torch.full((M, nh * 128 + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    tp.tp_attention_forward(Q, K, V, out=wide[:, : nh * 128])
    # rows of 264 bf16 (528 bytes): every other row starts on a 16-byte, not a
    # 32-byte, boundary, so both output store widths run
    odd = torch.full((M, nh * 128 + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    tp.tp_attention_forward(Q, K, V, out=odd[:, : nh * 128])
    _sync()
    assert torch.equal(a, b)
    assert torch.equal(wide[:, : nh * 128], a)
    assert torch.all(wide[:, nh * 128:] == 7.0)
    assert torch.equal(odd[:, : nh * 128], a)
    assert torch.all(odd[:, nh * 128:] == 7.0)


def test_attention_edge_cases_and_errors(tp):
    import torch
    z = torch.zeros((2, 0, 128), dtype=torch.bfloat16, device="cuda")
    assert tp.tp_attention_forward(z, z, z).shape == (0, 256)  # M == 0: no-op
    q64 = torch.zeros((2, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_attention_forward(q64, q64, q64)
    assert e.value.code == 9  # TP_ERR_UNSUPPORTED: head_dim must be 128
    q = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_attention_forward(q, q, q, out=q.view(16, 256))  # output overlaps the inputs
    assert e.value.code == 1
    assert tp.tp_attention_workspace_bytes(100, 2, 64) == 0


def test_attention_wait_timeout_reports_and_recovers(tp):
    """A 1 ns wait limit makes the attention kernel's waits run out: it returns
    early with TP_ERR_TIMEOUT in the status word, nothing faults, and the next
    call with the default limit is correct."""
    M, nh = 300, 2
    d = attention_inputs(M, nh, seed=6)
    Q, K, V = (to_device(d[k]) for k in ("Q", "K", "V"))
    assert tp.tp_last_device_status() == 0
    try:
        tp.tp_set_wait_limit_ns(1)
        tp.tp_attention_forward(Q, K, V)
        assert tp.tp_last_device_status() == 7
    finally:
        tp.tp_set_wait_limit_ns(0)
    got, ref, _ = _run(tp, d, True)
    assert _ok(got, ref, "after a timeout")
