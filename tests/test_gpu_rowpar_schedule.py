"""The row-parallel GEMM's two tile schedules (tp_set_rowpar_schedule): with
one TMEM accumulator over all shards, 256-column tiles in rounds of the
GPU's CTA pairs, or, where they fit one round, wider tiles (two MMAs per
k-step into two accumulators) of near-equal widths.  Both add every output
element's products over the same K order in one accumulator, so Z must be
the same bit for bit; and Z must match the fp64 oracle on sampled rows
within the bf16 tolerance.  The shapes are ones where the wide schedule
applies on a 152-SM GB300 (76 CTA pairs): the planner is restated below to
say which tiles it picks, and on another GPU the comparison still holds."""
import numpy as np
import pytest

import oracle
from synth import mlp_inputs
from tests.gpu_util import TOL_BF16_ROW_RMS, rowwise_rms_error, to_device

pytestmark = pytest.mark.gpu


def _wide_plan(m_tiles, H, clusters, kt, epi_ktiles=6):
    """Restated schedule choice: each 256-row block cut into q tiles of
    widths (multiples of 32, differing by at most 32), each over 256 and at
    most 480 columns, in one or two rounds of the clusters, q as large as that
    allows; priced as rounds x width x kt / 0.9 plus epi_ktiles x 480 per extra
    round (6 for the float32 output, 24 with a residual in the epilogue),
    against the 256-column tiles' rounds x 256 x kt / 0.8, and taken when at
    least 5 % cheaper.  Returns (widest, tiles of that width, tiles per
    block) or None."""
    units = H // 32
    rounds_u = -(-m_tiles * (H // 256) // clusters)
    best, best_cost = None, 0.95 * rounds_u * 256 * kt / 0.8
    for rounds in (1, 2):
        for q in range(rounds * clusters // m_tiles, 0, -1):
            w1 = -(-units // q)
            nb = units - q * (w1 - 1)
            narrowest = w1 if nb == q else w1 - 1
            if 32 * narrowest <= 256:
                continue
            if 32 * w1 > 480:
                break
            rounds_w = -(-m_tiles * q // clusters)
            cost = rounds_w * 32 * w1 * kt / 0.9 + (rounds_w - 1) * epi_ktiles * 480
            if cost < best_cost:
                best, best_cost = (32 * w1, nb, q), cost
            break
    return best


@pytest.fixture(scope="module")
def tp():
    import linear_sharding_gb300 as tp
    tp.load_library()
    yield tp
    tp.tp_set_rowpar_schedule(True)


@pytest.mark.parametrize("act,M,H,F,T", [
    ("gelu", 2048, 4096, 4096, 4),      # 8 row blocks: 2 tiles of 480 and 7 of 448 each
    ("swiglu", 1100, 4096, 2048, 2),    # 5 row blocks, ragged: tiles of 320 and 288
    ("identity", 700, 8192, 1024, 1),   # 3 row blocks: tiles of 352 and 320, T = 1
    ("gelu", 1900, 4096, 3072, 3),      # ragged last row block, T = 3
])
def test_wide_tiles_equal_256_column_tiles(tp, act, M, H, F, T):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    print(f"M={M} H={H}: wide plan on {sms // 2} pairs: {_wide_plan(-(-M // 256), H, sms // 2, F // T // 64 * T)}")
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=M + T)
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    X = to_device(d["X"])
    out = {}
    for wide in (True, False, True):
        tp.tp_set_rowpar_schedule(wide)
        Z = tp.tp_mlp_forward(s, X, variant="tmem_acc")
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0
        z = Z.cpu().numpy()
        if wide in out:
            assert np.array_equal(z, out[wide]), "the wide schedule is not deterministic"
        out[wide] = z
    tp.tp_set_rowpar_schedule(True)
    assert np.array_equal(out[True], out[False]), "wide and 256-column tiles differ"
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([[0, 255, 256, M - 1], rng.choice(M, 12, replace=False)]))
    ref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act, rows=rows)
    err = rowwise_rms_error(out[True][rows], ref)
    print(f"{act} M={M} H={H} T={T}: row-RMS err {err:.3e}")
    assert err <= TOL_BF16_ROW_RMS
    s.close()


def test_wide_plan_restatement_matches_documented_cases():
    """The restated planner picks the tiles the documentation states (host only)."""
    assert _wide_plan(8, 4096, 76, 256) == (480, 2, 9)    # prefill: one round
    assert _wide_plan(5, 4096, 76, 256) == (320, 2, 14)
    assert _wide_plan(3, 8192, 76, 16) == (352, 6, 25)
    assert _wide_plan(16, 4096, 76, 256) == (480, 2, 9)   # the block's MLP: two rounds
    assert _wide_plan(16, 4096, 76, 64) == (480, 2, 9)    # the block's O-projection
    assert _wide_plan(4, 4096, 76, 256) is None           # 64 tiles of 256 already fit one round
    assert _wide_plan(32, 8192, 76, 448) is None          # many rounds: no width fits two
    # with a residual in the epilogue (the block at M = 4096): the down-projection's 256 k-tiles
    # keep the wide tiles, the output projection's 64 do not
    assert _wide_plan(16, 4096, 76, 256, epi_ktiles=24) == (480, 2, 9)
    assert _wide_plan(16, 4096, 76, 64, epi_ktiles=24) is None
    assert _wide_plan(8, 4096, 76, 64, epi_ktiles=24) == (480, 2, 9)   # one round: no exposed epilogue priced


def test_backward_dx_wide_tiles_equal_256_column_tiles(tp):
    """The backward's dX = sum over shards of dP_i W1_i^T has the row-parallel
    shape and takes the same schedules: dX (and dW1, dW2, which do not depend
    on it) bit-identical between them."""
    import torch
    from synth import f32_to_bf16_bits
    M, H, F, T, act = 2048, 4096, 4096, 4, "gelu"
    d = mlp_inputs(M=M, H=H, F=F, act=act, dtype="bf16", seed=9)
    dZ = to_device(f32_to_bf16_bits(np.random.default_rng(9).standard_normal((M, H)).astype(np.float32)))
    s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
    tp.tp_shards_enable_backward(s, to_device(d["W1"]), to_device(d["W2"]))
    X = to_device(d["X"])
    out = {}
    for wide in (True, False):
        tp.tp_set_rowpar_schedule(wide)
        Z, Hs, Ps = tp.tp_mlp_forward_train(s, X, "auto")
        grads = tp.tp_mlp_backward(s, X, Hs, Ps, dZ, "auto")
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0
        out[wide] = [Z.cpu().numpy()] + [t.cpu().numpy() for t in grads]
    tp.tp_set_rowpar_schedule(True)
    for a, b in zip(out[True], out[False]):
        assert np.array_equal(a, b)
    s.close()


def test_block_wide_tiles_equal_256_column_tiles(tp):
    """One transformer block at the attention-projection workload's shapes
    (M = 4096, 32 heads of 128, T = 8, SwiGLU F = 4H): its MLP row-parallel
    GEMM, with the residual in its epilogue, runs on two rounds of wide tiles
    (the O-projection, with a K of 64 k-tiles, on 256-column tiles either
    way); the block's output and residual stream h must equal the 256-column
    tiles' bit for bit."""
    import torch
    from tests.test_gpu_block import _weights
    M, nh, hd, T = 4096, 32, 128, 8
    H, F = nh * hd, 4 * nh * hd
    d = _weights(M, H, F, "swiglu", seed=11)
    a = tp.tp_shard_weights_qkv(to_device(d["Wqkv"]), to_device(d["Wo"]), nh, hd, T)
    m = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, "swiglu")
    X = to_device(d["X"])
    out = {}
    for wide in (True, False):
        tp.tp_set_rowpar_schedule(wide)
        o, h = tp.tp_block_forward(a, m, X, causal=True, h_out=True)
        torch.cuda.synchronize()
        assert tp.tp_last_device_status() == 0
        out[wide] = (o.cpu().numpy(), h.cpu().numpy())
    tp.tp_set_rowpar_schedule(True)
    assert np.array_equal(out[True][1], out[False][1]), "h differs"
    assert np.array_equal(out[True][0], out[False][0]), "block output differs"
    a.close()
    m.close()


def test_random_shapes_both_schedules_agree(tp):
    """Random shapes around the sizes where the wide tiles apply (256-row blocks from 3 to 16,
    H from 2048 to 8192, ragged M, every activation, T from 1 to 8): Z from the wide tiles
    equals Z from 256-column tiles bit for bit, and two sampled rows match the oracle."""
    import torch
    rng = np.random.default_rng(2028)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wide_cases = 0
    for case in range(24):
        m_tiles = int(rng.integers(3, 17))
        M = int(rng.integers(256 * (m_tiles - 1) + 1, 256 * m_tiles + 1))
        H = 256 * int(rng.integers(8, 33))
        T = int(rng.choice([1, 2, 4, 8]))
        Fs = 128 * int(rng.integers(1, 4))
        act = str(rng.choice(["gelu", "swiglu", "identity"]))
        plan = _wide_plan(m_tiles, H, sms // 2, Fs * T // 64)
        wide_cases += plan is not None
        d = mlp_inputs(M=M, H=H, F=Fs * T, act=act, dtype="bf16", seed=500 + case)
        s = tp.tp_shard_weights(to_device(d["W1"]), to_device(d["W2"]), T, act)
        X = to_device(d["X"])
        out = {}
        for wide in (True, False):
            tp.tp_set_rowpar_schedule(wide)
            Z = tp.tp_mlp_forward(s, X, variant="tmem_acc")
            torch.cuda.synchronize()
            assert tp.tp_last_device_status() == 0
            out[wide] = Z.cpu().numpy()
        tp.tp_set_rowpar_schedule(True)
        assert np.array_equal(out[True], out[False]), (case, M, H, T, Fs, act, plan)
        rows = np.array([0, M - 1])
        ref = oracle.mlp_unsharded(d["X"], d["W1"], d["W2"], act, rows=rows)
        assert rowwise_rms_error(out[True][rows], ref) <= TOL_BF16_ROW_RMS, (case, M, H, T, act)
        s.close()
    print(f"{wide_cases} of 24 random shapes on wide tiles")
    assert wide_cases >= 6


def test_library_plan_matches_restatement(tp):
    """The library's own tile plan (tp_rowpar_tiles) against the restated planner, on 40 random
    shapes with one TMEM accumulator (M from 257 to 4096, H a multiple of 256 up to 8192), and
    none under tp_set_rowpar_schedule(False) or on the decode path."""
    import torch
    rng = np.random.default_rng(2029)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    hits = 0
    for case in range(40):
        M = int(rng.integers(257, 4097))
        H = 256 * int(rng.integers(4, 33))
        T = int(rng.choice([1, 2, 4, 8]))
        Fs = 128 * int(rng.integers(1, 4))
        W1 = torch.zeros((H, Fs * T), dtype=torch.bfloat16, device="cuda")
        W2 = torch.zeros((Fs * T, H), dtype=torch.bfloat16, device="cuda")
        s = tp.tp_shard_weights(W1, W2, T, "gelu")
        want = _wide_plan(-(-M // 256), H, sms // 2, Fs * T // 64)
        got = tp.tp_rowpar_tiles(s, M, "tmem_acc")
        assert got == want, (case, M, H, T, Fs, got, want)
        hits += got is not None
        tp.tp_set_rowpar_schedule(False)
        assert tp.tp_rowpar_tiles(s, M, "tmem_acc") is None
        tp.tp_set_rowpar_schedule(True)
        assert tp.tp_rowpar_tiles(s, 16, "tmem_acc") is None   # decode path
        s.close()
    print(f"{hits} of 40 shapes planned on wide tiles")
    assert hits >= 5
