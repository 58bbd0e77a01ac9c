"""Host-side checks that need no GPU: the C-ABI library builds, loads and
exports every symbol include/tp_mlp.h declares; argument errors come back as
status codes; the ring byte model matches the pages' worked example."""
import ctypes
import re
from pathlib import Path

import pytest

import linear_sharding_gb300 as tp
from linear_sharding_gb300 import build as tp_build

ROOT = Path(__file__).resolve().parents[1]
GOLDEN = Path(__file__).parent / "golden"


@pytest.fixture(scope="module")
def lib():
    tp_build.build()
    return tp.load_library()


def _declared_symbols():
    text = (ROOT / "include" / "tp_mlp.h").read_text()
    return sorted(set(re.findall(r"^TP_API[^(]*?\b(tp_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert _declared_symbols() == sorted(tp.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    assert lib.tp_abi_version() == 1


def test_status_strings(lib):
    for code, name in tp.STATUS.items():
        assert lib.tp_status_str(code).decode().startswith(name)
    assert lib.tp_status_str(99) == b"unknown tp_status_t"


def test_argument_errors_are_status_codes(lib):
    """Checks that run before any device call: null pointers, T out of range,
    F not divisible by T, a bad enum."""
    out = ctypes.c_void_p()
    dummy = ctypes.c_void_p(256)
    assert lib.tp_shard_weights(None, dummy, 64, 256, 2, 0, 1, None, ctypes.byref(out)) == 1
    assert lib.tp_shard_weights(dummy, dummy, 64, 256, 0, 0, 1, None, ctypes.byref(out)) == 1
    assert lib.tp_shard_weights(dummy, dummy, 64, 256, 65, 0, 1, None, ctypes.byref(out)) == 1
    assert lib.tp_shard_weights(dummy, dummy, 64, 250, 4, 0, 1, None, ctypes.byref(out)) == 2
    assert lib.tp_shard_weights(dummy, dummy, 64, 256, 2, 7, 1, None, ctypes.byref(out)) == 1
    assert lib.tp_shard_weights(dummy, dummy, 64, 256, 2, 0, 5, None, ctypes.byref(out)) == 3
    assert lib.tp_shard_weights(dummy, dummy, 100, 256, 2, 0, 1, None, ctypes.byref(out)) == 9
    assert lib.tp_shard_weights(dummy, dummy, 64, 256, 2, 0, 1, None, None) == 1
    assert lib.tp_shard_weights_qkv(dummy, dummy, 4096, 32, 128, 3, None, ctypes.byref(out)) == 2
    assert lib.tp_shard_weights_qkv(dummy, dummy, 4096, 32, 100, 4, None, ctypes.byref(out)) == 1
    assert out.value is None
    assert lib.tp_mlp_forward(None, dummy, 4, 0, 0, dummy, None, 0, None) == 1
    assert lib.tp_mlp_workspace_bytes(None, 4, 0) == 0
    assert lib.tp_shard_get(None, 0, 0, dummy) == 1
    arr = (ctypes.c_void_p * 2)(256, 512)
    assert lib.tp_partial_sum(arr, 0, 16, dummy, None) == 1
    assert lib.tp_partial_sum(arr, 65, 16, dummy, None) == 1
    assert lib.tp_partial_sum(None, 2, 16, dummy, None) == 1
    assert lib.tp_partial_sum(arr, 2, 16, None, None) == 1
    nulls = (ctypes.c_void_p * 2)(None, None)
    assert lib.tp_partial_sum(nulls, 2, 16, dummy, None) == 1
    assert lib.tp_partial_sum(nulls, 2, 0, None, None) == 0  # n == 0: no-op, pointers unused
    assert lib.tp_partial_sum(arr, 2, -1, dummy, None) == 1
    overlap = (ctypes.c_void_p * 2)(256, 4096)
    assert lib.tp_partial_sum(overlap, 2, 16, ctypes.c_void_p(4096 + 32), None) == 1
    assert lib.tp_attention_forward(dummy, dummy, dummy, 16, 2, 64, 1, dummy, 256, None, 0, None) == 9
    assert lib.tp_attention_forward(dummy, dummy, dummy, -1, 2, 128, 1, dummy, 256, None, 0, None) == 1
    assert lib.tp_attention_workspace_bytes(100, 2, 64) == 0
    assert lib.tp_inject_alloc_failures(-1) == 1
    assert lib.tp_inject_alloc_failures(3) == 0 and lib.tp_inject_alloc_failures(0) == 0
    lib.tp_set_machine_balance.argtypes = [ctypes.c_double]
    assert lib.tp_set_machine_balance(-1.0) == 1
    assert lib.tp_set_machine_balance(float("nan")) == 1
    assert lib.tp_set_machine_balance(2e6) == 1
    assert lib.tp_set_machine_balance(280.0) == 0 and lib.tp_set_machine_balance(0.0) == 0
    lib.tp_set_rowpar_schedule.argtypes = [ctypes.c_int]
    assert lib.tp_set_rowpar_schedule(2) == 1 and lib.tp_set_rowpar_schedule(-1) == 1
    assert lib.tp_set_rowpar_schedule(0) == 0 and lib.tp_set_rowpar_schedule(1) == 0
    lib.tp_rowpar_tiles.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    out3 = (ctypes.c_int32 * 3)(7, 7, 7)
    assert lib.tp_rowpar_tiles(None, 16, 0, out3) == 1 and list(out3) == [0, 0, 0]
    assert lib.tp_rowpar_tiles(None, 16, 0, None) == 1
    lib.tp_shards_destroy(None)


def _kv(name):
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = int(v)
    return out


def test_ring_volume_worked_example():
    """The pages' example: H = 8192 BF16, T = 8 -> 16 KiB payload, 28 KiB ring
    volume per rank, 80 layers x 2 collectives -> 4480 KiB per token."""
    g = _kv("ring_allreduce_worked_example.txt")
    assert g["H"] * g["B"] == g["payload_bytes"]
    assert tp.ring_allreduce_bytes(g["H"], g["T"], g["B"]) == g["ring_bytes_per_rank"]
    from linear_sharding_gb300.volume import decode_bytes_per_token
    assert decode_bytes_per_token(g["H"], g["T"], g["B"], g["layers"],
                                  g["collectives_per_layer"]) == g["per_token_decode_bytes"]
    assert tp.ring_allreduce_bytes(8192, 1, 2) == 0.0
