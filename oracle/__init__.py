"""fp64 CPU oracle for the tensor-parallel MLP (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference legs use this package.  It shares no code with the CUDA path:
the arithmetic lives in ``tp_oracle.c`` (plain loops in fp64, OpenMP over
output rows), built here with gcc into ``liboracle.so`` and called through
ctypes.  Inputs are numpy arrays: float32, or bfloat16 given as its uint16
bit patterns.  Outputs are float64 numpy arrays.

Pages followed (see ``tp_oracle.c`` for the per-function citations):
"Slice the matrix itself" (column/row-parallel GEMMs and the row-parallel
summation), "Tensor Parallelism in Action: Megatron-LM Matrix Splitting"
(W1 column split, W2 row split, the GeLU concatenation identity) and the
"Tensor parallelism" guide (head sharding in attention).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
ACTS = {"gelu": 0, "swiglu": 1, "identity": 2}
OK, ERR_ARG, ERR_INDIVISIBLE, ERR_OOM = 0, 1, 2, 5

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``tp_oracle.c`` into ``liboracle.so`` (plain gcc, fp64, no
    fast-math, no contraction) and return the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        vp, i64, i32, dp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.orc_value.restype = ctypes.c_double
        lib.orc_value.argtypes = [vp, i64, i32]
        lib.orc_gelu.restype = ctypes.c_double
        lib.orc_gelu.argtypes = [ctypes.c_double]
        lib.orc_silu.restype = ctypes.c_double
        lib.orc_silu.argtypes = [ctypes.c_double]
        lib.orc_shard_w1.argtypes = [vp, i32, i64, i64, i32, i32, i32, i32, vp]
        lib.orc_shard_w2.argtypes = [vp, i32, i64, i64, i32, i32, vp]
        lib.orc_shard_wqkv.argtypes = [vp, i32, i64, i32, i32, i32, i32, vp]
        lib.orc_shard_wo.argtypes = [vp, i32, i64, i32, i32, i32, i32, vp]
        lib.orc_linear.argtypes = [vp, vp, i32, i64, i64, i64, vp, i64, dp]
        lib.orc_colpar_full.argtypes = [vp, vp, i32, i64, i64, i64, i32, vp, i64, dp]
        lib.orc_colpar_shard.argtypes = [vp, vp, i32, i64, i64, i64, i32, i32, i32, vp, i64, dp]
        lib.orc_mlp_unsharded.argtypes = [vp, vp, vp, i32, i64, i64, i64, i32, vp, i64, dp]
        lib.orc_mlp_unsharded_hbf16.argtypes = [vp, vp, vp, i32, i64, i64, i64, i32, vp, i64, dp]
        lib.orc_mlp_sharded.argtypes = [vp, vp, vp, i32, i64, i64, i64, i32, i32, vp, i64, dp]
        lib.orc_qkv_shard.argtypes = [vp, vp, i32, i64, i64, i32, i32, i32, i32, vp, i64, dp]
        lib.orc_oproj_sharded.argtypes = [vp, vp, i32, i64, i64, i32, i32, i32, vp, i64, dp]
        lib.orc_partial_sum_f32.restype = None
        lib.orc_partial_sum_f32.argtypes = [vp, i32, i64, vp]
        lib.orc_max_threads.restype = i32
        lib.orc_gelu_grad.restype = ctypes.c_double
        lib.orc_gelu_grad.argtypes = [ctypes.c_double]
        lib.orc_silu_grad.restype = ctypes.c_double
        lib.orc_silu_grad.argtypes = [ctypes.c_double]
        lib.orc_mlp_backward_dx.restype = i32
        lib.orc_mlp_backward_dx.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, vp, i64, dp]
        lib.orc_mlp_backward_dw.restype = i32
        lib.orc_mlp_backward_dw.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, vp, i64, dp, dp]
        lib.orc_block_forward.restype = i32
        lib.orc_block_forward.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, i32, i32, i64, i32, i32, i32,
                                          i32, vp, i64, dp, dp]
        lib.orc_attention.restype = i32
        lib.orc_attention.argtypes = [vp, vp, vp, i32, i64, i32, i32, i32, vp, i64, dp]
        lib.orc_reduce_scatter_f32.restype = i32
        lib.orc_reduce_scatter_f32.argtypes = [vp, i32, i64, vp]
        lib.orc_all_gather.restype = i32
        lib.orc_all_gather.argtypes = [vp, i32, i64, i32, vp]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.orc_partial_sum_bf16.restype = None
        lib.orc_partial_sum_bf16.argtypes = [vp, i32, i64, vp]
        for name in ("orc_shard_w1", "orc_shard_w2", "orc_shard_wqkv", "orc_shard_wo",
                     "orc_linear", "orc_colpar_full", "orc_colpar_shard",
                     "orc_mlp_unsharded", "orc_mlp_unsharded_hbf16", "orc_mlp_sharded", "orc_qkv_shard",
                     "orc_oproj_sharded"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with status {code}")
        self.code = code


def _check(code: int, what: str) -> None:
    if code != OK:
        raise OracleError(code, what)


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle inputs are float32, float64 or bfloat16 bits (uint16), got {a.dtype}")


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, M: int) -> np.ndarray:
    if rows is None:
        return np.arange(M, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def max_threads() -> int:
    return int(_load().orc_max_threads())


def value(a: np.ndarray, idx: int) -> float:
    """Exact value of element ``idx`` of a float32 / bfloat16-bits array."""
    a = _c(a)
    return float(_load().orc_value(_ptr(a), int(idx), _dt(a)))


def gelu(y: float) -> float:
    return float(_load().orc_gelu(float(y)))


def silu(g: float) -> float:
    return float(_load().orc_silu(float(g)))


def shard_w1(W1: np.ndarray, F: int, T: int, act: str, i: int, which: int = 0) -> np.ndarray:
    """Column block i of W1 (or of its gate / up half) as [H x F/T]."""
    W1 = _c(W1)
    H = W1.shape[0]
    if T <= 0 or F % T:
        raise OracleError(ERR_INDIVISIBLE if T > 0 else ERR_ARG, "shard_w1")
    out = np.empty((H, F // T), dtype=W1.dtype)
    _check(_load().orc_shard_w1(_ptr(W1), _dt(W1), H, F, T, ACTS[act], i, which, _ptr(out)),
           "shard_w1")
    return out


def shard_w2(W2: np.ndarray, T: int, i: int) -> np.ndarray:
    """Row block i of W2 as [F/T x H]."""
    W2 = _c(W2)
    F, H = W2.shape
    if T <= 0 or F % T:
        raise OracleError(ERR_INDIVISIBLE if T > 0 else ERR_ARG, "shard_w2")
    out = np.empty((F // T, H), dtype=W2.dtype)
    _check(_load().orc_shard_w2(_ptr(W2), _dt(W2), F, H, T, i, _ptr(out)), "shard_w2")
    return out


def shard_wqkv(Wqkv: np.ndarray, n_heads: int, head_dim: int, T: int, i: int) -> np.ndarray:
    Wqkv = _c(Wqkv)
    H = Wqkv.shape[0]
    if T <= 0 or n_heads % T:
        raise OracleError(ERR_INDIVISIBLE if T > 0 else ERR_ARG, "shard_wqkv")
    W = (n_heads // T) * head_dim
    out = np.empty((H, 3 * W), dtype=Wqkv.dtype)
    _check(_load().orc_shard_wqkv(_ptr(Wqkv), _dt(Wqkv), H, n_heads, head_dim, T, i, _ptr(out)),
           "shard_wqkv")
    return out


def shard_wo(Wo: np.ndarray, n_heads: int, head_dim: int, T: int, i: int) -> np.ndarray:
    Wo = _c(Wo)
    H = Wo.shape[0]
    if T <= 0 or n_heads % T:
        raise OracleError(ERR_INDIVISIBLE if T > 0 else ERR_ARG, "shard_wo")
    W = (n_heads // T) * head_dim
    out = np.empty((W, H), dtype=Wo.dtype)
    _check(_load().orc_shard_wo(_ptr(Wo), _dt(Wo), H, n_heads, head_dim, T, i, _ptr(out)),
           "shard_wo")
    return out


def linear(A: np.ndarray, W: np.ndarray, rows=None) -> np.ndarray:
    A, W = _c(A), _c(W)
    M, K = A.shape
    if W.shape[0] != K or W.dtype != A.dtype:
        raise ValueError("W does not match A")
    N = W.shape[1]
    r = _rows(rows, M)
    out = np.empty((r.size, N), dtype=np.float64)
    _check(_load().orc_linear(_ptr(A), _ptr(W), _dt(A), M, K, N, _ptr(r), r.size, _ptr(out)),
           "linear")
    return out


def colpar_full(X, W1, F: int, act: str, rows=None) -> np.ndarray:
    """act(X W1) on the selected rows, [rows x F] (SwiGLU: SiLU(X Wg) * X Wu)."""
    X, W1 = _c(X), _c(W1)
    M, H = X.shape
    if W1.shape != (H, 2 * F if act == "swiglu" else F) or W1.dtype != X.dtype:
        raise ValueError("W1 does not match X and F")
    r = _rows(rows, M)
    out = np.empty((r.size, F), dtype=np.float64)
    _check(_load().orc_colpar_full(_ptr(X), _ptr(W1), _dt(X), M, H, F, ACTS[act], _ptr(r),
                                   r.size, _ptr(out)), "colpar_full")
    return out


def colpar_shard(X, W1, F: int, T: int, act: str, i: int, rows=None) -> np.ndarray:
    """act(X W1_i) on the selected rows, [rows x F/T]."""
    X, W1 = _c(X), _c(W1)
    M, H = X.shape
    if W1.shape != (H, 2 * F if act == "swiglu" else F) or W1.dtype != X.dtype:
        raise ValueError("W1 does not match X and F")
    if T <= 0 or F % T:
        raise OracleError(ERR_INDIVISIBLE if T > 0 else ERR_ARG, "colpar_shard")
    r = _rows(rows, M)
    out = np.empty((r.size, F // T), dtype=np.float64)
    _check(_load().orc_colpar_shard(_ptr(X), _ptr(W1), _dt(X), M, H, F, T, ACTS[act], i,
                                    _ptr(r), r.size, _ptr(out)), "colpar_shard")
    return out


def _mlp_shapes(X, W1, W2, act):
    if X.ndim != 2 or W1.ndim != 2 or W2.ndim != 2:
        raise ValueError("X, W1, W2 must be 2-D")
    if not (X.dtype == W1.dtype == W2.dtype):
        raise ValueError("X, W1, W2 must share one element type")
    M, H = X.shape
    F = W2.shape[0]
    ncols = 2 * F if act == "swiglu" else F
    if W1.shape != (H, ncols) or W2.shape != (F, H):
        raise ValueError(f"shapes X {X.shape}, W1 {W1.shape}, W2 {W2.shape} do not form an MLP"
                         f" (need W1 [H x {'2F' if act == 'swiglu' else 'F'}], W2 [F x H])")
    return M, H, F


def mlp_unsharded(X, W1, W2, act: str, rows=None) -> np.ndarray:
    """Dense Z = act(X W1) W2 on the selected rows, [rows x H], fp64."""
    X, W1, W2 = _c(X), _c(W1), _c(W2)
    M, H, F = _mlp_shapes(X, W1, W2, act)
    r = _rows(rows, M)
    out = np.empty((r.size, H), dtype=np.float64)
    _check(_load().orc_mlp_unsharded(_ptr(X), _ptr(W1), _ptr(W2), _dt(X), M, H, F, ACTS[act],
                                     _ptr(r), r.size, _ptr(out)), "mlp_unsharded")
    return out


def mlp_unsharded_hbf16(X, W1, W2, act: str, rows=None) -> np.ndarray:
    """Z = bf16(act(X W1)) W2 on the selected rows: the first layer's output
    rounded to float32 and then bfloat16 (nearest even) before the second
    layer, as the workloads store it; otherwise fp64 like mlp_unsharded."""
    X, W1, W2 = _c(X), _c(W1), _c(W2)
    M, H, F = _mlp_shapes(X, W1, W2, act)
    r = _rows(rows, M)
    out = np.empty((r.size, H), dtype=np.float64)
    _check(_load().orc_mlp_unsharded_hbf16(_ptr(X), _ptr(W1), _ptr(W2), _dt(X), M, H, F, ACTS[act],
                                           _ptr(r), r.size, _ptr(out)), "mlp_unsharded_hbf16")
    return out


def mlp_sharded(X, W1, W2, T: int, act: str, rows=None) -> np.ndarray:
    """Sharded Z = sum_i act(X W1_i) W2_i on the selected rows, [rows x H]."""
    X, W1, W2 = _c(X), _c(W1), _c(W2)
    M, H, F = _mlp_shapes(X, W1, W2, act)
    r = _rows(rows, M)
    out = np.empty((r.size, H), dtype=np.float64)
    _check(_load().orc_mlp_sharded(_ptr(X), _ptr(W1), _ptr(W2), _dt(X), M, H, F, T, ACTS[act],
                                   _ptr(r), r.size, _ptr(out)), "mlp_sharded")
    return out


def qkv_shard(X, Wqkv, n_heads: int, head_dim: int, T: int, i: int, rows=None) -> np.ndarray:
    X, Wqkv = _c(X), _c(Wqkv)
    M, H = X.shape
    if Wqkv.shape != (H, 3 * H) or Wqkv.dtype != X.dtype:
        raise ValueError("Wqkv must be [H x 3H] like X")
    r = _rows(rows, M)
    W = (n_heads // T) * head_dim if T > 0 else 0
    out = np.empty((r.size, 3 * W), dtype=np.float64)
    _check(_load().orc_qkv_shard(_ptr(X), _ptr(Wqkv), _dt(X), M, H, n_heads, head_dim, T, i,
                                 _ptr(r), r.size, _ptr(out)), "qkv_shard")
    return out


def oproj_sharded(A, Wo, n_heads: int, head_dim: int, T: int, rows=None) -> np.ndarray:
    A, Wo = _c(A), _c(Wo)
    M, H = A.shape
    if Wo.shape != (H, H) or Wo.dtype != A.dtype:
        raise ValueError("Wo must be [H x H] like A")
    r = _rows(rows, M)
    out = np.empty((r.size, H), dtype=np.float64)
    _check(_load().orc_oproj_sharded(_ptr(A), _ptr(Wo), _dt(A), M, H, n_heads, head_dim, T,
                                     _ptr(r), r.size, _ptr(out)), "oproj_sharded")
    return out


def partial_sum_f32(P: np.ndarray) -> np.ndarray:
    """All-reduce-sum of float32 partials [T x n], ascending shard order."""
    P = np.ascontiguousarray(P, dtype=np.float32)
    T, n = P.shape
    out = np.empty(n, dtype=np.float32)
    _load().orc_partial_sum_f32(_ptr(P), T, n, _ptr(out))
    return out


def reduce_scatter_f32(P: np.ndarray) -> np.ndarray:
    """Reduce-scatter of float32 partials [T x n]: row i of the [T x n/T]
    result is block i of the ascending-order sum."""
    P = np.ascontiguousarray(P, dtype=np.float32)
    T, n = P.shape
    if n % T:
        raise OracleError(ERR_INDIVISIBLE, "reduce_scatter_f32")
    out = np.empty((T, n // T), dtype=np.float32)
    _check(_load().orc_reduce_scatter_f32(_ptr(P), T, n, _ptr(out)), "reduce_scatter_f32")
    return out


def all_gather(parts: np.ndarray) -> np.ndarray:
    """All-gather of T blocks [T x nb] into one array of T * nb elements."""
    parts = np.ascontiguousarray(parts)
    T, nb = parts.shape
    out = np.empty(T * nb, dtype=parts.dtype)
    _check(_load().orc_all_gather(_ptr(parts), T, nb, parts.dtype.itemsize, _ptr(out)), "all_gather")
    return out


def f32_to_bf16(x: float) -> int:
    return int(_load().orc_f32_to_bf16(float(x)))


def partial_sum_bf16(P: np.ndarray) -> np.ndarray:
    """All-reduce-sum of float32 partials [T x n] rounded once to bfloat16 (bits)."""
    P = np.ascontiguousarray(P, dtype=np.float32)
    T, n = P.shape
    out = np.empty(n, dtype=np.uint16)
    _load().orc_partial_sum_bf16(_ptr(P), T, n, _ptr(out))
    return out


def gelu_grad(y: float) -> float:
    return float(_load().orc_gelu_grad(float(y)))


def silu_grad(g: float) -> float:
    return float(_load().orc_silu_grad(float(g)))


def mlp_backward_dx(X, W1, W2, dZ, act: str, rows=None) -> np.ndarray:
    """dX = dP W1^T on the selected token rows, [rows x H] (fp64)."""
    X, W1, W2, dZ = _c(X), _c(W1), _c(W2), _c(dZ)
    M, H, F = _mlp_shapes(X, W1, W2, act)
    if dZ.shape != (M, H) or dZ.dtype != X.dtype:
        raise ValueError("dZ must be [M x H] like X")
    r = _rows(rows, M)
    out = np.empty((r.size, H), dtype=np.float64)
    _check(_load().orc_mlp_backward_dx(_ptr(X), _ptr(W1), _ptr(W2), _ptr(dZ), _dt(X), M, H, F,
                                       ACTS[act], _ptr(r), r.size, _ptr(out)), "mlp_backward_dx")
    return out


def mlp_backward_dw(X, W1, W2, dZ, act: str, fcols=None):
    """(dW1 columns, dW2 rows) at the selected FFN indices f: dW1 [H x n]
    (SwiGLU [H x 2n]: gate columns then up columns), dW2 [n x H] (fp64)."""
    X, W1, W2, dZ = _c(X), _c(W1), _c(W2), _c(dZ)
    M, H, F = _mlp_shapes(X, W1, W2, act)
    if dZ.shape != (M, H) or dZ.dtype != X.dtype:
        raise ValueError("dZ must be [M x H] like X")
    f = _rows(fcols, F)
    n = f.size
    nparts = 2 if act == "swiglu" else 1
    dW1 = np.empty((H, nparts * n), dtype=np.float64)
    dW2 = np.empty((n, H), dtype=np.float64)
    _check(_load().orc_mlp_backward_dw(_ptr(X), _ptr(W1), _ptr(W2), _ptr(dZ), _dt(X), M, H, F,
                                       ACTS[act], _ptr(f), n, _ptr(dW1), _ptr(dW2)), "mlp_backward_dw")
    return dW1, dW2


def block_forward(X, Wqkv, Wo, W1, W2, n_heads: int, head_dim: int, T: int, act: str,
                  causal: bool = True, sharded: bool = True, rows=None):
    """One tensor-parallel transformer block on the selected token rows:
    returns (out, h), each [rows x H] fp64, h the residual stream after the
    attention all-reduce."""
    X, Wqkv, Wo, W1, W2 = _c(X), _c(Wqkv), _c(Wo), _c(W1), _c(W2)
    M, H = X.shape
    F = W2.shape[0]
    if Wqkv.shape != (H, 3 * H) or Wo.shape != (H, H) or W2.shape != (F, H) or \
            W1.shape != (H, 2 * F if act == "swiglu" else F):
        raise ValueError("block weight shapes do not match X")
    r = _rows(rows, M)
    out = np.empty((r.size, H), dtype=np.float64)
    h = np.empty((r.size, H), dtype=np.float64)
    _check(_load().orc_block_forward(_ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(W1), _ptr(W2), _dt(X), M, H,
                                     n_heads, head_dim, F, ACTS[act], int(causal), T, int(sharded),
                                     _ptr(r), r.size, _ptr(out), _ptr(h)), "block_forward")
    return out, h


def attention(Q, K, V, causal: bool = True, rows=None) -> np.ndarray:
    """Scaled dot-product attention per head on head-major Q, K, V
    [n_heads x M x head_dim] (bfloat16 bits, float32 or float64): returns the
    selected token rows [rows x n_heads*head_dim] fp64, heads side by side."""
    Q, K, V = _c(Q), _c(K), _c(V)
    if Q.ndim != 3 or K.shape != Q.shape or V.shape != Q.shape or not (Q.dtype == K.dtype == V.dtype):
        raise ValueError("Q, K and V must share one shape [n_heads, M, head_dim] and one dtype")
    nh, M, hd = Q.shape
    r = _rows(rows, M)
    out = np.empty((r.size, nh * hd), dtype=np.float64)
    _check(_load().orc_attention(_ptr(Q), _ptr(K), _ptr(V), _dt(Q), M, nh, hd, int(causal), _ptr(r), r.size,
                                 _ptr(out)), "attention")
    return out
