"""Tensor-parallel transformer MLP on one GB300: Python binding of libtpmlp.so.

Argument marshalling only.  Every step of the path runs in the library's CUDA
kernels; PyTorch provides device memory and the current stream.  There is no
CPU fallback: if the library is missing, loading it raises.

The functions keep the C names (see include/tp_mlp.h for the contract):
``tp_shard_weights``, ``tp_shard_weights_qkv``, ``tp_shard_get``,
``tp_mlp_forward``, ``tp_mlp_forward_host``, ``tp_attn_proj_forward``,
``tp_partial_sum``, ``tp_last_device_status``, ``tp_set_wait_limit_ns``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .volume import ring_allreduce_bytes  # noqa: F401  (host arithmetic, no GPU)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtpmlp.so")

ACT = {"gelu": 0, "swiglu": 1, "identity": 2}
DTYPE = {"f32": 0, "bf16": 1}
VARIANT = {"auto": 0, "partials": 1, "tmem_acc": 2}
STATUS = {
    0: "TP_OK", 1: "TP_ERR_ARG", 2: "TP_ERR_INDIVISIBLE", 3: "TP_ERR_DTYPE", 4: "TP_ERR_ARCH",
    5: "TP_ERR_OOM", 6: "TP_ERR_CUDA", 7: "TP_ERR_TIMEOUT", 8: "TP_ERR_DEVICE_CHECK",
    9: "TP_ERR_UNSUPPORTED", 10: "TP_ERR_WORKSPACE",
}
EXPORTS = (
    "tp_status_str", "tp_abi_version", "tp_shard_weights", "tp_shard_weights_qkv", "tp_shard_get",
    "tp_shard_info", "tp_shards_destroy", "tp_mlp_workspace_bytes", "tp_mlp_forward",
    "tp_mlp_host_workspace_bytes", "tp_mlp_forward_host", "tp_attn_proj_workspace_bytes",
    "tp_attn_proj_forward", "tp_partial_sum", "tp_last_device_status", "tp_set_wait_limit_ns",
    "tp_colpar_workspace_bytes", "tp_colpar_forward", "tp_rowpar_workspace_bytes",
    "tp_rowpar_forward", "tp_mlp_forward_noalloc", "tp_reduce_scatter", "tp_all_gather",
    "tp_partial_sum_bf16", "tp_shards_enable_backward", "tp_mlp_train_workspace_bytes",
    "tp_mlp_forward_train", "tp_mlp_backward_workspace_bytes", "tp_mlp_backward",
    "tp_block_workspace_bytes", "tp_block_forward", "tp_attention_workspace_bytes",
    "tp_attention_forward", "tp_inject_alloc_failures", "tp_set_machine_balance", "tp_set_rowpar_schedule",
    "tp_rowpar_tiles",
)

_lock = threading.Lock()
_lib = None


class TPError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtpmlp.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i64, i32, sz, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t,
                                 ctypes.c_uint64)
        lib.tp_status_str.restype = ctypes.c_char_p
        lib.tp_status_str.argtypes = [i32]
        lib.tp_abi_version.restype = i32
        lib.tp_shard_weights.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp, ctypes.POINTER(vp)]
        lib.tp_shard_weights_qkv.argtypes = [vp, vp, i64, i32, i32, i32, vp, ctypes.POINTER(vp)]
        lib.tp_shard_get.argtypes = [vp, i32, i32, vp]
        lib.tp_shard_info.argtypes = [vp] + [vp] * 6
        lib.tp_shards_destroy.restype = None
        lib.tp_shards_destroy.argtypes = [vp]
        lib.tp_mlp_workspace_bytes.restype = sz
        lib.tp_mlp_workspace_bytes.argtypes = [vp, i64, i32]
        lib.tp_mlp_forward.argtypes = [vp, vp, i64, i32, i32, vp, vp, sz, vp]
        lib.tp_mlp_host_workspace_bytes.restype = sz
        lib.tp_mlp_host_workspace_bytes.argtypes = [vp, i64, i32]
        lib.tp_mlp_forward_host.argtypes = [vp, vp, i64, i32, i32, vp, vp, sz, vp]
        lib.tp_attn_proj_workspace_bytes.restype = sz
        lib.tp_attn_proj_workspace_bytes.argtypes = [vp, i64, i32]
        lib.tp_attn_proj_forward.argtypes = [vp, vp, vp, i64, i32, vp, vp, vp, sz, vp]
        lib.tp_partial_sum.argtypes = [ctypes.POINTER(vp), i32, i64, vp, vp]
        lib.tp_last_device_status.argtypes = [vp]
        lib.tp_set_wait_limit_ns.argtypes = [u64]
        lib.tp_inject_alloc_failures.argtypes = [i32]
        lib.tp_set_machine_balance.argtypes = [ctypes.c_double]
        lib.tp_set_rowpar_schedule.argtypes = [i32]
        lib.tp_rowpar_tiles.argtypes = [vp, i64, i32, vp]
        lib.tp_colpar_workspace_bytes.restype = sz
        lib.tp_colpar_workspace_bytes.argtypes = [vp, i64]
        lib.tp_colpar_forward.argtypes = [vp, vp, i64, i32, vp, vp, sz, vp]
        lib.tp_rowpar_workspace_bytes.restype = sz
        lib.tp_rowpar_workspace_bytes.argtypes = [vp, i64, i32]
        lib.tp_rowpar_forward.argtypes = [vp, vp, i64, i32, vp, vp, sz, vp]
        lib.tp_mlp_forward_noalloc.argtypes = [vp, vp, i64, i32, vp, vp]
        lib.tp_reduce_scatter.argtypes = [ctypes.POINTER(vp), i32, i64, ctypes.POINTER(vp), vp]
        lib.tp_all_gather.argtypes = [ctypes.POINTER(vp), i32, i64, i32, vp, vp]
        lib.tp_partial_sum_bf16.argtypes = [ctypes.POINTER(vp), i32, i64, vp, vp]
        lib.tp_shards_enable_backward.argtypes = [vp, vp, vp, vp]
        lib.tp_mlp_train_workspace_bytes.restype = sz
        lib.tp_mlp_train_workspace_bytes.argtypes = [vp, i64, i32]
        lib.tp_mlp_forward_train.argtypes = [vp, vp, i64, i32, i32, vp, vp, vp, vp, sz, vp]
        lib.tp_mlp_backward_workspace_bytes.restype = sz
        lib.tp_mlp_backward_workspace_bytes.argtypes = [vp, i64, i32]
        lib.tp_mlp_backward.argtypes = [vp, vp, vp, vp, vp, i64, i32, vp, vp, vp, vp, sz, vp]
        lib.tp_block_workspace_bytes.restype = sz
        lib.tp_block_workspace_bytes.argtypes = [vp, vp, i64, i32]
        lib.tp_block_forward.argtypes = [vp, vp, vp, i64, i32, i32, vp, vp, vp, sz, vp]
        lib.tp_attention_workspace_bytes.restype = sz
        lib.tp_attention_workspace_bytes.argtypes = [i64, i32, i32]
        lib.tp_attention_forward.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp, i64, vp, sz, vp]
        for name in ("tp_shard_weights", "tp_shard_weights_qkv", "tp_shard_get", "tp_shard_info",
                     "tp_mlp_forward", "tp_mlp_forward_host", "tp_attn_proj_forward",
                     "tp_partial_sum", "tp_last_device_status", "tp_set_wait_limit_ns",
                     "tp_colpar_forward", "tp_rowpar_forward", "tp_mlp_forward_noalloc",
                     "tp_reduce_scatter", "tp_all_gather", "tp_partial_sum_bf16",
                     "tp_shards_enable_backward", "tp_mlp_forward_train", "tp_mlp_backward",
                     "tp_block_forward", "tp_attention_forward", "tp_inject_alloc_failures",
                     "tp_set_machine_balance"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def _check(code: int, what: str) -> None:
    if code != 0:
        raise TPError(code, what)


def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dtype_name(t) -> str:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return "bf16"
    if t.dtype == torch.float32:
        return "f32"
    raise TypeError(f"element type {t.dtype} is not supported (bfloat16 or float32)")


class Shards:
    """Library-owned sharded weights (a tp_shards_t handle)."""

    def __init__(self, handle: int, kind: str, H: int, F: int, T: int, act: str, dtype: str,
                 n_heads: int = 0, head_dim: int = 0):
        self.handle = ctypes.c_void_p(handle)
        self.kind, self.H, self.F, self.T, self.act, self.dtype = kind, H, F, T, act, dtype
        self.n_heads, self.head_dim = n_heads, head_dim

    @property
    def Fs(self) -> int:
        return self.F // self.T

    def close(self) -> None:
        if self.handle and self.handle.value:
            load_library().tp_shards_destroy(self.handle)
            self.handle = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tp_shard_weights(W1, W2, T: int, act: str = "gelu", stream=None) -> Shards:
    """Shard W1 [H x F] (or [H x 2F] = [Wg | Wu] for SwiGLU) by columns and
    W2 [F x H] by rows into T shards on W1's device."""
    lib = load_library()
    dt = _dtype_name(W1)
    if W2.dtype != W1.dtype:
        raise TypeError("W1 and W2 must share one element type")
    W1, W2 = W1.contiguous(), W2.contiguous()
    F, H = W2.shape
    out = ctypes.c_void_p()
    _check(lib.tp_shard_weights(_ptr(W1), _ptr(W2), H, F, T, ACT[act], DTYPE[dt], _stream(stream),
                                ctypes.byref(out)), "tp_shard_weights")
    return Shards(out.value, "mlp", H, F, T, act, dt)


def tp_shard_weights_qkv(Wqkv, Wo, n_heads: int, head_dim: int, T: int, stream=None) -> Shards:
    """Shard [Wq | Wk | Wv] ([H x 3H]) and Wo ([H x H]) by heads into T shards."""
    lib = load_library()
    if _dtype_name(Wqkv) != "bf16" or Wo.dtype != Wqkv.dtype:
        raise TypeError("attention projections take bfloat16 weights")
    Wqkv, Wo = Wqkv.contiguous(), Wo.contiguous()
    H = Wo.shape[0]
    out = ctypes.c_void_p()
    _check(lib.tp_shard_weights_qkv(_ptr(Wqkv), _ptr(Wo), H, n_heads, head_dim, T, _stream(stream),
                                    ctypes.byref(out)), "tp_shard_weights_qkv")
    return Shards(out.value, "qkv", H, H, T, "identity", "bf16", n_heads, head_dim)


def tp_shard_get(s: Shards, i: int, which: int):
    """The logical shard i as a host numpy array (bfloat16 as uint16 bits):
    which 0 = W1_i / Wg_i / Wqkv_i, 1 = Wu_i, 2 = W2_i / Wo_i."""
    import numpy as np
    lib = load_library()
    W = s.Fs
    if which == 2:
        shape = (W, s.H)
    elif s.kind == "qkv":
        shape = (s.H, 3 * W)
    else:
        shape = (s.H, W)
    out = np.empty(shape, dtype=np.uint16 if s.dtype == "bf16" else np.float32)
    _check(lib.tp_shard_get(s.handle, i, which, out.ctypes.data_as(ctypes.c_void_p)), "tp_shard_get")
    return out


def tp_mlp_workspace_bytes(s: Shards, M: int, variant: str = "auto") -> int:
    return int(load_library().tp_mlp_workspace_bytes(s.handle, M, VARIANT[variant]))


def tp_mlp_forward(s: Shards, X, variant: str = "auto", Z=None, workspace=None, act=None,
                   stream=None):
    """Z = sum_i act(X W1_i) W2_i ([M x H] float32) on X's device."""
    torch = _torch()
    lib = load_library()
    if X.dim() != 2 or X.shape[1] != s.H or _dtype_name(X) != s.dtype:
        raise ValueError("X must be [M x H] with the shards' element type")
    X = X.contiguous()
    M = X.shape[0]
    if Z is None:
        Z = torch.empty((M, s.H), dtype=torch.float32, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.tp_mlp_forward(s.handle, _ptr(X), M, ACT[act or s.act], VARIANT[variant], _ptr(Z),
                              _ptr(workspace), ws_bytes, _stream(stream)), "tp_mlp_forward")
    return Z


def tp_colpar_workspace_bytes(s: Shards, M: int) -> int:
    return int(load_library().tp_colpar_workspace_bytes(s.handle, M))


def tp_colpar_forward(s: Shards, X, Y=None, workspace=None, act=None, stream=None):
    """Y_i = act(X W1_i) for every shard: Y is [T x M x F/T] (shard blocks contiguous)."""
    torch = _torch()
    lib = load_library()
    X = X.contiguous()
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((s.T, M, s.Fs), dtype=X.dtype, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.tp_colpar_forward(s.handle, _ptr(X), M, ACT[act or s.act], _ptr(Y), _ptr(workspace),
                                 ws_bytes, _stream(stream)), "tp_colpar_forward")
    return Y


def tp_rowpar_workspace_bytes(s: Shards, M: int, variant: str = "auto") -> int:
    return int(load_library().tp_rowpar_workspace_bytes(s.handle, M, VARIANT[variant]))


def tp_rowpar_forward(s: Shards, Y, variant: str = "auto", Z=None, workspace=None, stream=None):
    """Z = sum_i Y_i W2_i ([M x H] float32), the row-parallel layer and its all-reduce-sum."""
    torch = _torch()
    lib = load_library()
    M = Y.shape[1]
    if Z is None:
        Z = torch.empty((M, s.H), dtype=torch.float32, device=Y.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.tp_rowpar_forward(s.handle, _ptr(Y), M, VARIANT[variant], _ptr(Z), _ptr(workspace),
                                 ws_bytes, _stream(stream)), "tp_rowpar_forward")
    return Z


def tp_mlp_host_workspace_bytes(s: Shards, M: int, variant: str = "auto") -> int:
    return int(load_library().tp_mlp_host_workspace_bytes(s.handle, M, VARIANT[variant]))


def tp_mlp_forward_host(s: Shards, X_host, Z_host, workspace, variant: str = "auto", stream=None):
    """The forward pass from host buffers (pinned CPU tensors): copies X in,
    computes, copies Z back, all enqueued on the stream."""
    lib = load_library()
    M = X_host.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.tp_mlp_forward_host(s.handle, _ptr(X_host), M, ACT[s.act], VARIANT[variant],
                                   _ptr(Z_host), _ptr(workspace), ws_bytes, _stream(stream)),
           "tp_mlp_forward_host")
    return Z_host


def tp_attn_proj_workspace_bytes(s: Shards, M: int, variant: str = "auto") -> int:
    return int(load_library().tp_attn_proj_workspace_bytes(s.handle, M, VARIANT[variant]))


def tp_attn_proj_forward(s: Shards, X=None, A=None, variant: str = "auto", QKV=None, Z=None,
                         workspace=None, stream=None):
    """QKV_i = X Wqkv_i ([T x M x 3W] bf16) and Z = sum_i A_i Wo_i ([M x H] float32)."""
    torch = _torch()
    lib = load_library()
    ref = X if X is not None else A
    M = ref.shape[0]
    W = s.Fs
    if X is not None and QKV is None:
        QKV = torch.empty((s.T, M, 3 * W), dtype=torch.bfloat16, device=ref.device)
    if A is not None and Z is None:
        Z = torch.empty((M, s.H), dtype=torch.float32, device=ref.device)
    X = X.contiguous() if X is not None else None
    A = A.contiguous() if A is not None else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.tp_attn_proj_forward(s.handle, _ptr(X), _ptr(A), M, VARIANT[variant],
                                    _ptr(QKV if X is not None else None),
                                    _ptr(Z if A is not None else None), _ptr(workspace), ws_bytes,
                                    _stream(stream)), "tp_attn_proj_forward")
    return QKV, Z


def tp_partial_sum(parts, Z=None, stream=None):
    """Z = ((parts[0] + parts[1]) + ...) + parts[T-1], float32, on the GPU."""
    torch = _torch()
    lib = load_library()
    T = len(parts)
    n = parts[0].numel()
    if Z is None:
        Z = torch.empty_like(parts[0])
    arr = (ctypes.c_void_p * T)(*[p.data_ptr() for p in parts])
    _check(lib.tp_partial_sum(arr, T, n, _ptr(Z), _stream(stream)), "tp_partial_sum")
    return Z


def _ptr_array(tensors):
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def tp_reduce_scatter(parts, out=None, stream=None):
    """Rank i keeps block i of the sum: out[i] = sum_t parts[t][i*nb:(i+1)*nb]."""
    torch = _torch()
    T, n = len(parts), parts[0].numel()
    if out is None:
        out = [torch.empty(n // T, dtype=torch.float32, device=parts[0].device) for _ in range(T)]
    _check(load_library().tp_reduce_scatter(_ptr_array(parts), T, n, _ptr_array(out), _stream(stream)),
           "tp_reduce_scatter")
    return out


def tp_all_gather(parts, out=None, stream=None):
    """out = concatenation of the T parts (same element type and size)."""
    torch = _torch()
    T, n = len(parts), parts[0].numel()
    if out is None:
        out = torch.empty(T * n, dtype=parts[0].dtype, device=parts[0].device)
    _check(load_library().tp_all_gather(_ptr_array(parts), T, n, parts[0].element_size(), _ptr(out),
                                        _stream(stream)), "tp_all_gather")
    return out


def tp_partial_sum_bf16(parts, Z=None, stream=None):
    """The all-reduce-sum rounded once to bfloat16."""
    torch = _torch()
    n = parts[0].numel()
    if Z is None:
        Z = torch.empty(n, dtype=torch.bfloat16, device=parts[0].device)
    _check(load_library().tp_partial_sum_bf16(_ptr_array(parts), len(parts), n, _ptr(Z), _stream(stream)),
           "tp_partial_sum_bf16")
    return Z


def tp_shards_enable_backward(s: Shards, W1, W2, stream=None) -> None:
    """Give the handle W1/W2 in the caller's layout for the backward GEMMs."""
    _check(load_library().tp_shards_enable_backward(s.handle, _ptr(W1.contiguous()), _ptr(W2.contiguous()),
                                                    _stream(stream)), "tp_shards_enable_backward")


def tp_mlp_forward_train(s: Shards, X, variant: str = "auto", stream=None):
    """Forward pass keeping (Hsave, Psave) for the backward; returns (Z, Hsave, Psave)."""
    torch = _torch()
    lib = load_library()
    X = X.contiguous()
    M = X.shape[0]
    Z = torch.empty((M, s.H), dtype=torch.float32, device=X.device)
    Hs = torch.empty((s.T, M, s.Fs), dtype=torch.bfloat16, device=X.device)
    nP = 2 if s.act == "swiglu" else 1
    Ps = torch.empty((nP, s.T, M, s.Fs), dtype=torch.bfloat16, device=X.device)
    ws = torch.empty(max(lib.tp_mlp_train_workspace_bytes(s.handle, M, VARIANT[variant]), 1),
                     dtype=torch.uint8, device=X.device)
    _check(lib.tp_mlp_forward_train(s.handle, _ptr(X), M, ACT[s.act], VARIANT[variant], _ptr(Z), _ptr(Hs),
                                    _ptr(Ps), _ptr(ws), ws.numel(), _stream(stream)), "tp_mlp_forward_train")
    return Z, Hs, Ps


def tp_mlp_backward(s: Shards, X, Hsave, Psave, dZ, variant: str = "auto", stream=None):
    """Gradients (dX [M x H], dW1 [H x F or 2F], dW2 [F x H]), float32."""
    torch = _torch()
    lib = load_library()
    M = X.shape[0]
    ncols = 2 * s.F if s.act == "swiglu" else s.F
    dX = torch.empty((M, s.H), dtype=torch.float32, device=X.device)
    dW1 = torch.empty((s.H, ncols), dtype=torch.float32, device=X.device)
    dW2 = torch.empty((s.F, s.H), dtype=torch.float32, device=X.device)
    ws = torch.empty(max(lib.tp_mlp_backward_workspace_bytes(s.handle, M, VARIANT[variant]), 1),
                     dtype=torch.uint8, device=X.device)
    _check(lib.tp_mlp_backward(s.handle, _ptr(X.contiguous()), _ptr(Hsave), _ptr(Psave), _ptr(dZ.contiguous()),
                               M, VARIANT[variant], _ptr(dX), _ptr(dW1), _ptr(dW2), _ptr(ws), ws.numel(),
                               _stream(stream)), "tp_mlp_backward")
    return dX, dW1, dW2


def tp_block_workspace_bytes(attn: Shards, mlp: Shards, M: int, variant: str = "auto") -> int:
    return int(load_library().tp_block_workspace_bytes(attn.handle, mlp.handle, M, VARIANT[variant]))


def tp_block_forward(attn: Shards, mlp: Shards, X, causal: bool = True, variant: str = "auto",
                     out=None, h_out=None, workspace=None, stream=None):
    """One TP transformer block: returns (out, h) float32 [M x H] (h is None
    unless h_out=True or a tensor is given)."""
    torch = _torch()
    lib = load_library()
    X = X.contiguous()
    M = X.shape[0]
    if out is None:
        out = torch.empty((M, attn.H), dtype=torch.float32, device=X.device)
    if h_out is True:
        h_out = torch.empty((M, attn.H), dtype=torch.float32, device=X.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.tp_block_forward(attn.handle, mlp.handle, _ptr(X), M, int(bool(causal)), VARIANT[variant],
                                _ptr(out), _ptr(h_out if h_out is not False else None), _ptr(workspace),
                                ws_bytes, _stream(stream)), "tp_block_forward")
    return out, (h_out if h_out is not False else None)


def tp_attention_workspace_bytes(M: int, n_heads: int, head_dim: int = 128) -> int:
    return int(load_library().tp_attention_workspace_bytes(M, n_heads, head_dim))


def tp_attention_forward(Q, K, V, causal: bool = True, out=None, workspace=None, stream=None):
    """Attention per head: Q, K, V bf16 [n_heads, M, head_dim] (device) ->
    O bf16 [M, n_heads * head_dim], heads side by side."""
    torch = _torch()
    lib = load_library()
    Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
    nh, M, hd = Q.shape
    if K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("Q, K and V must have the same shape [n_heads, M, head_dim]")
    if not (Q.dtype == K.dtype == V.dtype == torch.bfloat16):
        raise TypeError("tp_attention_forward takes bfloat16 Q, K and V")
    if out is None:
        out = torch.empty((M, nh * hd), dtype=torch.bfloat16, device=Q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.tp_attention_forward(_ptr(Q), _ptr(K), _ptr(V), M, nh, hd, int(bool(causal)), _ptr(out),
                                    out.stride(0), _ptr(workspace), ws_bytes, _stream(stream)),
           "tp_attention_forward")
    return out


def tp_last_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load_library().tp_last_device_status(_stream(stream)))


def tp_set_wait_limit_ns(ns: int) -> None:
    _check(load_library().tp_set_wait_limit_ns(int(ns)), "tp_set_wait_limit_ns")


def tp_set_machine_balance(flop_per_byte: float) -> None:
    """Flop per HBM byte the AUTO planners weigh partial traffic with (0: the
    device's own figures)."""
    _check(load_library().tp_set_machine_balance(float(flop_per_byte)), "tp_set_machine_balance")


def tp_set_rowpar_schedule(wide: bool) -> None:
    """Let the row-parallel GEMM with one accumulator use wide output tiles
    where they fit one round of CTA pairs (True, the default), or always
    256-column tiles (False).  The results are identical."""
    _check(load_library().tp_set_rowpar_schedule(1 if wide else 0), "tp_set_rowpar_schedule")


def tp_rowpar_tiles(s: Shards, M: int, variant: str = "auto"):
    """The row-parallel GEMM's wide tiles for M tokens: (widest tile's columns, tiles of that
    width per 256-row block, tiles per block), or None where it takes another form."""
    out = (ctypes.c_int32 * 3)()
    _check(load_library().tp_rowpar_tiles(s.handle, int(M), VARIANT[variant], ctypes.cast(out, ctypes.c_void_p)),
           "tp_rowpar_tiles")
    return tuple(out) if out[0] else None


def tp_inject_alloc_failures(count: int) -> None:
    """Make the library's next `count` device allocations fail (tests); 0 cancels."""
    _check(load_library().tp_inject_alloc_failures(int(count)), "tp_inject_alloc_failures")
