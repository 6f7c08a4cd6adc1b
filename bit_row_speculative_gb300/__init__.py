"""Python binding of libq4 (include/q4.h): argument marshalling only.

Every step of the verify matmul runs in the library's CUDA kernels; PyTorch
only supplies device memory and streams.  The binding fails loudly when the
compiled library is missing -- there is no fallback path.

Build the library with ``python -c "import __graft_entry__ as g; g.build()"``
(or ``python bit_row_speculative_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libq4.so")

Q4_OK = 0
Q4_ERR_INVALID_ARG = 1
Q4_ERR_UNSUPPORTED_SHAPE = 2
Q4_ERR_MISALIGNED = 3
Q4_ERR_UNSUPPORTED_DEVICE = 4
Q4_ERR_CUDA = 5
Q4_ERR_TIMEOUT = 6
Q4_ERR_OVERFLOW = 7
Q4_ERR_INVALID_INDEX = 8
MAX_ROWS = 32
GROUP = 64

# Exported symbols (one per function declared in include/q4.h).
SYMBOLS = ("q4_packed_bytes", "q4_matmul", "q4_matmul_noalloc", "q4_glue", "q4_decode_step_workspace_bytes",
           "q4_decode_step", "q4_topk_probs", "q4_lm_head_topk", "q4_draft_select_edges", "q4_check_wait_timeout", "q4_device_status", "q4_last_error", "q4_status_string")

GLUE_NONE = 0
GLUE_RMSNORM = 1
GLUE_SWIGLU_RMSNORM = 2


class Layer(ctypes.Structure):
    """q4_layer: packed W [N, K] (device pointer) and the glue to the next layer."""
    _fields_ = [("W", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("glue", ctypes.c_int)]


class Q4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def _declare(lib: ctypes.CDLL) -> None:
    c = ctypes
    lib.q4_packed_bytes.restype = c.c_uint64
    lib.q4_packed_bytes.argtypes = [c.c_uint64, c.c_uint64]
    lib.q4_matmul.restype = c.c_int
    lib.q4_matmul.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_int64, c.c_int64, c.c_void_p, c.c_void_p]
    lib.q4_matmul_noalloc.restype = c.c_int
    lib.q4_matmul_noalloc.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_int64, c.c_int64, c.c_void_p, c.c_void_p]
    lib.q4_glue.restype = c.c_int
    lib.q4_glue.argtypes = [c.c_void_p, c.c_int, c.c_int64, c.c_int64, c.c_int, c.c_void_p, c.c_void_p]
    lib.q4_decode_step_workspace_bytes.restype = c.c_size_t
    lib.q4_decode_step_workspace_bytes.argtypes = [c.c_void_p, c.c_int, c.c_int]
    lib.q4_decode_step.restype = c.c_int
    lib.q4_decode_step.argtypes = [c.c_void_p, c.c_int, c.c_void_p, c.c_int, c.c_void_p, c.c_size_t, c.c_void_p,
                                   c.c_void_p]
    lib.q4_topk_probs.restype = c.c_int
    lib.q4_topk_probs.argtypes = [c.c_void_p, c.c_int, c.c_int64, c.c_int, c.c_float, c.c_float, c.c_void_p,
                                  c.c_void_p, c.c_void_p]
    lib.q4_lm_head_topk.restype = c.c_int
    lib.q4_lm_head_topk.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_int64, c.c_int64, c.c_int, c.c_float,
                                    c.c_float, c.c_void_p, c.c_void_p, c.c_void_p]
    lib.q4_draft_select_edges.restype = c.c_int
    lib.q4_draft_select_edges.argtypes = [c.c_void_p, c.c_void_p, c.c_int64, c.c_int, c.c_void_p, c.c_void_p,
                                          c.c_void_p, c.c_int, c.c_void_p, c.c_void_p]
    lib.q4_check_wait_timeout.restype = c.c_int
    lib.q4_check_wait_timeout.argtypes = [c.c_longlong, c.c_void_p]
    lib.q4_device_status.restype = c.c_int
    lib.q4_device_status.argtypes = [c.c_void_p]
    lib.q4_last_error.restype = c.c_char_p
    lib.q4_last_error.argtypes = []
    lib.q4_status_string.restype = c.c_char_p
    lib.q4_status_string.argtypes = [c.c_int]


def lib() -> ctypes.CDLL:
    """The loaded libq4.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libq4.so is not built ({LIB_PATH} missing); run __graft_entry__.build()")
            handle = ctypes.CDLL(LIB_PATH)
            _declare(handle)
            _lib = handle
        return _lib


def status_name(status: int) -> str:
    try:
        return lib().q4_status_string(status).decode()
    except Exception:
        return f"status {status}"


def _check(status: int) -> None:
    if status != Q4_OK:
        raise Q4Error(status, lib().q4_last_error().decode())


def packed_bytes(N: int, K: int) -> int:
    return int(lib().q4_packed_bytes(N, K))


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _tensor(t, name: str, dtype, shape=None, dim=None):
    """A tensor argument checked before its pointer reaches the library (which
    cannot see sizes): dtype, rank, shape and contiguity.  The device is checked
    last, by _on_device, so that every other check also runs without a GPU."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must be {dim}-D, got shape {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _packed(W, name: str, N: int, K: int):
    """A packed Q4 matrix: contiguous uint8 of exactly q4_packed_bytes(N, K) bytes."""
    import torch
    if not isinstance(W, torch.Tensor) or W.dtype != torch.uint8 or not W.is_contiguous():
        raise ValueError(f"{name} must be a contiguous uint8 tensor")
    want = packed_bytes(N, K)
    if want == 0 or W.numel() != want:
        raise ValueError(f"{name} has {W.numel()} bytes, expected {want} for N = {N}, K = {K}")
    return W


def _on_device(*named) -> None:
    """Every tensor on one CUDA device: the library dereferences the pointers there."""
    dev = None
    for name, t in named:
        if not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other arguments on {dev}")


def matmul(x, W, N: int, K: int, y=None, stream=None):
    """y[M, N] (fp32) = x[M, K] (bf16) times the packed Q4 matrix W[N, K]."""
    import torch
    _tensor(x, "x", torch.bfloat16, dim=2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError(f"x has {x.shape[1]} columns, K = {K}")
    _packed(W, "W", N, K)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _tensor(y, "y", torch.float32, shape=(M, N))
    _on_device(("x", x), ("W", W), ("y", y))
    _check(lib().q4_matmul(x.data_ptr(), W.data_ptr(), M, N, K, y.data_ptr(), _stream_handle(stream)))
    return y


def matmul_noalloc(x, W, N: int, K: int, y, stream=None):
    """q4_matmul_noalloc: the same product, with the library's fixed static
    scratch instead of memory it allocates, for callers that may not allocate
    device memory.  y must be given (a contiguous float32 [M, N] tensor)."""
    import torch
    _tensor(x, "x", torch.bfloat16, dim=2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError(f"x has {x.shape[1]} columns, K = {K}")
    _packed(W, "W", N, K)
    _tensor(y, "y", torch.float32, shape=(M, N))
    _on_device(("x", x), ("W", W), ("y", y))
    _check(lib().q4_matmul_noalloc(x.data_ptr(), W.data_ptr(), M, N, K, y.data_ptr(), _stream_handle(stream)))
    return y


def glue(y, K_next: int, kind: int, x_next=None, stream=None):
    """q4_glue: x_next[M, K_next] (bf16) from y[M, N_prev] (fp32), both on the device."""
    import torch
    _tensor(y, "y", torch.float32, dim=2)
    M, n_prev = y.shape
    if x_next is None:
        x_next = torch.empty((M, K_next), dtype=torch.bfloat16, device=y.device)
    _tensor(x_next, "x_next", torch.bfloat16, shape=(M, K_next))
    _on_device(("y", y), ("x_next", x_next))
    _check(lib().q4_glue(y.data_ptr(), M, n_prev, K_next, kind, x_next.data_ptr(), _stream_handle(stream)))
    return x_next


def _layer_array(layers):
    """layers: sequence of (W tensor, N, K, glue) -> ctypes array of q4_layer."""
    arr = (Layer * len(layers))()
    for i, (W, N, K, g) in enumerate(layers):
        arr[i] = Layer(W.data_ptr(), N, K, g)
    return arr


def decode_step_workspace_bytes(layers, M: int) -> int:
    arr = _layer_array(layers)
    return int(lib().q4_decode_step_workspace_bytes(ctypes.addressof(arr), len(layers), M))


def decode_step(layers, x0, y_last=None, workspace=None, stream=None):
    """q4_decode_step over `layers` = [(W, N, K, glue), ...] from x0 [M, K_0]
    (bf16); returns y_last [M, N_last] (fp32).  The workspace (a uint8 device
    tensor) is allocated here when not given."""
    import torch
    _tensor(x0, "x0", torch.bfloat16, dim=2)
    M = x0.shape[0]
    if len(layers) == 0:
        raise ValueError("layers must not be empty")
    for j, (W, N, K, _g) in enumerate(layers):
        _packed(W, f"layers[{j}].W", N, K)
    if x0.shape[1] != layers[0][2]:
        raise ValueError(f"x0 has {x0.shape[1]} columns, the first layer's K = {layers[0][2]}")
    arr = _layer_array(layers)
    need = int(lib().q4_decode_step_workspace_bytes(ctypes.addressof(arr), len(layers), M))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x0.device)
    _tensor(workspace, "workspace", torch.uint8)
    if y_last is None:
        y_last = torch.empty((M, layers[-1][1]), dtype=torch.float32, device=x0.device)
    _tensor(y_last, "y_last", torch.float32, shape=(M, layers[-1][1]))
    _on_device(("x0", x0), ("workspace", workspace), ("y_last", y_last),
               *((f"layers[{j}].W", layer[0]) for j, layer in enumerate(layers)))
    _check(lib().q4_decode_step(ctypes.addressof(arr), len(layers), x0.data_ptr(), M, workspace.data_ptr(),
                                workspace.numel(), y_last.data_ptr(), _stream_handle(stream)))
    return y_last


def matmul_raw(x_ptr: int, W_ptr: int, M: int, N: int, K: int, y_ptr: int, stream_handle: int) -> None:
    """Pointer-level call of q4_matmul (for callers that manage their own buffers)."""
    _check(lib().q4_matmul(x_ptr, W_ptr, M, N, K, y_ptr, stream_handle))


def _topk_outputs(M: int, device, idx, probs):
    import torch
    if idx is None:
        idx = torch.empty((M, 32), dtype=torch.int32, device=device)
    if probs is None:
        probs = torch.empty((M, 32), dtype=torch.float32, device=device)
    _tensor(idx, "idx", torch.int32, shape=(M, 32))
    _tensor(probs, "probs", torch.float32, shape=(M, 32))
    return idx, probs


def topk_probs(logits, top_k: int, temperature: float, top_p: float, idx=None, probs=None, stream=None):
    """Sampling epilogue: (idx int32 [M, 32], probs fp32 [M, 32]) of fp32 device logits [M, N]."""
    import torch
    _tensor(logits, "logits", torch.float32, dim=2)
    M, N = logits.shape
    idx, probs = _topk_outputs(M, logits.device, idx, probs)
    _on_device(("logits", logits), ("idx", idx), ("probs", probs))
    _check(lib().q4_topk_probs(logits.data_ptr(), M, N, int(top_k), float(temperature), float(top_p),
                               idx.data_ptr(), probs.data_ptr(), _stream_handle(stream)))
    return idx, probs


def lm_head_topk(x, W, N: int, K: int, top_k: int, temperature: float, top_p: float, idx=None, probs=None,
                 stream=None):
    """The LM head and its sampling epilogue in one call: (idx int32 [M, 32], probs fp32 [M, 32])
    for bf16 device x [M, K] and the packed head W; the logits stay in the library's scratch."""
    import torch
    _tensor(x, "x", torch.bfloat16, dim=2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError(f"x has {x.shape[1]} columns, K = {K}")
    _packed(W, "W", N, K)
    idx, probs = _topk_outputs(M, x.device, idx, probs)
    _on_device(("x", x), ("W", W), ("idx", idx), ("probs", probs))
    _check(lib().q4_lm_head_topk(x.data_ptr(), W.data_ptr(), M, N, K, int(top_k), float(temperature), float(top_p),
                                 idx.data_ptr(), probs.data_ptr(), _stream_handle(stream)))
    return idx, probs


def draft_select_edges(pred_cb, succ_cb, hidden, pred_ids, cand_ids, score=None, stream=None):
    """Edge scores fp32 [rows, 16, 16] of bf16 codebooks [V, R], fp32 hidden [rows, R]
    and int32 ids [rows, 16] (all device tensors)."""
    import torch
    _tensor(pred_cb, "pred_cb", torch.bfloat16, dim=2)
    V, R = pred_cb.shape
    _tensor(succ_cb, "succ_cb", torch.bfloat16, shape=(V, R))
    _tensor(hidden, "hidden", torch.float32, dim=2)
    rows = hidden.shape[0]
    if hidden.shape[1] != R:
        raise ValueError(f"hidden has {hidden.shape[1]} columns, the codebooks' rank R = {R}")
    _tensor(pred_ids, "pred_ids", torch.int32, shape=(rows, 16))
    _tensor(cand_ids, "cand_ids", torch.int32, shape=(rows, 16))
    if score is None:
        score = torch.empty((rows, 16, 16), dtype=torch.float32, device=hidden.device)
    _tensor(score, "score", torch.float32, shape=(rows, 16, 16))
    _on_device(("pred_cb", pred_cb), ("succ_cb", succ_cb), ("hidden", hidden), ("pred_ids", pred_ids),
               ("cand_ids", cand_ids), ("score", score))
    _check(lib().q4_draft_select_edges(pred_cb.data_ptr(), succ_cb.data_ptr(), V, R, hidden.data_ptr(),
                                       pred_ids.data_ptr(), cand_ids.data_ptr(), rows, score.data_ptr(),
                                       _stream_handle(stream)))
    return score


def check_wait_timeout(limit_cycles: int, stream=None) -> None:
    """Launch the timeout self-check: a bounded wait that runs out after
    `limit_cycles` and is then reported by device_status()."""
    _check(lib().q4_check_wait_timeout(int(limit_cycles), _stream_handle(stream)))


def device_status(stream=None) -> None:
    """Synchronise and raise Q4Error (Q4_ERR_INVALID_INDEX for an out-of-range codebook id,
    Q4_ERR_TIMEOUT for a device-side wait that gave up) if a kernel recorded one."""
    _check(lib().q4_device_status(_stream_handle(stream)))
