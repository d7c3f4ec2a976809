"""ctypes binding of liblogra.so: argument marshalling only.

Each Python function has the name of the C entry point it calls and takes
torch tensors for device buffers.  Every step of the path runs in the
library's kernels; there is no fallback of any kind.  If the shared library
is missing, importing this module raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "liblogra.so")

LOGRA_OK = 0
LOGRA_DTYPE_BF16 = 0
LOGRA_DTYPE_FP32 = 1
LOGRA_PROJ_INT8_PM1 = 0
LOGRA_PROJ_BF16 = 1
LOGRA_PROJ_FP32 = 2
LOGRA_PROJ_GAUSS_BF16 = 3
LOGRA_PROJ_GAUSS_FP32 = 4
LOGRA_PROJ_SIGN_BF16 = 5

STATUS_NAMES = {
    0: "LOGRA_OK", 1: "LOGRA_ERR_INVALID_ARG", 2: "LOGRA_ERR_SHAPE", 3: "LOGRA_ERR_ALIGNMENT",
    4: "LOGRA_ERR_WORKSPACE", 5: "LOGRA_ERR_UNSUPPORTED", 6: "LOGRA_ERR_CUDA", 7: "LOGRA_ERR_DEVICE",
}


class LograError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"liblogra.so not found at {_LIB_PATH}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')"
        )
    return ctypes.CDLL(_LIB_PATH)


lib = _load()

_i64, _u64, _u32, _int, _f32, _f64 = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                                      ctypes.c_float, ctypes.c_double)
_vp, _sz = ctypes.c_void_p, ctypes.c_size_t

lib.logra_last_error.restype = ctypes.c_char_p
lib.logra_last_error.argtypes = []
lib.logra_status_string.restype = ctypes.c_char_p
lib.logra_status_string.argtypes = [_int]
lib.logra_version.restype = _int
lib.logra_version.argtypes = []
lib.logra_sketch_workspace_bytes.restype = _sz
lib.logra_sketch_workspace_bytes.argtypes = [_i64, _i64, _i64, _int]
lib.logra_sketch_splits.restype = _int
lib.logra_sketch_splits.argtypes = [_i64, _i64, _i64, _int]
lib.logra_sketch_accumulate.restype = _int
lib.logra_sketch_accumulate.argtypes = [_vp, _i64, _vp, _i64, _i64, _i64, _i64, _int, _u64, _u32, _vp, _i64, _vp,
                                        _sz, _vp]
class logra_sketch_target(ctypes.Structure):
    _fields_ = [("dY", ctypes.c_void_p), ("lddy", ctypes.c_int64), ("d", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("stream_id", ctypes.c_uint32), ("S", ctypes.c_void_p), ("lds", ctypes.c_int64)]


LOGRA_MAX_SHARED_X_TARGETS = 4
lib.logra_sketch_shared_x_workspace_bytes.restype = _sz
lib.logra_sketch_shared_x_workspace_bytes.argtypes = [_i64, _i64, _int, ctypes.POINTER(_i64), _int]
lib.logra_sketch_accumulate_shared_x.restype = _int
lib.logra_sketch_accumulate_shared_x.argtypes = [_vp, _i64, _i64, _i64, _int, ctypes.POINTER(logra_sketch_target),
                                                 _int, _vp, _sz, _vp]
lib.logra_sketch_accumulate_shared_x_proj.restype = _int
lib.logra_sketch_accumulate_shared_x_proj.argtypes = [_vp, _i64, _i64, _i64, _int, ctypes.POINTER(logra_sketch_target),
                                                      ctypes.POINTER(_vp), ctypes.POINTER(_i64), _int, _vp, _sz, _vp]
lib.logra_sketch_accumulate_proj.restype = _int
lib.logra_sketch_accumulate_proj.argtypes = [_vp, _i64, _vp, _i64, _i64, _i64, _i64, _int, _vp, _i64, _vp, _i64, _vp,
                                             _sz, _vp]
lib.logra_merge_update_proj.restype = _int
lib.logra_merge_update_proj.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _f32, _vp, _vp]
lib.logra_sum_squares_workspace_bytes.restype = _sz
lib.logra_sum_squares_workspace_bytes.argtypes = []
lib.logra_sum_squares.restype = _int
lib.logra_sum_squares.argtypes = [_vp, _int, _i64, _i64, _i64, _vp, _int, _vp, _sz, _vp]
lib.logra_self_test_wait_timeout.restype = _int
lib.logra_self_test_wait_timeout.argtypes = [_vp]
lib.logra_refreshed_seed.restype = _u64
lib.logra_refreshed_seed.argtypes = [_u64, _u64]
lib.logra_merge_update.restype = _int
lib.logra_merge_update.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _int, _u64, _u32, _f32, _vp, _vp]


class logra_merge_target(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("ldw", ctypes.c_int64), ("d", ctypes.c_int64), ("k", ctypes.c_int64),
                ("S", ctypes.c_void_p), ("lds", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("stream_id", ctypes.c_uint32), ("A", ctypes.c_void_p), ("lda", ctypes.c_int64)]


class logra_sketch_group_target(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("dY", ctypes.c_void_p), ("lddy", ctypes.c_int64),
                ("T", ctypes.c_int64), ("d", ctypes.c_int64), ("k", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("stream_id", ctypes.c_uint32), ("A", ctypes.c_void_p), ("lda", ctypes.c_int64),
                ("S", ctypes.c_void_p), ("lds", ctypes.c_int64)]


lib.logra_sketch_group_plan_bytes.restype = _sz
lib.logra_sketch_group_plan_bytes.argtypes = [_int]
lib.logra_sketch_group_workspace_bytes.restype = _sz
lib.logra_sketch_group_workspace_bytes.argtypes = [_int, ctypes.POINTER(logra_sketch_group_target), _int]
lib.logra_sketch_group_plan.restype = _int
lib.logra_sketch_group_plan.argtypes = [_int, ctypes.POINTER(logra_sketch_group_target), _int, _vp, _sz, _vp, _sz]
lib.logra_sketch_accumulate_group.restype = _int
lib.logra_sketch_accumulate_group.argtypes = [_vp, _vp, _vp]
lib.logra_merge_group_plan_bytes.restype = _sz
lib.logra_merge_group_plan_bytes.argtypes = [_int]
lib.logra_merge_group_plan.restype = _int
lib.logra_merge_group_plan.argtypes = [_int, ctypes.POINTER(logra_merge_target), _int, _vp, _sz]
lib.logra_merge_update_group.restype = _int
lib.logra_merge_update_group.argtypes = [_vp, _vp, _f32, _vp, _vp]
lib.logra_sketch_momentum.restype = _int
lib.logra_sketch_momentum.argtypes = [_vp, _i64, _vp, _i64, _i64, _int, _f32, _int, _vp]
lib.logra_regen_projection.restype = _int
lib.logra_regen_projection.argtypes = [_u64, _u32, _int, _i64, _int, _vp, _i64, _vp]
lib.logra_kl_workspace_bytes.restype = _sz
lib.logra_kl_workspace_bytes.argtypes = [_i64]
lib.logra_predicted_kl.restype = _int
lib.logra_predicted_kl.argtypes = [_vp, _vp, _int, _i64, _i64, _i64, _f32, _vp, _vp, _vp, _vp, _sz, _vp]
lib.logra_predicted_kl_noalloc.restype = _int
lib.logra_predicted_kl_noalloc.argtypes = [_vp, _vp, _int, _i64, _i64, _i64, _f32, _vp, _vp, _vp, _vp]
lib.logra_step_size.restype = _int
lib.logra_step_size.argtypes = [_f64, _f64, _f64, ctypes.POINTER(_f64)]
lib.logra_step_size_device.restype = _int
lib.logra_step_size_device.argtypes = [_vp, _f64, _f64, _f64, _vp, _vp, _vp]
lib.logra_device_error.restype = _int
lib.logra_device_error.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint)]


def _check(status: int) -> None:
    if status != LOGRA_OK:
        raise LograError(status, lib.logra_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _torch_stream(stream, device=None) -> torch.cuda.Stream:
    """A torch stream object for `stream` (None: the current stream; a raw
    cudaStream_t handle is wrapped without taking ownership)."""
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def _row_major(t: torch.Tensor, name: str) -> int:
    """The row stride (elements) of a 2-D row-major tensor.  A tensor with at
    most one row, or no elements, has no meaningful row stride (torch may give
    it any value), so any stride of at least one row serves."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D row-major tensor with unit inner stride")
    rows, cols = t.shape
    if cols > 1 and rows > 0 and t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major tensor with unit inner stride")
    if rows <= 1 or cols == 0:
        return max(t.stride(0), cols)
    return t.stride(0)


def logra_version() -> int:
    return lib.logra_version()


def logra_last_error() -> str:
    return lib.logra_last_error().decode(errors="replace")


def logra_sketch_workspace_bytes(T: int, d: int, k: int, r: int) -> int:
    return int(lib.logra_sketch_workspace_bytes(T, d, k, r))


def logra_sketch_splits(T: int, d: int, k: int, r: int) -> int:
    return int(lib.logra_sketch_splits(T, d, k, r))


def sketch_workspace(T: int, d: int, k: int, r: int, device) -> torch.Tensor:
    """A uint8 device buffer large enough for logra_sketch_accumulate."""
    return torch.empty(max(1, logra_sketch_workspace_bytes(T, d, k, r)), dtype=torch.uint8, device=device)


def logra_sketch_accumulate(X: torch.Tensor, dY: torch.Tensor, S: torch.Tensor, seed: int, stream_id: int, r: int,
                            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """S += dYᵀ (X Aᵀ) in place; X bf16 T×k, dY bf16 T×d, S fp32 d×r."""
    if X.dtype != torch.bfloat16 or dY.dtype != torch.bfloat16 or S.dtype != torch.float32:
        raise TypeError("X and dY must be bfloat16 and S float32")
    ldx, lddy, lds = _row_major(X, "X"), _row_major(dY, "dY"), _row_major(S, "S")
    T, k = X.shape
    d = dY.shape[1]
    if dY.shape[0] != T or S.shape[0] != d or S.shape[1] != r:
        raise ValueError("shapes must be X T×k, dY T×d, S d×r")
    if workspace is None:
        workspace = sketch_workspace(T, d, k, r, X.device)
    _check(lib.logra_sketch_accumulate(_ptr(X), ldx, _ptr(dY), lddy, T, d, k, r, seed, stream_id, _ptr(S), lds,
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))
    return S


def _operand(A: torch.Tensor, r: int, k: int) -> int:
    if A.dtype != torch.bfloat16 or A.dim() != 2 or A.shape[0] != r or A.shape[1] != k:
        raise ValueError("the projection operand must be bfloat16 r×k")
    return _row_major(A, "A")


def logra_sketch_accumulate_proj(X: torch.Tensor, dY: torch.Tensor, S: torch.Tensor, A: torch.Tensor, r: int,
                                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """S += (1/√r)·dYᵀ(X Ãᵀ) in place with a given bf16 operand Ã (r×k)."""
    if X.dtype != torch.bfloat16 or dY.dtype != torch.bfloat16 or S.dtype != torch.float32:
        raise TypeError("X and dY must be bfloat16 and S float32")
    ldx, lddy, lds = _row_major(X, "X"), _row_major(dY, "dY"), _row_major(S, "S")
    T, k = X.shape
    d = dY.shape[1]
    if dY.shape[0] != T or S.shape[0] != d or S.shape[1] != r:
        raise ValueError("shapes must be X T×k, dY T×d, S d×r")
    lda = _operand(A, r, k)
    if workspace is None:
        workspace = sketch_workspace(T, d, k, r, X.device)
    _check(lib.logra_sketch_accumulate_proj(_ptr(X), ldx, _ptr(dY), lddy, T, d, k, r, _ptr(A), lda, _ptr(S), lds,
                                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _stream(stream)))
    return S


def logra_sum_squares(x: torch.Tensor, out: torch.Tensor, accumulate: bool = False,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """‖x‖_F² (fp32 or bf16 2-D x) into the device fp64 scalar `out` (added to it when accumulate)."""
    dtype = {torch.bfloat16: LOGRA_DTYPE_BF16, torch.float32: LOGRA_DTYPE_FP32}.get(x.dtype)
    if dtype is None:
        raise TypeError("x must be bfloat16 or float32")
    if out.dtype != torch.float64 or out.numel() != 1:
        raise TypeError("out must be one float64 element")
    ld = _row_major(x, "x")
    if workspace is None:
        workspace = torch.empty(int(lib.logra_sum_squares_workspace_bytes()), dtype=torch.uint8, device=x.device)
    _check(lib.logra_sum_squares(_ptr(x), dtype, x.shape[0], x.shape[1], ld, _ptr(out), int(bool(accumulate)),
                                 _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def logra_refreshed_seed(base_seed: int, step: int) -> int:
    """Seed of step `step` of a refreshed projection basis."""
    return int(lib.logra_refreshed_seed(base_seed, step))


def logra_sketch_shared_x_workspace_bytes(T: int, k: int, ds, r: int) -> int:
    arr = (ctypes.c_int64 * len(ds))(*ds)
    return int(lib.logra_sketch_shared_x_workspace_bytes(T, k, len(ds), arr, r))


def logra_sketch_accumulate_shared_x(X: torch.Tensor, targets, r: int, workspace: torch.Tensor | None = None,
                                     stream=None) -> None:
    """S_j += dY_jᵀ (X A_jᵀ) for targets [(dY_j, S_j, seed_j, stream_id_j)] that share X (one read of X)."""
    if X.dtype != torch.bfloat16:
        raise TypeError("X must be bfloat16")
    ldx = _row_major(X, "X")
    T, k = X.shape
    arr = (logra_sketch_target * len(targets))()
    for j, (dY, S, seed, sid) in enumerate(targets):
        if dY.dtype != torch.bfloat16 or S.dtype != torch.float32:
            raise TypeError("dY must be bfloat16 and S float32")
        if dY.shape[0] != T or S.shape[0] != dY.shape[1] or S.shape[1] != r:
            raise ValueError("shapes must be dY T×d and S d×r")
        arr[j] = logra_sketch_target(_ptr(dY), _row_major(dY, "dY"), dY.shape[1], seed, sid, _ptr(S),
                                     _row_major(S, "S"))
    if workspace is None:
        workspace = torch.empty(max(1, logra_sketch_shared_x_workspace_bytes(T, k, [t[0].shape[1] for t in targets],
                                                                             r)),
                                dtype=torch.uint8, device=X.device)
    _check(lib.logra_sketch_accumulate_shared_x(_ptr(X), ldx, T, k, len(targets), arr, r, _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream(stream)))


def logra_sketch_accumulate_shared_x_proj(X: torch.Tensor, targets, r: int, workspace: torch.Tensor | None = None,
                                          stream=None) -> None:
    """S_j += (1/√r)·dY_jᵀ(X Ã_jᵀ) for targets [(dY_j, S_j, Ã_j)] that share X, Ã_j a bf16 r×k operand."""
    if X.dtype != torch.bfloat16:
        raise TypeError("X must be bfloat16")
    ldx = _row_major(X, "X")
    T, k = X.shape
    n = len(targets)
    arr = (logra_sketch_target * n)()
    ops = (_vp * n)()
    ldas = (_i64 * n)()
    for j, (dY, S, A) in enumerate(targets):
        if dY.dtype != torch.bfloat16 or S.dtype != torch.float32:
            raise TypeError("dY must be bfloat16 and S float32")
        if dY.shape[0] != T or S.shape[0] != dY.shape[1] or S.shape[1] != r:
            raise ValueError("shapes must be dY T×d and S d×r")
        ldas[j] = _operand(A, r, k)
        ops[j] = _ptr(A)
        arr[j] = logra_sketch_target(_ptr(dY), _row_major(dY, "dY"), dY.shape[1], 0, 0, _ptr(S), _row_major(S, "S"))
    if workspace is None:
        workspace = torch.empty(max(1, logra_sketch_shared_x_workspace_bytes(T, k, [t[0].shape[1] for t in targets],
                                                                             r)),
                                dtype=torch.uint8, device=X.device)
    _check(lib.logra_sketch_accumulate_shared_x_proj(_ptr(X), ldx, T, k, n, arr, ops, ldas, r, _ptr(workspace),
                                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def logra_merge_update(W: torch.Tensor, S: torch.Tensor, seed: int, stream_id: int, r: int, alpha_eta: float,
                       alpha_eta_dev: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """W ← bf16(W − αη·S·A) in place; W bf16 d×k, S fp32 d×r."""
    if W.dtype != torch.bfloat16 or S.dtype != torch.float32:
        raise TypeError("W must be bfloat16 and S float32")
    if alpha_eta_dev is not None and alpha_eta_dev.dtype != torch.float32:
        raise TypeError("alpha_eta_dev must be float32")
    ldw, lds = _row_major(W, "W"), _row_major(S, "S")
    d, k = W.shape
    if S.shape[0] != d or S.shape[1] != r:
        raise ValueError("S must be d×r")
    _check(lib.logra_merge_update(_ptr(W), ldw, d, k, _ptr(S), lds, r, seed, stream_id, float(alpha_eta),
                                  _ptr(alpha_eta_dev), _stream(stream)))
    return W


def logra_merge_update_proj(W: torch.Tensor, S: torch.Tensor, A: torch.Tensor, r: int, alpha_eta: float,
                            alpha_eta_dev: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """W ← bf16(W − (αη/√r)·S·Ã) in place with a given bf16 operand Ã (r×k)."""
    if W.dtype != torch.bfloat16 or S.dtype != torch.float32:
        raise TypeError("W must be bfloat16 and S float32")
    if alpha_eta_dev is not None and alpha_eta_dev.dtype != torch.float32:
        raise TypeError("alpha_eta_dev must be float32")
    ldw, lds = _row_major(W, "W"), _row_major(S, "S")
    d, k = W.shape
    if S.shape[0] != d or S.shape[1] != r:
        raise ValueError("S must be d×r")
    lda = _operand(A, r, k)
    _check(lib.logra_merge_update_proj(_ptr(W), ldw, d, k, _ptr(S), lds, r, _ptr(A), lda, float(alpha_eta),
                                       _ptr(alpha_eta_dev), _stream(stream)))
    return W


def _aligned_view(buf: torch.Tensor, nbytes: int, align: int = 128) -> torch.Tensor:
    off = (-buf.data_ptr()) % align
    return buf[off:off + nbytes]


class MergeGroupPlan:
    """A plan of logra_merge_update_group: its host copy (pinned), its device
    copy and the tensors it points at (kept alive with the plan)."""

    def __init__(self, host: torch.Tensor, dev: torch.Tensor, n: int, r: int, tensors: list):
        self.host, self.dev, self.n, self.r = host, dev, n, r
        self._tensors = tensors


class SketchGroupPlan:
    """A plan of logra_sketch_accumulate_group: its host copy (pinned), its
    device copy, the workspace it lays out and the tensors it points at (kept
    alive with the plan)."""

    def __init__(self, host: torch.Tensor, dev: torch.Tensor, workspace: torch.Tensor, n: int, r: int,
                 tensors: list):
        self.host, self.dev, self.workspace, self.n, self.r = host, dev, workspace, n, r
        self._tensors = tensors


def _sketch_group_targets(targets, r: int):
    n = len(targets)
    arr = (logra_sketch_group_target * max(n, 1))()
    keep = []
    for j, t in enumerate(targets):
        if len(t) == 5:
            X, dY, S, seed, sid = t
            A, lda = None, 0
        else:
            X, dY, S, A = t
            seed, sid = 0, 0
            lda = _operand(A, r, X.shape[1])
        if X.dtype != torch.bfloat16 or dY.dtype != torch.bfloat16 or S.dtype != torch.float32:
            raise TypeError("X and dY must be bfloat16 and S float32")
        T, k = X.shape
        d = dY.shape[1]
        if dY.shape[0] != T or S.shape[0] != d or S.shape[1] != r:
            raise ValueError("X is T×k, dY T×d and S d×r")
        arr[j] = logra_sketch_group_target(_ptr(X), _row_major(X, "X"), _ptr(dY), _row_major(dY, "dY"), T, d, k,
                                           seed, sid, _ptr(A), lda, _ptr(S), _row_major(S, "S"))
        keep += [X, dY, S] + ([A] if A is not None else [])
    return arr, keep


def logra_sketch_group_plan_bytes(n: int) -> int:
    return lib.logra_sketch_group_plan_bytes(n)


def logra_sketch_group_workspace_bytes(targets, r: int) -> int:
    arr, _ = _sketch_group_targets(targets, r)
    return int(lib.logra_sketch_group_workspace_bytes(len(targets), arr, r))


def logra_sketch_group_plan(targets, r: int, workspace: torch.Tensor | None = None, device=None, stream=None,
                            reuse: SketchGroupPlan | None = None) -> SketchGroupPlan:
    """Plan the sketch of several matrices with one launch per phase.

    targets: [(X, dY, S, seed, stream_id)] (signs from the seed) or
    [(X, dY, S, A)] (a bf16 r×k operand), X bf16 T×k, dY bf16 T×d, S fp32 d×r.
    The workspace is `workspace`, else that of `reuse` when large enough,
    else a new device buffer; the plan is written into pinned host memory and
    copied to the device on `stream` (default: the current stream)."""
    n = len(targets)
    arr, keep = _sketch_group_targets(targets, r)
    ws_bytes = int(lib.logra_sketch_group_workspace_bytes(n, arr, r))
    nbytes = lib.logra_sketch_group_plan_bytes(n)
    host = _aligned_view(torch.empty(nbytes + 128, dtype=torch.uint8, pin_memory=True), nbytes)
    if device is None:
        device = targets[0][0].device if n else torch.device("cuda")
    s = _torch_stream(stream, device)
    # Device buffers are allocated and filled on the plan's stream, so the
    # caching allocator only hands their memory to work ordered after it.
    with torch.cuda.stream(s):
        if workspace is None:
            if reuse is not None and reuse.workspace.numel() >= ws_bytes:
                workspace = reuse.workspace
            else:
                workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
        _check(lib.logra_sketch_group_plan(n, arr, r, _ptr(workspace), workspace.numel(), _ptr(host), nbytes))
        if reuse is not None and reuse.dev.numel() >= nbytes:
            dev = reuse.dev[:nbytes]
        else:
            dev = _aligned_view(torch.empty(nbytes + 128, dtype=torch.uint8, device=device), nbytes)
        dev.copy_(host, non_blocking=True)
    return SketchGroupPlan(host, dev, workspace, n, r, keep)


def logra_sketch_accumulate_group(plan: SketchGroupPlan, stream=None) -> None:
    """S_j += (1/√r)·dY_jᵀ(X_j A_jᵀ) for every target of the plan, one launch
    per phase.  The launch must be ordered after the plan's copy to the
    device: launch on the stream the plan was built with, or make this stream
    wait for it."""
    _check(lib.logra_sketch_accumulate_group(_ptr(plan.host), _ptr(plan.dev), _stream(stream)))


def logra_merge_group_plan_bytes(n: int) -> int:
    return lib.logra_merge_group_plan_bytes(n)


def logra_merge_group_plan(targets, r: int, device=None, stream=None,
                           reuse: MergeGroupPlan | None = None) -> MergeGroupPlan:
    """Plan the merge of several weights in one launch.

    targets: [(W, S, seed, stream_id)] (signs from the seed) or [(W, S, A)]
    (a bf16 r×k operand per weight), W bf16 d×k, S fp32 d×r.  The plan is
    written into pinned host memory and copied to the device on `stream`
    (default: the current stream), into the device buffer of `reuse` when it
    is large enough (stream order keeps earlier launches reading the old
    plan ahead of the copy)."""
    n = len(targets)
    arr = (logra_merge_target * max(n, 1))()
    keep = []
    for j, t in enumerate(targets):
        if len(t) == 4:
            W, S, seed, sid = t
            A, lda = None, 0
        else:
            W, S, A = t
            seed, sid = 0, 0
            lda = _operand(A, r, W.shape[1])
        if W.dtype != torch.bfloat16 or S.dtype != torch.float32:
            raise TypeError("W must be bfloat16 and S float32")
        d, k = W.shape
        if S.shape[0] != d or S.shape[1] != r:
            raise ValueError("S must be d×r")
        arr[j] = logra_merge_target(_ptr(W), _row_major(W, "W"), d, k, _ptr(S), _row_major(S, "S"), seed, sid,
                                    _ptr(A), lda)
        keep += [W, S] + ([A] if A is not None else [])
    nbytes = lib.logra_merge_group_plan_bytes(n)
    host = _aligned_view(torch.empty(nbytes + 128, dtype=torch.uint8, pin_memory=True), nbytes)
    _check(lib.logra_merge_group_plan(n, arr, r, _ptr(host), nbytes))
    if device is None:
        device = targets[0][0].device if n else torch.device("cuda")
    s = _torch_stream(stream, device)
    # The device copy is allocated and filled on the plan's stream, so the
    # caching allocator only hands its memory to work ordered after it.
    with torch.cuda.stream(s):
        if reuse is not None and reuse.dev.numel() >= nbytes:
            dev = reuse.dev[:nbytes]
        else:
            dev = _aligned_view(torch.empty(nbytes + 128, dtype=torch.uint8, device=device), nbytes)
        dev.copy_(host, non_blocking=True)
    return MergeGroupPlan(host, dev, n, r, keep)


def logra_merge_update_group(plan: MergeGroupPlan, alpha_eta: float, alpha_eta_dev: torch.Tensor | None = None,
                             stream=None) -> None:
    """W_j ← bf16(W_j − αη·S_j·A_j) for every weight of the plan, in one launch.

    The launch must be ordered after the plan's copy to the device: launch on
    the stream the plan was built with, or make this stream wait for it."""
    if alpha_eta_dev is not None and alpha_eta_dev.dtype != torch.float32:
        raise TypeError("alpha_eta_dev must be float32")
    _check(lib.logra_merge_update_group(_ptr(plan.host), _ptr(plan.dev), float(alpha_eta), _ptr(alpha_eta_dev),
                                        _stream(stream)))


def logra_sketch_momentum(M: torch.Tensor, S: torch.Tensor, beta: float, clear_s: bool = False,
                          stream=None) -> torch.Tensor:
    """M ← β·M + S in place (and S ← 0 when clear_s); both fp32 d×r."""
    if M.dtype != torch.float32 or S.dtype != torch.float32:
        raise TypeError("M and S must be float32")
    if M.dim() != 2 or M.shape != S.shape:
        raise ValueError("M and S must be d×r of the same shape")
    ldm, lds = _row_major(M, "M"), _row_major(S, "S")
    d, r = M.shape
    _check(lib.logra_sketch_momentum(_ptr(M), ldm, _ptr(S), lds, d, r, float(beta), int(bool(clear_s)),
                                     _stream(stream)))
    return M


def logra_regen_projection(seed: int, stream_id: int, r: int, k: int, out_kind: int = LOGRA_PROJ_INT8_PM1,
                           out: torch.Tensor | None = None, device="cuda", stream=None) -> torch.Tensor:
    dt = {LOGRA_PROJ_INT8_PM1: torch.int8, LOGRA_PROJ_BF16: torch.bfloat16, LOGRA_PROJ_FP32: torch.float32,
          LOGRA_PROJ_GAUSS_BF16: torch.bfloat16, LOGRA_PROJ_GAUSS_FP32: torch.float32,
          LOGRA_PROJ_SIGN_BF16: torch.bfloat16}[out_kind]
    if out is None:
        out = torch.empty((r, k), dtype=dt, device=device)
    lda = _row_major(out, "out")
    _check(lib.logra_regen_projection(seed, stream_id, r, k, out_kind, _ptr(out), lda, _stream(stream)))
    return out


def logra_kl_workspace_bytes(rows: int) -> int:
    return int(lib.logra_kl_workspace_bytes(rows))


def logra_predicted_kl(cur: torch.Tensor, prop: torch.Tensor, temperature: float = 1.0,
                       row_mask: torch.Tensor | None = None, q_out: torch.Tensor | None = None,
                       row_kl_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """q(D) into a device fp64 scalar tensor (returned); rows × V logits."""
    if cur.dtype != prop.dtype or cur.shape != prop.shape or cur.stride() != prop.stride():
        raise ValueError("cur and prop must have the same dtype, shape and strides")
    dtype = {torch.bfloat16: LOGRA_DTYPE_BF16, torch.float32: LOGRA_DTYPE_FP32}.get(cur.dtype)
    if dtype is None:
        raise TypeError("logits must be bfloat16 or float32")
    ld = _row_major(cur, "cur")
    rows, V = cur.shape
    if row_mask is not None and (row_mask.dtype != torch.uint8 or row_mask.numel() != rows):
        raise ValueError("row_mask must be uint8 with one entry per row")
    if q_out is None:
        q_out = torch.empty((), dtype=torch.float64, device=cur.device)
    if workspace is None:
        workspace = torch.empty(logra_kl_workspace_bytes(rows), dtype=torch.uint8, device=cur.device)
    _check(lib.logra_predicted_kl(_ptr(cur), _ptr(prop), dtype, rows, V, ld, float(temperature), _ptr(row_mask),
                                  _ptr(q_out), _ptr(row_kl_out), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))
    return q_out


LOGRA_KL_NOALLOC_MAX_ROWS = 65536


def logra_predicted_kl_noalloc(cur: torch.Tensor, prop: torch.Tensor, temperature: float = 1.0,
                               row_mask: torch.Tensor | None = None, q_out: torch.Tensor | None = None,
                               row_kl_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q(D) like logra_predicted_kl, with no workspace: for callers that can
    not hand the library device memory (see include/logra.h).  At most
    LOGRA_KL_NOALLOC_MAX_ROWS rows; calls must not overlap on the GPU."""
    if cur.dtype != prop.dtype or cur.shape != prop.shape or cur.stride() != prop.stride():
        raise ValueError("cur and prop must have the same dtype, shape and strides")
    dtype = {torch.bfloat16: LOGRA_DTYPE_BF16, torch.float32: LOGRA_DTYPE_FP32}.get(cur.dtype)
    if dtype is None:
        raise TypeError("logits must be bfloat16 or float32")
    ld = _row_major(cur, "cur")
    rows, V = cur.shape
    if q_out is None:
        q_out = torch.empty((), dtype=torch.float64, device=cur.device)
    _check(lib.logra_predicted_kl_noalloc(_ptr(cur), _ptr(prop), dtype, rows, V, ld, float(temperature),
                                          _ptr(row_mask), _ptr(q_out), _ptr(row_kl_out), _stream(stream)))
    return q_out


def logra_step_size(q: float, delta: float, alpha_max: float) -> float:
    out = ctypes.c_double()
    _check(lib.logra_step_size(float(q), float(delta), float(alpha_max), ctypes.byref(out)))
    return out.value


def logra_step_size_device(q_dev: torch.Tensor, delta: float, alpha_max: float, eta: float,
                           alpha_eta_out: torch.Tensor, alpha_out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    if q_dev.dtype != torch.float64 or alpha_eta_out.dtype != torch.float32:
        raise TypeError("q_dev must be float64 and alpha_eta_out float32")
    if alpha_out is not None and alpha_out.dtype != torch.float64:
        raise TypeError("alpha_out must be float64")
    _check(lib.logra_step_size_device(_ptr(q_dev), float(delta), float(alpha_max), float(eta), _ptr(alpha_eta_out),
                                      _ptr(alpha_out), _stream(stream)))
    return alpha_eta_out


def logra_self_test_wait_timeout(stream=None) -> None:
    """Enqueues the failure-reporting self-test (a bounded wait that runs out, code 7)."""
    _check(lib.logra_self_test_wait_timeout(_stream(stream)))


def logra_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the kernels' error code."""
    code = ctypes.c_uint(0)
    st = lib.logra_device_error(_stream(stream), ctypes.byref(code))
    if st not in (LOGRA_OK, 7):
        _check(st)
    return int(code.value)
