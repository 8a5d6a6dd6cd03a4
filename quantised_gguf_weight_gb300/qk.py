"""Python binding of libqk (include/qk.h): argument marshalling only.

Every call forwards device pointers, sizes and the current torch CUDA stream
to the C ABI; all the work runs in the library's CUDA kernels.  There is no
fallback: if the library is missing or fails to load, every call raises.
PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

QK_OK = 0
STATUS = {0: "QK_OK", 1: "QK_ERR_NULL", 2: "QK_ERR_BAD_DIM", 3: "QK_ERR_ALIGN", 4: "QK_ERR_BATCH",
          5: "QK_ERR_CUDA", 6: "QK_ERR_TIMEOUT", 7: "QK_ERR_WORKSPACE", 8: "QK_ERR_TOO_LARGE",
          9: "QK_ERR_BAD_INDEX"}
MAX_BATCH = 8

EXPORTS = ["qmatvec_q8_0", "qmatvec_q4_k", "qmatvec_q6_k", "qmatvec_swiglu_q8_0", "qmatvec_swiglu_q4_k",
           "qmatvec_swiglu_q6_k", "qmatvec_experts_q8_0", "qmatvec_experts_q4_k", "qmatvec_experts_q6_k",
           "qk_row_bytes_q6_k", "qgemm_q4_k", "qgemm_q4_k_acc", "qgemm_swiglu_q4_k", "qgemm_q8_0",
           "qgemm_q8_0_acc", "qgemm_swiglu_q8_0", "qgemm_q4_k_workspace_bytes",
           "qgemm_q4_k_noalloc", "qk_row_bytes_q8_0", "qk_row_bytes_q4_k",
           "qk_status_string", "qk_device_error", "qk_set_wait_limit_ns", "qk_set_programmatic_launch",
           "qk_set_strict_blocks", "qk_version"]


class QKError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = load().qk_status_string(status).decode()
        super().__init__(f"{what}: {STATUS.get(status, status)} ({msg})")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the in-tree libqk.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"libqk.so not built ({p}); run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        for name in ("qmatvec_q8_0", "qmatvec_q4_k", "qmatvec_q6_k"):
            fn = getattr(lib, name)
            fn.argtypes = [P, I64, I64, I64, P, I, P, I64, P]
            fn.restype = I
        for name in ("qmatvec_swiglu_q8_0", "qmatvec_swiglu_q4_k", "qmatvec_swiglu_q6_k"):
            fn = getattr(lib, name)
            fn.argtypes = [P, I64, I64, I64, I64, P, I, P, I64, P]
            fn.restype = I
        for name in ("qmatvec_experts_q8_0", "qmatvec_experts_q4_k", "qmatvec_experts_q6_k"):
            fn = getattr(lib, name)
            fn.argtypes = [P, I64, I64, I64, P, I, P, I64, P, I64, P]
            fn.restype = I
        for name in ("qgemm_q4_k", "qgemm_q4_k_acc", "qgemm_q8_0", "qgemm_q8_0_acc"):
            getattr(lib, name).argtypes = [P, I64, I64, I64, P, I64, P, I64, P, ctypes.c_size_t, P]
            getattr(lib, name).restype = I
        for name in ("qgemm_swiglu_q4_k", "qgemm_swiglu_q8_0"):
            getattr(lib, name).argtypes = [P, I64, I64, I64, I64, P, I64, P, I64, P, ctypes.c_size_t, P]
            getattr(lib, name).restype = I
        lib.qgemm_q4_k_workspace_bytes.argtypes = [I64, I64, I64]
        lib.qgemm_q4_k_workspace_bytes.restype = ctypes.c_size_t
        lib.qk_debug_gemm_skip_chunk.argtypes = [I]
        lib.qk_debug_gemm_skip_chunk.restype = I
        for name in ("qk_row_bytes_q8_0", "qk_row_bytes_q4_k", "qk_row_bytes_q6_k"):
            getattr(lib, name).argtypes = [I64]
            getattr(lib, name).restype = I64
        lib.qk_status_string.argtypes = [I]
        lib.qk_status_string.restype = ctypes.c_char_p
        lib.qk_device_error.argtypes = [P]
        lib.qk_device_error.restype = I
        lib.qk_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.qk_set_wait_limit_ns.restype = ctypes.c_uint64
        lib.qk_version.restype = I
        lib.qk_set_programmatic_launch.argtypes = [I]
        lib.qk_set_programmatic_launch.restype = I
        lib.qk_set_strict_blocks.argtypes = [I]
        lib.qk_set_strict_blocks.restype = I
        lib.qk_debug_skip_item.argtypes = [I64]
        lib.qk_debug_skip_item.restype = I64
        lib.qk_debug_gemv_plan.argtypes = [I, I64, I64, I, ctypes.POINTER(ctypes.c_int64), I]
        lib.qk_debug_gemv_plan.restype = I
        lib.qk_debug_gemv_plan_for.argtypes = [I, I64, I64, I, I, I64, I, I, ctypes.POINTER(ctypes.c_int64), I]
        lib.qk_debug_gemv_plan_for.restype = I
        lib.qk_debug_gemv_tc.argtypes = [I]
        lib.qk_debug_gemv_tc.restype = I
        lib.qk_debug_gemv_tc_plan_for.argtypes = [I, I64, I64, I, I, ctypes.POINTER(ctypes.c_int64), I]
        lib.qk_debug_gemv_tc_plan_for.restype = I
        _lib = lib
        return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def row_bytes(fmt: str, K: int) -> int:
    lib = load()
    return int({"q8_0": lib.qk_row_bytes_q8_0, "q4_k": lib.qk_row_bytes_q4_k, "q6_k": lib.qk_row_bytes_q6_k}[fmt](K))


def _check(status: int, what: str):
    if status != QK_OK:
        raise QKError(status, what)


def _on_device(t, name: str, dtype=None) -> None:
    """A tensor the library reads or writes through its data pointer: a CUDA
    tensor on the current device, of the given dtype."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, not {t.dtype}")


def _bytes_after(t: torch.Tensor) -> int:
    """Bytes from t's first element to the end of its storage."""
    return t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()


def _check_w(w, rows_end: int, rb: int) -> None:
    """Weight bytes: rows [0, rows_end) of rb bytes each, contiguous from w."""
    _on_device(w, "w")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    if rows_end * rb > _bytes_after(w):
        raise ValueError(f"w holds {_bytes_after(w)} bytes, the call reads {rows_end * rb}")


def _check_x(x, K: int, name: str = "x") -> None:
    """Activations [n][K] fp32, row stride K."""
    _on_device(x, name, torch.float32)
    if x.dim() != 2 or x.shape[1] != K or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [n][{K}] tensor, got shape {tuple(x.shape)}")


def _check_out(y, n: int, cols: int, ld: int, name: str = "y") -> None:
    """Output rows b < n of `cols` fp32 values, row b at element b*ld of y: a
    [>= n][>= cols] tensor whose rows are ld apart, or a flat one."""
    _on_device(y, name, torch.float32)
    if y.dim() == 0 or y.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride in its last dimension")
    ld = ld or cols
    if y.dim() == 2:
        if y.shape[0] < n or y.shape[1] < cols:
            raise ValueError(f"{name} {tuple(y.shape)} is too small for {n} rows of {cols}")
        if n > 1 and y.stride(0) != ld:
            raise ValueError(f"{name} rows are {y.stride(0)} elements apart, the call writes them {ld} apart")
    elif not y.is_contiguous() or y.numel() < (n - 1) * ld + cols:
        raise ValueError(f"{name} is too small for {n} rows of {cols} at stride {ld} (or not contiguous)")
    if ((n - 1) * ld + cols) * 4 > _bytes_after(y):
        raise ValueError(f"{name} is too small for {n} rows of {cols} at stride {ld}")


def _fmt_row_bytes(fmt: str, K: int) -> int:
    """Row bytes computed here (no library call), for the binding's checks."""
    if K <= 0:
        return 0
    return {"q8_0": -(-K // 32) * 34, "q4_k": -(-K // 256) * 144, "q6_k": -(-K // 256) * 210}[fmt]


def _qmatvec(name: str, w: torch.Tensor, row_offset: int, rows: int, K: int, x: torch.Tensor,
             y: torch.Tensor | None, ldy: int, stream) -> torch.Tensor:
    if isinstance(x, torch.Tensor) and x.dim() == 1:
        x = x.view(1, -1)
    _check_x(x, K)
    batch = x.shape[0]
    if rows > 0 and row_offset >= 0:
        _check_w(w, row_offset + rows, _fmt_row_bytes(name[-4:], K))
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
        ldy = rows
    if rows > 0:
        _check_out(y, batch, rows, ldy)
    st = getattr(load(), name)(w.data_ptr(), row_offset, rows, K, x.data_ptr(), batch, y.data_ptr(),
                               ldy, _stream(stream))
    _check(st, name)
    return y


def qmatvec_q8_0(w: torch.Tensor, row_offset: int, rows: int, K: int, x: torch.Tensor,
                 y: torch.Tensor | None = None, ldy: int = 0, stream=None) -> torch.Tensor:
    """y[b][r] = sum_c W[row_offset + r][c] x[b][c] for Q8_0 block bytes `w` (uint8, device)."""
    return _qmatvec("qmatvec_q8_0", w, row_offset, rows, K, x, y, ldy, stream)


def qmatvec_q4_k(w: torch.Tensor, row_offset: int, rows: int, K: int, x: torch.Tensor,
                 y: torch.Tensor | None = None, ldy: int = 0, stream=None) -> torch.Tensor:
    """y[b][r] = sum_c W[row_offset + r][c] x[b][c] for Q4_K block bytes `w` (uint8, device)."""
    return _qmatvec("qmatvec_q4_k", w, row_offset, rows, K, x, y, ldy, stream)


def qmatvec_swiglu(fmt: str, w: torch.Tensor, gate_offset: int, up_offset: int, F: int, K: int,
                   x: torch.Tensor, h: torch.Tensor | None = None, ldh: int = 0, stream=None) -> torch.Tensor:
    """h[b][p] = silu(sum_c W[gate_offset+p][c] x[b][c]) * sum_c W[up_offset+p][c] x[b][c], p < F."""
    if isinstance(x, torch.Tensor) and x.dim() == 1:
        x = x.view(1, -1)
    _check_x(x, K)
    batch = x.shape[0]
    if F > 0 and gate_offset >= 0 and up_offset >= 0:
        _check_w(w, max(gate_offset, up_offset) + F, _fmt_row_bytes(fmt, K))
    if h is None:
        h = torch.empty((batch, F), dtype=torch.float32, device=x.device)
        ldh = F
    if F > 0:
        _check_out(h, batch, F, ldh, "h")
    name = {"q8_0": "qmatvec_swiglu_q8_0", "q4_k": "qmatvec_swiglu_q4_k", "q6_k": "qmatvec_swiglu_q6_k"}[fmt]
    st = getattr(load(), name)(w.data_ptr(), gate_offset, up_offset, F, K, x.data_ptr(), batch, h.data_ptr(),
                               ldh, _stream(stream))
    _check(st, name)
    return h


def qmatvec_experts(fmt: str, w: torch.Tensor, n_experts: int, rows: int, K: int, x: torch.Tensor, xk: int,
                    expert_ids: torch.Tensor, y: torch.Tensor | None = None, ldy: int = 0,
                    stream=None) -> torch.Tensor:
    """y[a][r] = sum_c W[expert_ids[a]*rows + r][c] x[a // xk][c] (expert_ids: int32 device tensor)."""
    if isinstance(x, torch.Tensor) and x.dim() == 1:
        x = x.view(1, -1)
    _check_x(x, K)
    _on_device(expert_ids, "expert_ids", torch.int32)
    if not expert_ids.is_contiguous():
        raise ValueError("expert_ids must be contiguous")
    n_assign = expert_ids.numel()
    if n_assign > 0 and xk > 0 and (n_assign - 1) // xk >= x.shape[0]:
        raise ValueError(f"x has {x.shape[0]} rows, assignment {n_assign - 1} reads row {(n_assign - 1) // xk}")
    if n_experts > 0 and rows > 0:
        _check_w(w, n_experts * rows, _fmt_row_bytes(fmt, K))
    if y is None:
        y = torch.empty((n_assign, rows), dtype=torch.float32, device=x.device)
        ldy = rows
    if n_assign > 0 and rows > 0:
        _check_out(y, n_assign, rows, ldy)
    name = {"q8_0": "qmatvec_experts_q8_0", "q4_k": "qmatvec_experts_q4_k", "q6_k": "qmatvec_experts_q6_k"}[fmt]
    st = getattr(load(), name)(w.data_ptr(), n_experts, rows, K, x.data_ptr(), xk, expert_ids.data_ptr(),
                               n_assign, y.data_ptr(), ldy, _stream(stream))
    _check(st, name)
    return y


def qmatvec_q6_k(w: torch.Tensor, row_offset: int, rows: int, K: int, x: torch.Tensor,
                 y: torch.Tensor | None = None, ldy: int = 0, stream=None) -> torch.Tensor:
    """y[b][r] = sum_c W[row_offset + r][c] x[b][c] for Q6_K block bytes `w` (uint8, device)."""
    return _qmatvec("qmatvec_q6_k", w, row_offset, rows, K, x, y, ldy, stream)


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().qgemm_q4_k_workspace_bytes(M, N, K))


def _gemm(name: str, w: torch.Tensor, row_offset: int, N: int, K: int, x: torch.Tensor,
          y: torch.Tensor | None, ldy: int, workspace: torch.Tensor | None, stream) -> torch.Tensor:
    _check_x(x, K)
    M = x.shape[0]
    if N > 0 and row_offset >= 0:
        _check_w(w, row_offset + N, _fmt_row_bytes("q8_0" if "q8_0" in name else "q4_k", K))
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
        ldy = N
    if N > 0 and M > 0:
        _check_out(y, M, N, ldy)
    if workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device=x.device)
    _on_device(workspace, "workspace")
    st = getattr(load(), name)(w.data_ptr(), row_offset, N, K, x.data_ptr(), M, y.data_ptr(), ldy,
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, name)
    return y


def qgemm_q4_k(w: torch.Tensor, row_offset: int, N: int, K: int, x: torch.Tensor,
               y: torch.Tensor | None = None, ldy: int = 0, workspace: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """y[m][n] = sum_c bf16(W[row_offset + n][c]) bf16(x[m][c]) on the tensor cores (Q4_K bytes `w`).

    `workspace` is caller-owned device scratch (uint8) of gemm_workspace_bytes(M, N, K) bytes;
    it is allocated here through torch when not given."""
    return _gemm("qgemm_q4_k", w, row_offset, N, K, x, y, ldy, workspace, stream)


def qgemm_q8_0(w: torch.Tensor, row_offset: int, N: int, K: int, x: torch.Tensor,
               y: torch.Tensor | None = None, ldy: int = 0, workspace: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """qgemm_q4_k for Q8_0 block bytes `w`."""
    return _gemm("qgemm_q8_0", w, row_offset, N, K, x, y, ldy, workspace, stream)


def qgemm_acc(fmt: str, w: torch.Tensor, row_offset: int, N: int, K: int, x: torch.Tensor, y: torch.Tensor,
              ldy: int = 0, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[m][n] += sum_c bf16(W[row_offset + n][c]) bf16(x[m][c]) (in place on `y`)."""
    name = {"q4_k": "qgemm_q4_k_acc", "q8_0": "qgemm_q8_0_acc"}[fmt]
    return _gemm(name, w, row_offset, N, K, x, y, ldy, workspace, stream)


def qgemm_q4_k_acc(w, row_offset, N, K, x, y, ldy=0, workspace=None, stream=None):
    return qgemm_acc("q4_k", w, row_offset, N, K, x, y, ldy, workspace, stream)


def qgemm_swiglu(fmt: str, w: torch.Tensor, gate_offset: int, up_offset: int, F: int, K: int, x: torch.Tensor,
                 h: torch.Tensor | None = None, ldh: int = 0, workspace: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """h[m][p] = silu(g) * u with g, u the bf16 GEMM rows gate_offset + p and up_offset + p."""
    _check_x(x, K)
    M = x.shape[0]
    if F > 0 and gate_offset >= 0 and up_offset >= 0:
        _check_w(w, max(gate_offset, up_offset) + F, _fmt_row_bytes(fmt, K))
    if h is None:
        h = torch.empty((M, F), dtype=torch.float32, device=x.device)
        ldh = F
    if F > 0 and M > 0:
        _check_out(h, M, F, ldh, "h")
    if workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, F, K), dtype=torch.uint8, device=x.device)
    _on_device(workspace, "workspace")
    name = {"q4_k": "qgemm_swiglu_q4_k", "q8_0": "qgemm_swiglu_q8_0"}[fmt]
    st = getattr(load(), name)(w.data_ptr(), gate_offset, up_offset, F, K, x.data_ptr(), M, h.data_ptr(), ldh,
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, name)
    return h


def qgemm_swiglu_q4_k(w, gate_offset, up_offset, F, K, x, h=None, ldh=0, workspace=None, stream=None):
    return qgemm_swiglu("q4_k", w, gate_offset, up_offset, F, K, x, h, ldh, workspace, stream)


def debug_gemm_skip_chunk(chunk: int) -> int:
    """Test hook: CTA 0 of later GEMM launches never loads K chunk `chunk` (-1: off)."""
    return int(load().qk_debug_gemm_skip_chunk(int(chunk)))


def device_error(stream=None) -> int:
    """Synchronise the stream, then read and clear the device error word."""
    return int(load().qk_device_error(_stream(stream)))


def set_wait_limit_ns(ns: int) -> int:
    return int(load().qk_set_wait_limit_ns(int(ns)))


def set_programmatic_launch(enable: bool) -> bool:
    """Programmatic dependent launch for later calls (see include/qk.h)."""
    return bool(load().qk_set_programmatic_launch(1 if enable else 0))


def set_strict_blocks(enable: bool) -> bool:
    """Strict-blocks mode for later calls: a K that is not a whole number of the
    format's blocks is refused with QK_ERR_BAD_DIM (see include/qk.h)."""
    return bool(load().qk_set_strict_blocks(1 if enable else 0))


def debug_skip_item(item: int) -> int:
    """Test hook: in CTA 0 of later GEMV launches, consumer warp 0's item number
    `item` is never copied (-1: off)."""
    return int(load().qk_debug_skip_item(int(item)))


PLAN_FIELDS = ("SW", "R", "nkc", "rows_w", "stages", "stage_bytes", "smem", "grid", "XU", "cpl", "nw", "m")


PLAN_FOR_FIELDS = PLAN_FIELDS + ("LU", "cpa", "off_stage", "wide", "kw")


def debug_gemv_plan_for(fmt: str, rows: int, K: int, batch: int, sms: int, smem_optin: int,
                        pair: bool = False, n_assign: int = 0) -> dict | None:
    """Test hook: the GEMV plan for an explicit device, computed on the host (no GPU needed);
    None if nothing fits."""
    out = (ctypes.c_int64 * len(PLAN_FOR_FIELDS))()
    n = load().qk_debug_gemv_plan_for({"q8_0": 0, "q4_k": 1, "q6_k": 2}[fmt], int(rows), int(K), int(batch),
                                      int(bool(pair)), int(n_assign), int(sms), int(smem_optin), out,
                                      len(PLAN_FOR_FIELDS))
    if n < 0:
        return None
    return dict(zip(PLAN_FOR_FIELDS, list(out)[:n]))


def debug_gemv_tc(mode: int) -> int:
    """Test hook: the tensor-core form of later batch 2..8 GEMV calls: 0 never (the
    fp32 form), 1 where it is the faster form (the default), 2 wherever the format
    and K allow it.  Returns the previous setting."""
    return int(load().qk_debug_gemv_tc(int(mode)))


TC_PLAN_FIELDS = ("G", "NC", "row_stride", "stage_bytes", "NS", "smem", "grid", "off_stage", "off_bop", "ks")


def debug_gemv_tc_plan_for(fmt: str, rows: int, K: int, sms: int, smem_optin: int) -> dict | None:
    """Test hook: the tensor-core GEMV plan (batch 2..8) for an explicit device, computed
    on the host; None when the format and K do not take that form."""
    out = (ctypes.c_int64 * len(TC_PLAN_FIELDS))()
    n = load().qk_debug_gemv_tc_plan_for({"q8_0": 0, "q4_k": 1, "q6_k": 2}[fmt], int(rows), int(K), int(sms),
                                         int(smem_optin), out, len(TC_PLAN_FIELDS))
    if n < 0:
        return None
    return dict(zip(TC_PLAN_FIELDS, list(out)[:n]))


def debug_gemv_plan(fmt: str, rows: int, K: int, batch: int) -> dict:
    """Test hook: the launch plan a GEMV call of this shape uses (needs a GPU)."""
    out = (ctypes.c_int64 * len(PLAN_FIELDS))()
    n = load().qk_debug_gemv_plan({"q8_0": 0, "q4_k": 1, "q6_k": 2}[fmt], int(rows), int(K), int(batch), out, len(PLAN_FIELDS))
    if n < 0:
        raise QKError(8, "no GEMV plan fits")
    return dict(zip(PLAN_FIELDS, list(out)[:n]))
