"""Python binding of libwo, the GB300 weight-only quantized fpA.intB GEMM.

Argument marshalling only: every step runs in the CUDA kernels of
``csrc/`` behind the C ABI declared in ``include/wo.h``.  PyTorch provides
device memory and streams.  There is no CPU fallback: if ``libwo.so`` has
not been built, every call raises.

The functions named ``wo_*`` mirror the C entry points one for one and take
torch tensors (device memory) where the C call takes device pointers.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "WO_F16", "WO_BF16", "WoError", "load_library", "library_path",
    "wo_status_string", "wo_packed_bytes", "wo_pack", "wo_unpack", "wo_workspace_size",
    "wo_gemm", "wo_moe_workspace_size", "wo_moe_ffn", "wo_check_workspace",
    "wo_gemm_tc_noalloc", "wo_noalloc_check", "wo_noalloc_selftest_wait_timeout",
    "wo_selftest_wait_timeout", "wo_embed",
    "wo_act_order_perm", "wo_pack_act_order", "wo_act_order_workspace_size",
    "wo_gemm_act_order",
    "pack", "unpack", "pack_experts", "gemm", "embed", "moe_ffn", "Workspace",
    "act_order_perm", "pack_act_order", "gemm_act_order", "wo_gemm_plan", "gemm_plan",
]

WO_F16 = 0
WO_BF16 = 1

_STATUS = {0: "WO_OK", 1: "WO_ERR_INVALID_ARG", 2: "WO_ERR_UNSUPPORTED",
           3: "WO_ERR_WORKSPACE", 4: "WO_ERR_CUDA", 5: "WO_ERR_TIMEOUT", 6: "WO_ERR_BOUNDS"}


class WoError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS.get(status, status)}")


_lock = threading.Lock()
_lib = None


def debug_bounds_requested() -> bool:
    """WO_DEBUG_BOUNDS=1 in the environment selects the index-checked build."""
    return os.environ.get("WO_DEBUG_BOUNDS", "") == "1"


def library_path() -> str:
    return _build.LIB_DEBUG_BOUNDS if debug_bounds_requested() else _build.LIB


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libwo.so; raise if it is not built (no fallback path exists)."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"libwo.so is not built ({path}); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            _build.build(debug_bounds=debug_bounds_requested())
        lib = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.wo_status_string.argtypes = [I]
        lib.wo_status_string.restype = ctypes.c_char_p
        lib.wo_packed_bytes.argtypes = [I, I, I]
        lib.wo_packed_bytes.restype = S
        lib.wo_pack.argtypes = [P, P, I, I, I, P]
        lib.wo_pack.restype = I
        lib.wo_unpack.argtypes = [P, P, I, I, I, P]
        lib.wo_unpack.restype = I
        lib.wo_workspace_size.argtypes = [I, I, I, I, I]
        lib.wo_workspace_size.restype = S
        lib.wo_gemm.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, S, P]
        lib.wo_gemm.restype = I
        lib.wo_moe_workspace_size.argtypes = [I, I, I, I, I]
        lib.wo_moe_workspace_size.restype = S
        lib.wo_moe_ffn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, S, P]
        lib.wo_moe_ffn.restype = I
        lib.wo_embed.argtypes = [P, I, P, P, P, P, I, I, I, I, I, P]
        lib.wo_embed.restype = I
        lib.wo_gemm_plan.argtypes = [I, I, I, I, I, I, ctypes.POINTER(GemmPlan)]
        lib.wo_gemm_plan.restype = I
        lib.wo_act_order_perm.argtypes = [P, I, I, P]
        lib.wo_act_order_perm.restype = I
        lib.wo_pack_act_order.argtypes = [P, P, P, I, I, I, P]
        lib.wo_pack_act_order.restype = I
        lib.wo_act_order_workspace_size.argtypes = [I, I, I, I, I]
        lib.wo_act_order_workspace_size.restype = S
        lib.wo_gemm_act_order.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, S, P]
        lib.wo_gemm_act_order.restype = I
        lib.wo_check_workspace.argtypes = [P, S, P]
        lib.wo_check_workspace.restype = I
        lib.wo_gemm_tc_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P]
        lib.wo_gemm_tc_noalloc.restype = I
        lib.wo_selftest_wait_timeout.argtypes = [P, S, ctypes.c_uint, P]
        lib.wo_selftest_wait_timeout.restype = I
        lib.wo_noalloc_check.argtypes = [P]
        lib.wo_noalloc_check.restype = I
        lib.wo_noalloc_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
        lib.wo_noalloc_selftest_wait_timeout.restype = I
        lib.wo_debug_bounds.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.wo_debug_bounds.restype = I
        _lib = lib
        return lib


# ---------------------------------------------------------------- helpers --

class GemmPlan(ctypes.Structure):
    """wo_gemm_plan_t (include/wo.h)."""
    _fields_ = [("kernel", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("k_splits", ctypes.c_int), ("ctas", ctypes.c_int), ("stages", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t)]


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _raise(status: int, what: str):
    if status != 0:
        raise WoError(status, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return WO_F16
    if t.dtype == torch.bfloat16:
        return WO_BF16
    raise TypeError(f"activations must be float16 or bfloat16, got {t.dtype}")


# ------------------------------------------------------ raw C-ABI mirrors --

def wo_status_string(status: int) -> str:
    return load_library().wo_status_string(int(status)).decode()


def wo_packed_bytes(n: int, k: int, bits: int) -> int:
    return int(load_library().wo_packed_bytes(n, k, bits))


def wo_pack(B_rowmajor, B_packed, n: int, k: int, bits: int, stream=None) -> None:
    _raise(load_library().wo_pack(_ptr(B_rowmajor), _ptr(B_packed), n, k, bits,
                                  _stream_ptr(stream)), "wo_pack")


def wo_unpack(B_packed, B_rowmajor, n: int, k: int, bits: int, stream=None) -> None:
    _raise(load_library().wo_unpack(_ptr(B_packed), _ptr(B_rowmajor), n, k, bits,
                                    _stream_ptr(stream)), "wo_unpack")


_ws_sizes: dict = {}


def wo_workspace_size(m: int, n: int, k: int, group_size: int, bits: int) -> int:
    key = (m, n, k, group_size, bits)
    v = _ws_sizes.get(key)
    if v is None:  # a pure function of the shape: computed once per shape
        v = _ws_sizes[key] = int(load_library().wo_workspace_size(m, n, k, group_size, bits))
    return v


def wo_gemm(A, B_packed, scales, zeros, bias, C, m: int, n: int, k: int, group_size: int,
            bits: int, act_dtype: int, workspace, workspace_bytes: int, stream=None) -> None:
    _raise(load_library().wo_gemm(_ptr(A), _ptr(B_packed), _ptr(scales), _ptr(zeros),
                                  _ptr(bias), _ptr(C), m, n, k, group_size, bits, act_dtype,
                                  _ptr(workspace), workspace_bytes, _stream_ptr(stream)),
           "wo_gemm")


def wo_embed(ids, T: int, B_packed, scales, zeros, out, vocab: int, hidden: int, group_size: int,
             bits: int, act_dtype: int, stream=None) -> None:
    _raise(load_library().wo_embed(_ptr(ids), T, _ptr(B_packed), _ptr(scales), _ptr(zeros),
                                   _ptr(out), vocab, hidden, group_size, bits, act_dtype,
                                   _stream_ptr(stream)), "wo_embed")


def wo_gemm_plan(m: int, n: int, k: int, group_size: int, bits: int, act_dtype: int) -> GemmPlan:
    plan = GemmPlan()
    _raise(load_library().wo_gemm_plan(m, n, k, group_size, bits, act_dtype, ctypes.byref(plan)),
           "wo_gemm_plan")
    return plan


def gemm_plan(m: int, n: int, k: int, bits: int, group_size: int = -1,
              act_dtype: int = WO_BF16) -> dict:
    """The configuration wo_gemm runs for this problem, as a dict."""
    p = wo_gemm_plan(m, n, k, group_size, bits, act_dtype)
    kernel = {0: "stream", 1: "tensor_core", 2: "stream_persistent",
              3: "tensor_core_swap_ab"}[int(p.kernel)]
    return {"kernel": kernel, "tile_m": p.tile_m,
            "tile_n": p.tile_n, "k_splits": p.k_splits, "ctas": p.ctas, "stages": p.stages,
            "workspace_bytes": int(p.workspace_bytes)}


def _host_i32(a, k: int, what: str):
    """A host int32 array of k entries (CPU tensor or numpy) and its address."""
    import numpy as np
    if hasattr(a, "device") and hasattr(a, "data_ptr"):
        if a.device.type != "cpu":
            raise ValueError(f"{what} must be in host memory")
        a = a.numpy()
    arr = np.ascontiguousarray(a, dtype=np.int32).reshape(-1)
    if arr.size != k:
        raise ValueError(f"{what} must have k = {k} entries, got {arr.size}")
    return arr, arr.ctypes.data


def wo_act_order_perm(g_idx, k: int, group_size: int, perm) -> None:
    """HOST arrays: g_idx int32 [k] in, perm int32 [k] out (numpy, filled in place)."""
    import numpy as np
    gi, gp = _host_i32(g_idx, k, "g_idx")  # gi keeps the array alive across the call
    if not (isinstance(perm, np.ndarray) and perm.dtype == np.int32 and perm.size == k
            and perm.flags.c_contiguous):
        raise ValueError("perm must be a contiguous numpy int32 array of k entries")
    _raise(load_library().wo_act_order_perm(gp, k, group_size, perm.ctypes.data),
           "wo_act_order_perm")


def wo_pack_act_order(B_rowmajor, B_packed, perm, n: int, k: int, bits: int,
                      stream=None) -> None:
    _raise(load_library().wo_pack_act_order(_ptr(B_rowmajor), _ptr(B_packed), _ptr(perm), n, k,
                                            bits, _stream_ptr(stream)), "wo_pack_act_order")


def wo_act_order_workspace_size(m: int, n: int, k: int, group_size: int, bits: int) -> int:
    return int(load_library().wo_act_order_workspace_size(m, n, k, group_size, bits))


def wo_gemm_act_order(A, B_packed, perm, scales, zeros, bias, C, m: int, n: int, k: int,
                      group_size: int, bits: int, act_dtype: int, workspace, workspace_bytes: int,
                      stream=None) -> None:
    _raise(load_library().wo_gemm_act_order(_ptr(A), _ptr(B_packed), _ptr(perm), _ptr(scales),
                                            _ptr(zeros), _ptr(bias), _ptr(C), m, n, k,
                                            group_size, bits, act_dtype, _ptr(workspace),
                                            workspace_bytes, _stream_ptr(stream)),
           "wo_gemm_act_order")


def wo_moe_workspace_size(T: int, hidden: int, inter: int, experts: int, topk: int) -> int:
    return int(load_library().wo_moe_workspace_size(T, hidden, inter, experts, topk))


def wo_moe_ffn(A, gating_logits, fc1_packed, fc1_scales, fc2_packed, fc2_scales, out, T: int,
               hidden: int, inter: int, experts: int, topk: int, renormalize: int,
               act_dtype: int, workspace, workspace_bytes: int, stream=None) -> None:
    _raise(load_library().wo_moe_ffn(_ptr(A), _ptr(gating_logits), _ptr(fc1_packed),
                                     _ptr(fc1_scales), _ptr(fc2_packed), _ptr(fc2_scales),
                                     _ptr(out), T, hidden, inter, experts, topk,
                                     int(renormalize), act_dtype, _ptr(workspace),
                                     workspace_bytes, _stream_ptr(stream)), "wo_moe_ffn")


def wo_gemm_tc_noalloc(A, B_packed, scales, zeros, bias, C, m: int, n: int, k: int,
                       group_size: int, bits: int, act_dtype: int, stream=None) -> None:
    """The tensor-core GEMM with the library's built-in scratch: for callers
    that cannot allocate device memory.  Calls that overlap on the GPU race
    on the shared scratch."""
    _raise(load_library().wo_gemm_tc_noalloc(_ptr(A), _ptr(B_packed), _ptr(scales), _ptr(zeros),
                                             _ptr(bias), _ptr(C), m, n, k, group_size, bits,
                                             act_dtype, _stream_ptr(stream)),
           "wo_gemm_tc_noalloc")


def wo_noalloc_check(stream=None) -> int:
    """Synchronise and return the status the kernels left in the built-in
    scratch of wo_gemm_tc_noalloc (the word is cleared)."""
    return int(load_library().wo_noalloc_check(_stream_ptr(stream)))


def wo_debug_bounds() -> tuple[int, int]:
    """(status, site) of the index checks since the last call: (WO_OK, 0), or
    WO_ERR_BOUNDS with the first failing check's site; WO_ERR_UNSUPPORTED in
    a library built without them.  Waits for the device; clears the words."""
    site = ctypes.c_uint(0)
    st = int(load_library().wo_debug_bounds(ctypes.byref(site)))
    return st, int(site.value)


def wo_noalloc_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """A wait that runs out after limit_us, reporting into the built-in scratch."""
    _raise(load_library().wo_noalloc_selftest_wait_timeout(limit_us, _stream_ptr(stream)),
           "wo_noalloc_selftest_wait_timeout")


def wo_selftest_wait_timeout(workspace, workspace_bytes: int, limit_us: int, stream=None) -> None:
    """Launch a wait that runs out after limit_us (the kernels' failure path)."""
    _raise(load_library().wo_selftest_wait_timeout(_ptr(workspace), workspace_bytes, limit_us,
                                                   _stream_ptr(stream)), "wo_selftest_wait_timeout")


def wo_check_workspace(workspace, workspace_bytes: int, stream=None) -> int:
    """Synchronise and return the status the kernels left in the workspace."""
    return int(load_library().wo_check_workspace(_ptr(workspace), workspace_bytes,
                                                 _stream_ptr(stream)))


# ------------------------------------------------- torch-level conveniences --

class Workspace:
    """A zero-filled device workspace that grows on demand (allocated by torch)."""

    def __init__(self, device=None):
        import torch
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int):
        import torch
        if nbytes <= 0:
            return None, 0
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf, self.buf.numel()


_default_ws: dict = {}


def _workspace_for(device, nbytes):
    key = str(device)
    ws = _default_ws.get(key)
    if ws is None:
        ws = _default_ws[key] = Workspace(device)
    return ws.get(nbytes)


def _sync(stream):
    import torch
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()


def pack(B_rowmajor, n: int, k: int, bits: int, stream=None):
    """Row-major codes (uint8 [n, k] or [n, k/2]) -> packed uint8 buffer.
    A load-time step: it waits for the packing to finish, so the GEMMs that
    prefetch weights early always see the packed bytes."""
    import torch
    out = torch.empty(wo_packed_bytes(n, k, bits), dtype=torch.uint8, device=B_rowmajor.device)
    wo_pack(B_rowmajor, out, n, k, bits, stream)
    _sync(stream)
    return out


def pack_experts(B_rowmajor, experts: int, n: int, k: int, bits: int, stream=None):
    """Row-major codes of `experts` matrices [experts, n, ...] -> one buffer of
    consecutive wo_pack outputs (the layout wo_moe_ffn reads)."""
    import torch
    per = wo_packed_bytes(n, k, bits)
    out = torch.empty(experts * per, dtype=torch.uint8, device=B_rowmajor.device)
    src = B_rowmajor.reshape(experts, -1)
    for e in range(experts):
        wo_pack(src[e], out.data_ptr() + e * per, n, k, bits, stream)
    _sync(stream)
    return out


def unpack(B_packed, n: int, k: int, bits: int, stream=None):
    import torch
    shape = (n, k) if bits == 8 else (n, k // 2)
    out = torch.empty(shape, dtype=torch.uint8, device=B_packed.device)
    wo_unpack(B_packed, out, n, k, bits, stream)
    return out


def gemm(A, B_packed, scales, n: int, k: int, bits: int, group_size: int = -1, zeros=None,
         bias=None, out=None, workspace=None, stream=None):
    """C = A . dequant(B)^T + bias through wo_gemm; returns C [m, n]."""
    import torch
    m = A.shape[0]
    act = _dtype_code(A)
    if out is None:
        out = torch.empty((m, n), dtype=A.dtype, device=A.device)
    need = wo_workspace_size(m, n, k, group_size, bits)
    if workspace is None:
        ws, ws_bytes = _workspace_for(A.device, need)
    else:
        ws, ws_bytes = workspace, workspace.numel()
    wo_gemm(A, B_packed, scales, zeros, bias, out, m, n, k, group_size, bits, act, ws, ws_bytes,
            stream)
    return out


def act_order_perm(g_idx, k: int, group_size: int):
    """The channel order that sorts a GPTQ act-order group index (host work):
    returns an int32 CPU tensor perm [k], perm[j] = the j-th channel in order
    of (g_idx[c], c).  Copy it to the device for pack_act_order and
    gemm_act_order."""
    import numpy as np
    import torch
    perm = np.empty(k, dtype=np.int32)
    wo_act_order_perm(g_idx, k, group_size, perm)
    return torch.from_numpy(perm)


def _check_perm(perm, k: int, device) -> None:
    """perm must be a contiguous int32 tensor of k entries on `device` (the
    C layer reads it as a device array and cannot check where it lives)."""
    import torch
    if not isinstance(perm, torch.Tensor):
        raise TypeError("perm must be a torch tensor (the output of act_order_perm, "
                        "moved to the device)")
    if perm.dtype != torch.int32 or perm.numel() != k or not perm.is_contiguous():
        raise ValueError(f"perm must be a contiguous int32 tensor of k = {k} entries")
    if perm.device != torch.device(device):
        raise ValueError(f"perm is on {perm.device}, the operands on {device}")


def pack_act_order(B_rowmajor, perm, n: int, k: int, bits: int, stream=None):
    """wo_pack of the codes with input channels in the order perm (a device
    int32 [k] tensor); waits for the packing, as pack() does."""
    import torch
    _check_perm(perm, k, B_rowmajor.device)
    out = torch.empty(wo_packed_bytes(n, k, bits), dtype=torch.uint8, device=B_rowmajor.device)
    wo_pack_act_order(B_rowmajor, out, perm, n, k, bits, stream)
    _sync(stream)
    return out


def gemm_act_order(A, B_packed, perm, scales, n: int, k: int, bits: int, group_size: int,
                   zeros=None, bias=None, out=None, workspace=None, stream=None):
    """The GPTQ act-order GEMM through wo_gemm_act_order: A [m, k] in the
    checkpoint's channel order, B_packed from pack_act_order with the same
    device perm; returns C [m, n]."""
    import torch
    _check_perm(perm, k, A.device)
    m = A.shape[0]
    act = _dtype_code(A)
    if out is None:
        out = torch.empty((m, n), dtype=A.dtype, device=A.device)
    need = wo_act_order_workspace_size(m, n, k, group_size, bits)
    if workspace is None:
        ws, ws_bytes = _workspace_for(A.device, need)
    else:
        ws, ws_bytes = workspace, workspace.numel()
    wo_gemm_act_order(A, B_packed, perm, scales, zeros, bias, out, m, n, k, group_size, bits, act,
                      ws, ws_bytes, stream)
    return out


def embed(ids, B_packed, scales, vocab: int, hidden: int, bits: int, group_size: int = -1,
          zeros=None, out=None, stream=None):
    """Rows ids of a packed [vocab, hidden] table, dequantised to the scales'
    dtype through wo_embed; returns [len(ids), hidden]."""
    import torch
    T = ids.numel()
    act = _dtype_code(scales)
    if out is None:
        out = torch.empty((T, hidden), dtype=scales.dtype, device=scales.device)
    wo_embed(ids, T, B_packed, scales, zeros, out, vocab, hidden, group_size, bits, act, stream)
    return out


def moe_ffn(A, gating_logits, fc1_packed, fc1_scales, fc2_packed, fc2_scales, hidden: int,
            inter: int, experts: int, topk: int, renormalize: bool = False, out=None,
            workspace=None, stream=None):
    import torch
    T = A.shape[0]
    act = _dtype_code(A)
    if out is None:
        out = torch.empty((T, hidden), dtype=A.dtype, device=A.device)
    need = wo_moe_workspace_size(T, hidden, inter, experts, topk)
    if workspace is None:
        ws, ws_bytes = _workspace_for(A.device, need)
    else:
        ws, ws_bytes = workspace, workspace.numel()
    wo_moe_ffn(A, gating_logits, fc1_packed, fc1_scales, fc2_packed, fc2_scales, out, T, hidden,
               inter, experts, topk, int(renormalize), act, ws, ws_bytes, stream)
    return out
