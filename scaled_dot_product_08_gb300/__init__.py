"""Python binding of the GB300 exact-attention library (argument marshalling only).

The functions ``attn_fwd``, ``attn_bwd``, ``attn_bwd_workspace_size``,
``attn_get_device_status``, ``attn_status_string`` and
``attn_selftest_wait_timeout`` call the C ABI of ``include/attn.h`` with raw
device pointers.  ``forward`` and ``backward`` are conveniences that take
torch CUDA tensors, allocate the outputs (and the backward workspace) with
torch and call the same C ABI; they compute nothing themselves.

There is no fallback: if the compiled library is missing, or the device is
not a GB300, every call raises.
"""
from __future__ import annotations

import ctypes
import enum
import math
import os

from .build import LIB, build  # noqa: F401  (build() is the supported way to compile)

__all__ = [
    "AttnError", "Status", "load", "attn_fwd", "attn_bwd", "attn_bwd_workspace_size",
    "attn_bwd_prep", "attn_bwd_grad", "attn_bwd_dq", "attn_bwd_dq_rows", "attn_bwd_noalloc",
    "attn_get_device_status", "attn_get_timeout_info", "attn_status_string", "attn_selftest_wait_timeout",
    "attn_debug_drop_load", "attn_debug_build", "attn_debug_plant_index",
    "attn_decode", "attn_decode_workspace_size", "attn_fwd_cross", "attn_bwd_cross",
    "attn_bwd_grad_cross", "attn_bwd_dq_cross", "attn_fwd_varlen", "attn_bwd_varlen",
    "attn_bwd_varlen_workspace_size", "attn_bwd_varlen_stages", "forward_varlen", "backward_varlen",
    "AttnMask", "attn_masked_workspace_size", "attn_fwd_masked", "attn_bwd_masked", "attn_bwd_masked_stages",
    "forward_masked", "backward_masked", "attn_fwd_fp8", "forward_fp8",
    "attn_decode_paged", "attn_decode_paged_workspace_size", "decode_paged",
    "forward", "forward_cross", "backward", "backward_cross", "decode", "build",
]


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED_SHAPE = 2
    UNSUPPORTED_DEVICE = 3
    MISALIGNED = 4
    WORKSPACE = 5
    LAUNCH = 6
    TIMEOUT = 7
    CUDA = 8
    CHECK = 9


class AttnMask(ctypes.Structure):
    """attn_mask_t of include/attn.h (device pointers as integers, 0 = none)."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("key_lengths", ctypes.c_void_p), ("mask", ctypes.c_void_p),
                ("mask_batch", ctypes.c_int), ("mask_heads", ctypes.c_int),
                ("bias", ctypes.c_void_p), ("bias_batch", ctypes.c_int), ("bias_heads", ctypes.c_int),
                ("bias_bf16", ctypes.c_int)]


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{where}: {attn_status_string(status)}")


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def library_path() -> str:
    """The library this process loads: the in-tree release build, or the file
    that the environment variable SDPA08_LIBRARY names (e.g. the debug build,
    _lib/libsdpa08_debug.so from build(debug=True))."""
    return os.environ.get("SDPA08_LIBRARY") or LIB


def load() -> ctypes.CDLL:
    """Load the in-tree shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built ({path} missing): run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.attn_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_fwd.restype = _I
        lib.attn_bwd_workspace_size.argtypes = [_I, _I, _I, _I, _I]
        lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                 _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd.restype = _I
        lib.attn_bwd_prep.argtypes = [_P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, _P]
        lib.attn_bwd_prep.restype = _I
        lib.attn_bwd_grad.argtypes = [_P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                      _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_grad.restype = _I
        lib.attn_bwd_dq.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_dq.restype = _I
        lib.attn_debug_drop_load.argtypes = [_I, _I, ctypes.c_uint]
        lib.attn_debug_drop_load.restype = _I
        lib.attn_debug_build.argtypes = []
        lib.attn_debug_build.restype = _I
        lib.attn_debug_plant_index.argtypes = [_I]
        lib.attn_debug_plant_index.restype = _I
        lib.attn_get_device_status.argtypes = [_P]
        lib.attn_get_device_status.restype = _I
        lib.attn_status_string.argtypes = [_I]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_fwd_cross.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_fwd_cross.restype = _I
        lib.attn_bwd_cross.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                       _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_cross.restype = _I
        lib.attn_bwd_grad_cross.argtypes = [_P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                            _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_grad_cross.restype = _I
        lib.attn_bwd_dq_cross.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                          _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_dq_cross.restype = _I
        lib.attn_bwd_dq_rows.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                         _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_dq_rows.restype = _I
        lib.attn_fwd_varlen.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                        ctypes.c_float, _I, _P]
        lib.attn_fwd_varlen.restype = _I
        lib.attn_bwd_varlen_workspace_size.argtypes = [_I, _I, _I, _I, _I]
        lib.attn_bwd_varlen_workspace_size.restype = ctypes.c_size_t
        lib.attn_bwd_varlen.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                        _I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_varlen.restype = _I
        lib.attn_bwd_varlen_stages.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                               _I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, ctypes.c_uint,
                                               _P]
        lib.attn_bwd_varlen_stages.restype = _I
        lib.attn_decode_paged_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I, _I]
        lib.attn_decode_paged_workspace_size.restype = ctypes.c_size_t
        lib.attn_decode_paged.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, _I, _I,
                                          _I, ctypes.c_float, _I, _P]
        lib.attn_decode_paged.restype = _I
        _F = ctypes.c_float
        lib.attn_fwd_fp8.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _F, _I, _P]
        lib.attn_fwd_fp8.restype = _I
        _M = ctypes.POINTER(AttnMask)
        lib.attn_masked_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I, _M, _I]
        lib.attn_masked_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_masked.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _M, _P,
                                        ctypes.c_size_t, _P]
        lib.attn_fwd_masked.restype = _I
        lib.attn_bwd_masked.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I,
                                        _M, _P, ctypes.c_size_t, _P]
        lib.attn_bwd_masked.restype = _I
        lib.attn_bwd_masked_stages.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                               ctypes.c_float, _I, _M, _P, ctypes.c_size_t, ctypes.c_uint, _P]
        lib.attn_bwd_masked_stages.restype = _I
        lib.attn_decode_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I]
        lib.attn_decode_workspace_size.restype = ctypes.c_size_t
        lib.attn_decode.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, _I,
                                    ctypes.c_float, _I, _P]
        lib.attn_decode.restype = _I
        lib.attn_abi_version.argtypes = []
        lib.attn_abi_version.restype = _I
        lib.attn_bwd_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P,
                                         _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]
        lib.attn_bwd_noalloc.restype = _I
        lib.attn_get_timeout_info.argtypes = [ctypes.POINTER(ctypes.c_int), _P]
        lib.attn_get_timeout_info.restype = _I
        lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, _P]
        lib.attn_selftest_wait_timeout.restype = _I
        _lib = lib
    return _lib


# ------------------------------------------------------------------ raw C ABI
def attn_status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def attn_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, stream) -> int:
    return load().attn_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, int(causal), stream)


def attn_bwd_workspace_size(B, H, Hkv, N, d) -> int:
    return load().attn_bwd_workspace_size(B, H, Hkv, N, d)


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes,
             B, H, Hkv, N, d, scale, causal, stream) -> int:
    return load().attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes,
                           B, H, Hkv, N, d, scale, int(causal), stream)


def attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, scale, causal, stream) -> int:
    """attn_bwd without a caller workspace (fixed 64 MiB scratch inside the library)."""
    return load().attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, scale, int(causal), stream)


def attn_bwd_prep(o, lse, dout, workspace, workspace_bytes, B, H, Hkv, N, d, stream) -> int:
    return load().attn_bwd_prep(o, lse, dout, workspace, workspace_bytes, B, H, Hkv, N, d, stream)


def attn_bwd_grad(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal,
                  stream) -> int:
    return load().attn_bwd_grad(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d,
                                scale, int(causal), stream)


def attn_bwd_dq(q, k, v, dout, dq, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal, stream) -> int:
    return load().attn_bwd_dq(q, k, v, dout, dq, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal, stream)


def attn_bwd_dq_rows(q, k, v, o, lse, dout, dq, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal,
                     stream) -> int:
    return load().attn_bwd_dq_rows(q, k, v, o, lse, dout, dq, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d,
                                   scale, int(causal), stream)


def attn_fwd_cross(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, stream) -> int:
    return load().attn_fwd_cross(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, stream)


def attn_bwd_cross(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes,
                   B, H, Hkv, Nq, Nk, d, scale, causal, stream) -> int:
    return load().attn_bwd_cross(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes,
                                 B, H, Hkv, Nq, Nk, d, scale, causal, stream)


def attn_bwd_grad_cross(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale,
                        causal, stream) -> int:
    return load().attn_bwd_grad_cross(q, k, v, dout, dk, dv, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d,
                                      scale, causal, stream)


def attn_bwd_dq_cross(q, k, v, dout, dq, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal,
                      stream) -> int:
    return load().attn_bwd_dq_cross(q, k, v, dout, dq, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d,
                                    scale, causal, stream)


def attn_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, B, H, Hkv, total_q, total_k, max_q, max_k, d, scale, causal,
                    stream) -> int:
    return load().attn_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, B, H, Hkv, total_q, total_k, max_q, max_k, d,
                                  scale, causal, stream)


def attn_bwd_varlen_workspace_size(B, H, Hkv, total_q, d) -> int:
    return load().attn_bwd_varlen_workspace_size(B, H, Hkv, total_q, d)


def attn_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, workspace, workspace_bytes, B, H, Hkv,
                    total_q, total_k, max_q, max_k, d, scale, causal, stream) -> int:
    return load().attn_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, workspace, workspace_bytes,
                                  B, H, Hkv, total_q, total_k, max_q, max_k, d, scale, causal, stream)


def attn_bwd_varlen_stages(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, workspace, workspace_bytes, B, H, Hkv,
                           total_q, total_k, max_q, max_k, d, scale, causal, stages, stream) -> int:
    return load().attn_bwd_varlen_stages(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, workspace, workspace_bytes,
                                         B, H, Hkv, total_q, total_k, max_q, max_k, d, scale, causal, stages,
                                         stream)


def attn_fwd_fp8(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, q_scale, k_scale, v_scale, causal, stream) -> int:
    return load().attn_fwd_fp8(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, q_scale, k_scale, v_scale, causal,
                               stream)


def attn_decode_paged_workspace_size(B, H, Hkv, Nq, page_size, max_pages, d) -> int:
    return load().attn_decode_paged_workspace_size(B, H, Hkv, Nq, page_size, max_pages, d)


def attn_decode_paged(q, k_cache, v_cache, o, lse, block_table, seq_lens, workspace, workspace_bytes, B, H, Hkv, Nq,
                      page_size, num_pages, max_pages, d, scale, causal, stream) -> int:
    return load().attn_decode_paged(q, k_cache, v_cache, o, lse, block_table, seq_lens, workspace, workspace_bytes,
                                    B, H, Hkv, Nq, page_size, num_pages, max_pages, d, scale, causal, stream)


def attn_masked_workspace_size(B, H, Hkv, Nq, Nk, d, mask: AttnMask, backward) -> int:
    return load().attn_masked_workspace_size(B, H, Hkv, Nq, Nk, d, ctypes.byref(mask), int(backward))


def attn_fwd_masked(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, mask: AttnMask, workspace,
                    workspace_bytes, stream) -> int:
    return load().attn_fwd_masked(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, ctypes.byref(mask),
                                  workspace, workspace_bytes, stream)


def attn_bwd_masked(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, scale, causal, mask: AttnMask,
                    workspace, workspace_bytes, stream) -> int:
    return load().attn_bwd_masked(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, scale, causal,
                                  ctypes.byref(mask), workspace, workspace_bytes, stream)


def attn_bwd_masked_stages(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, scale, causal, mask: AttnMask,
                           workspace, workspace_bytes, stages, stream) -> int:
    return load().attn_bwd_masked_stages(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, scale, causal,
                                         ctypes.byref(mask), workspace, workspace_bytes, stages, stream)


def attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d) -> int:
    return load().attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d)


def attn_decode(q, k, v, o, lse, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal, stream) -> int:
    return load().attn_decode(q, k, v, o, lse, workspace, workspace_bytes, B, H, Hkv, Nq, Nk, d, scale, causal,
                              stream)


def attn_get_device_status(stream=None) -> int:
    return load().attn_get_device_status(stream)


def attn_get_timeout_info(stream=None):
    """(status, [site<<16|step, block, thread, waited_us]) of the first timed-out wait."""
    buf = (ctypes.c_int * 4)()
    st = load().attn_get_timeout_info(buf, stream)
    return st, list(buf)


def attn_selftest_wait_timeout(timeout_us: int, stream=None) -> int:
    return load().attn_selftest_wait_timeout(timeout_us, stream)


def attn_debug_drop_load(kernel: int, load_index: int, limit_us: int) -> int:
    return load().attn_debug_drop_load(kernel, load_index, limit_us)


def attn_debug_build() -> int:
    """1 if the loaded library is the debug build (in-kernel index checks)."""
    return load().attn_debug_build()


def attn_debug_plant_index(kernel: int) -> int:
    return load().attn_debug_plant_index(kernel)


# ------------------------------------------------------------ torch marshalling
def _check(status: int, where: str):
    if status != 0:
        raise AttnError(status, where)


def _shape(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be (B, H, N, d)")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, N, d) or tuple(v.shape) != (B, Hkv, N, d):
        raise ValueError("k and v must be (B, Hkv, N, d) with q's B, N, d")
    return B, H, Hkv, N, d


def _stream_ptr(t):
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def forward(q, k, v, scale: float | None = None, causal: bool = False, out=None, lse=None):
    """O, lse = attention(q, k, v) on the current CUDA stream.

    q: bf16 (B, H, N, d); k, v: bf16 (B, Hkv, N, d); all contiguous on one
    CUDA device.  Returns O bf16 (B, H, N, d) and lse float32 (B, H, N)."""
    import torch
    B, H, Hkv, N, d = _shape(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t in (q, k, v):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    B, H, Hkv, N, d, scale, causal, _stream_ptr(q)), "attn_fwd")
    return out, lse


def backward(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False,
             workspace=None):
    """dQ, dK, dV of attention given the forward's O and lse and dL/dO."""
    import torch
    B, H, Hkv, N, d = _shape(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws_bytes = attn_bwd_workspace_size(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check(attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                    workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                    B, H, Hkv, N, d, scale, causal, _stream_ptr(q)), "attn_bwd")
    return dq, dk, dv


def decode(q, k, v, scale: float | None = None, causal: bool = False, workspace=None):
    """O, lse of Nq new queries against a cache of Nk keys/values.

    q: bf16 (B, H, Nq, d); k, v: bf16 (B, Hkv, Nk, d), Nk >= Nq; contiguous
    on one CUDA device.  causal: query t sits at position Nk - Nq + t."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != (B, Hkv, Nk, d):
        raise ValueError("k and v must be (B, Hkv, Nk, d) with q's B and d")
    for t in (q, k, v):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws_bytes = attn_decode_workspace_size(B, H, Hkv, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                       B, H, Hkv, Nq, Nk, d, scale, causal, _stream_ptr(q)), "attn_decode")
    return o, lse


def forward_cross(q, k, v, scale: float | None = None, causal: bool = False):
    """O, lse of Nq queries against Nk keys/values per head.

    q: bf16 (B, H, Nq, d); k, v: bf16 (B, Hkv, Nk, d); causal: query row i
    sits at position Nk - Nq + i (needs Nq <= Nk)."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != (B, Hkv, Nk, d):
        raise ValueError("k and v must be (B, Hkv, Nk, d) with q's B and d")
    for t in (q, k, v):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check(attn_fwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, Hkv, Nq, Nk, d, scale, causal, _stream_ptr(q)), "attn_fwd_cross")
    return o, lse


def backward_cross(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False,
                   workspace=None):
    """dQ, dK, dV of forward_cross given its O and lse and dL/dO.

    q, o, dout: bf16 (B, H, Nq, d); k, v: bf16 (B, Hkv, Nk, d); lse float32
    (B, H, Nq); causal alignment as in forward_cross."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != (B, Hkv, Nk, d):
        raise ValueError("k and v must be (B, Hkv, Nk, d) with q's B and d")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must have q's shape")
    for t in (q, k, v, o, dout):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws_bytes = attn_bwd_workspace_size(B, H, Hkv, Nq, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(attn_bwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          B, H, Hkv, Nq, Nk, d, scale, causal, _stream_ptr(q)), "attn_bwd_cross")
    return dq, dk, dv


def _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k):
    import torch
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("packed q, k, v must be (total, heads, d)")
    total_q, H, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    if tuple(v.shape) != tuple(k.shape) or k.shape[2] != d:
        raise ValueError("k and v must be (total_k, Hkv, d) with q's d")
    for t in (q, k, v):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16")
    for c in (cu_seqlens_q, cu_seqlens_k):
        if c.dtype != torch.int32 or c.dim() != 1 or not c.is_cuda or not c.is_contiguous():
            raise ValueError("cu_seqlens must be contiguous int32 CUDA vectors")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 offsets")
    B = cu_seqlens_q.numel() - 1
    return B, H, Hkv, total_q, total_k, d, int(max_seqlen_q), int(max_seqlen_k)


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale: float | None = None,
                   causal: bool = False):
    """O, lse of a packed variable-length batch.

    q: bf16 (total_q, H, d); k, v: bf16 (total_k, Hkv, d); cu_seqlens_*:
    int32 CUDA vectors of B + 1 offsets.  Returns O (total_q, H, d) and lse
    float32 (H, total_q)."""
    import torch
    B, H, Hkv, total_q, total_k, d, mq, mk = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                                           max_seqlen_k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    _check(attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, H, Hkv, total_q, total_k, mq, mk, d,
                           scale, causal, _stream_ptr(q)), "attn_fwd_varlen")
    return o, lse


def backward_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    scale: float | None = None, causal: bool = False, workspace=None):
    """dQ, dK, dV of forward_varlen (packed layouts as its inputs)."""
    import torch
    B, H, Hkv, total_q, total_k, d, mq, mk = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                                           max_seqlen_k)
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("o and dout must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = attn_bwd_varlen_workspace_size(B, H, Hkv, total_q, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    _check(attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens_q.data_ptr(),
                           cu_seqlens_k.data_ptr(), workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), B, H, Hkv, total_q, total_k, mq, mk, d,
                           scale, causal, _stream_ptr(q)), "attn_bwd_varlen")
    return dq, dk, dv


def make_mask(window=None, key_lengths=None, mask=None, B=1, H=1, bias=None) -> AttnMask:
    """AttnMask from Python values: window (left, right) with -1 for an open
    side, key_lengths an int32 CUDA vector (B,), mask a bool / uint8 CUDA
    tensor (1 or B, 1 or H, Nq, Nk), bias a float32 or bfloat16 CUDA tensor of the same
    broadcasting shape added to the scaled scores (finite or -inf).  The
    tensors must stay alive while the calls that use the AttnMask run."""
    import torch
    wl, wr = window if window is not None else (-1, -1)
    m = AttnMask(int(wl), int(wr), 0, 0, 1, 1, 0, 1, 1, 0)
    if key_lengths is not None:
        if key_lengths.dtype != torch.int32 or not key_lengths.is_cuda or not key_lengths.is_contiguous():
            raise ValueError("key_lengths must be a contiguous int32 CUDA vector")
        m.key_lengths = key_lengths.data_ptr()
    if mask is not None:
        if mask.dim() != 4 or mask.dtype not in (torch.bool, torch.uint8) or not mask.is_cuda:
            raise ValueError("mask must be a 4-D bool / uint8 CUDA tensor")
        if not mask.is_contiguous():
            raise ValueError("mask must be contiguous")
        m.mask = mask.data_ptr()
        m.mask_batch, m.mask_heads = int(mask.shape[0]), int(mask.shape[1])
    if bias is not None:
        if (bias.dim() != 4 or bias.dtype not in (torch.float32, torch.bfloat16) or not bias.is_cuda
                or not bias.is_contiguous()):
            raise ValueError("bias must be a contiguous 4-D float32 or bfloat16 CUDA tensor")
        m.bias = bias.data_ptr()
        m.bias_bf16 = int(bias.dtype == torch.bfloat16)
        m.bias_batch, m.bias_heads = int(bias.shape[0]), int(bias.shape[1])
    return m


def _masked_shapes(q, k, v):
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != (B, Hkv, Nk, d):
        raise ValueError("k and v must be (B, Hkv, Nk, d) with q's B and d")
    for t in (q, k, v):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16")
    return B, H, Hkv, Nq, Nk, d


def forward_masked(q, k, v, scale: float | None = None, causal: bool = False, window=None, key_lengths=None,
                   mask=None, bias=None):
    """O, lse under a sliding window / key lengths / boolean mask / additive
    float32 mask (see include/attn.h, attn_mask_t); q (B, H, Nq, d), k, v
    (B, Hkv, Nk, d)."""
    import torch
    B, H, Hkv, Nq, Nk, d = _masked_shapes(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    m = make_mask(window, key_lengths, mask, B, H, bias)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    wsb = attn_masked_workspace_size(B, H, Hkv, Nq, Nk, d, m, 0)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=q.device)
    _check(attn_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, Nq, Nk,
                           d, scale, causal, m, ws.data_ptr(), ws.numel(), _stream_ptr(q)), "attn_fwd_masked")
    return o, lse


def backward_masked(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False, window=None,
                    key_lengths=None, mask=None, bias=None):
    """dQ, dK, dV of forward_masked with the same masks."""
    import torch
    B, H, Hkv, Nq, Nk, d = _masked_shapes(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    m = make_mask(window, key_lengths, mask, B, H, bias)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = attn_masked_workspace_size(B, H, Hkv, Nq, Nk, d, m, 1)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=q.device)
    _check(attn_bwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, Nq, Nk, d, scale, causal, m,
                           ws.data_ptr(), ws.numel(), _stream_ptr(q)), "attn_bwd_masked")
    return dq, dk, dv


def forward_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float, scale: float | None = None,
                causal: bool = False):
    """O (bf16), lse of attention on e4m3 inputs: q8 (B, H, Nq, d), k8, v8
    (B, Hkv, Nk, d) uint8 CUDA tensors holding e4m3 bytes (d in {64, 96,
    128}), each with its dequantisation factor."""
    import torch
    for t in (q8, k8, v8):
        if t.dim() != 4 or t.dtype != torch.uint8 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q8, k8, v8 must be contiguous 4-D uint8 CUDA tensors of e4m3 bytes")
    B, H, Nq, d = q8.shape
    Hkv, Nk = k8.shape[1], k8.shape[2]
    if tuple(k8.shape) != (B, Hkv, Nk, d) or tuple(v8.shape) != (B, Hkv, Nk, d):
        raise ValueError("k8 and v8 must be (B, Hkv, Nk, d) with q8's B and d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device)
    _check(attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, Nq, Nk,
                        d, scale, q_scale, k_scale, v_scale, causal, _stream_ptr(q8)), "attn_fwd_fp8")
    return o, lse


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale: float | None = None, causal: bool = False,
                 workspace=None):
    """O, lse of Nq new queries per head against a paged KV cache.

    q: bf16 (B, H, Nq, d); k_cache, v_cache: bf16 (num_pages, page_size,
    Hkv, d); block_table: int32 CUDA (B, max_pages); seq_lens: int32 CUDA
    (B,)."""
    import torch
    if q.dim() != 4 or k_cache.dim() != 4 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q must be (B, H, Nq, d), k_cache and v_cache (num_pages, page_size, Hkv, d)")
    B, H, Nq, d = q.shape
    num_pages, page_size, Hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape[3] != d:
        raise ValueError("the cache's head_dim must be q's")
    for t in (q, k_cache, v_cache):
        if not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("q and the caches must be contiguous bf16")
    for t in (block_table, seq_lens):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("block_table and seq_lens must be contiguous int32 CUDA tensors")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_table must be (B, max_pages) and seq_lens (B,)")
    max_pages = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    wsb = attn_decode_paged_workspace_size(B, H, Hkv, Nq, page_size, max_pages, d)
    if workspace is None:
        workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=q.device)
    _check(attn_decode_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             block_table.data_ptr(), seq_lens.data_ptr(), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), B, H, Hkv, Nq, page_size, num_pages,
                             max_pages, d, scale, causal, _stream_ptr(q)), "attn_decode_paged")
    return o, lse
