"""Python binding of libfa (include/fa.h): exact IO-aware attention on GB300.

Argument marshalling only: every step of the forward and backward pass runs in
libfa's CUDA kernels.  PyTorch supplies device memory and streams.  There is
no fallback: if libfa.so is missing or the device is not an sm_103 GPU, calls
raise.

Layout [B, N, H, d] bf16 (contiguous); lse [B, Hq, N] fp32.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_DEVICE_TIMEOUT = 4

# fa_bwd_stage bits
FA_BWD_DSUM, FA_BWD_DKDV, FA_BWD_DQ, FA_BWD_PREP, FA_BWD_PREP_DOUT = 1, 2, 4, 8, 16
FA_BWD_ALL = FA_BWD_PREP | FA_BWD_DSUM | FA_BWD_DKDV | FA_BWD_DQ
# backward after fa_fwd_train on the same workspace: q, k, v copies already there
FA_BWD_AFTER_FWD_TRAIN = FA_BWD_PREP_DOUT | FA_BWD_DSUM | FA_BWD_DKDV | FA_BWD_DQ

# every entry point include/fa.h declares
EXPORTS = ("fa_fwd", "fa_fwd_train", "fa_bwd", "fa_bwd_stage", "fa_bwd_noalloc",
           "fa_bwd_workspace_size", "fa_fwd_splitkv", "fa_fwd_splitkv_num_splits",
           "fa_fwd_splitkv_workspace_size", "fa_fwd_blocksparse", "fa_fwd_fp8",
           "fa_fwd_fp8_workspace_size",
           "fa_get_device_error",
           "fa_status_string", "fa_last_cuda_error", "fa_debug_watchdog_probe")

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} {last_cuda_error()}".strip())


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libfa.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"libfa.so not found at {path}; build it with "
                      "`python exact_io_aware_35_gb300/build.py`")
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_train.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.fa_fwd_train.restype = i
    lib.fa_bwd.argtypes = [vp] * 11 + [i, i, i, i, i, i, f, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_stage.argtypes = [i] + [vp] * 11 + [i, i, i, i, i, i, f, vp]
    lib.fa_bwd_stage.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp] * 10 + [i, i, i, i, i, i, f, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_fwd_splitkv.argtypes = [vp] * 6 + [i] * 7 + [f, i, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_splitkv_num_splits.argtypes = [i] * 8
    lib.fa_fwd_splitkv_num_splits.restype = i
    lib.fa_fwd_splitkv_workspace_size.argtypes = [i] * 8
    lib.fa_fwd_splitkv_workspace_size.restype = ctypes.c_size_t
    lib.fa_fwd_blocksparse.argtypes = [vp] * 6 + [i] * 6 + [f, vp]
    lib.fa_fwd_blocksparse.restype = i
    lib.fa_fwd_fp8.argtypes = [vp] * 6 + [i] * 6 + [f, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8_workspace_size.argtypes = [i] * 5
    lib.fa_fwd_fp8_workspace_size.restype = ctypes.c_size_t

    lib.fa_get_device_error.argtypes = [vp]
    lib.fa_get_device_error.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_cuda_error.argtypes = []
    lib.fa_last_cuda_error.restype = ctypes.c_char_p
    lib.fa_debug_watchdog_probe.argtypes = [ctypes.c_uint64, i, vp]
    lib.fa_debug_watchdog_probe.restype = i
    _lib = lib
    return lib


def status_string(s: int) -> str:
    return load_library().fa_status_string(int(s)).decode()


def last_cuda_error() -> str:
    return load_library().fa_last_cuda_error().decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t: torch.Tensor, name: str, shape, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _on_device(device, **tensors):
    """Every given tensor must sit on `device` (q's): the kernels take raw
    pointers, and a tensor on another GPU would be read through the wrong
    device's address space."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, q on {device}")


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k must be [B, N, H, d]")
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    return B, N, Hq, Hkv, d


def fa_fwd(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
           stream=None, o_lo=None, workspace=None):
    """Forward pass.  Returns (o, lse); o, lse are allocated if not given.
    With o_lo (a bf16 tensor shaped like q) this is the training forward
    (fa_fwd_train): o_lo receives the low bf16 half of O for fa_bwd, and P
    enters P V in fp16.  `workspace` is the training workspace
    (fa_bwd_workspace_size bytes, allocated if not given); it keeps the fp16
    copies of q, k, v for a backward that uses stages=FA_BWD_AFTER_FWD_TRAIN."""
    lib = load_library()
    B, N, Hq, Hkv, d = _dims(q, k)
    _check(q, "q", (B, N, Hq, d))
    _check(k, "k", (B, N, Hkv, d))
    _check(v, "v", (B, N, Hkv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), device=q.device, dtype=torch.float32)
    _check(o, "o", (B, N, Hq, d))
    _check(lse, "lse", (B, Hq, N), torch.float32)
    if o_lo is None:
        _on_device(q.device, k=k, v=v, o=o, lse=lse)
        with torch.cuda.device(q.device):
            st = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                            _stream_handle(stream))
    else:
        _check(o_lo, "o_lo", (B, N, Hq, d))
        ws_bytes = fa_bwd_workspace_size(B, Hq, Hkv, N, d)
        if workspace is None:
            workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
        if workspace.numel() * workspace.element_size() < ws_bytes:
            raise ValueError("workspace too small")
        _on_device(q.device, k=k, v=v, o=o, lse=lse, o_lo=o_lo, workspace=workspace)
        with torch.cuda.device(q.device):
            st = lib.fa_fwd_train(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  o_lo.data_ptr(), lse.data_ptr(), workspace.data_ptr(), B, Hq,
                                  Hkv, N, d, int(bool(causal)), float(scale),
                                  _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd")
    return o, lse


def fa_bwd_workspace_size(B: int, H: int, Hkv: int, N: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, Hkv, N, d))


def fa_bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
           dq=None, dk=None, dv=None, workspace=None, stream=None,
           stages: int = FA_BWD_ALL, o_lo=None):
    """Backward pass.  Returns (dq, dk, dv); buffers are allocated if not given.
    `stages` selects a subset of the steps (fa_bwd_stage); o_lo is the
    training forward's low half of O (None: D from o alone)."""
    lib = load_library()
    B, N, Hq, Hkv, d = _dims(q, k)
    _check(q, "q", (B, N, Hq, d))
    _check(k, "k", (B, N, Hkv, d))
    _check(v, "v", (B, N, Hkv, d))
    _check(o, "o", (B, N, Hq, d))
    _check(dout, "dout", (B, N, Hq, d))
    _check(lse, "lse", (B, Hq, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(dq, "dq", (B, N, Hq, d))
    _check(dk, "dk", (B, N, Hkv, d))
    _check(dv, "dv", (B, N, Hkv, d))
    ws_bytes = fa_bwd_workspace_size(B, Hq, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    if workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError("workspace too small")
    if o_lo is not None:
        _check(o_lo, "o_lo", (B, N, Hq, d))
    _on_device(q.device, k=k, v=v, o=o, dout=dout, lse=lse, dq=dq, dk=dk, dv=dv,
               workspace=workspace, o_lo=o_lo)
    with torch.cuda.device(q.device):
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                None if o_lo is None else o_lo.data_ptr(),
                B, Hq, Hkv, N, d, int(bool(causal)), float(scale), _stream_handle(stream))
        st = lib.fa_bwd(*args) if stages == FA_BWD_ALL else lib.fa_bwd_stage(int(stages), *args)
    if st != FA_OK:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv


def fa_fwd_splitkv_num_splits(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int,
                              causal: bool = False, num_splits: int = 0) -> int:
    return int(load_library().fa_fwd_splitkv_num_splits(B, H, Hkv, Nq, Nk, d, int(bool(causal)),
                                                        int(num_splits)))


def fa_fwd_splitkv_workspace_size(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int,
                                  causal: bool = False, num_splits: int = 0) -> int:
    return int(load_library().fa_fwd_splitkv_workspace_size(B, H, Hkv, Nq, Nk, d,
                                                            int(bool(causal)), int(num_splits)))


def fa_fwd_splitkv(q, k, v, causal: bool = False, scale: float | None = None,
                   num_splits: int = 0, o=None, lse=None, workspace=None, stream=None):
    """Split-KV forward (fa_fwd_splitkv): q [B, Nq, H, d] against k, v
    [B, Nk, Hkv, d]; causal means the queries are the sequence's last Nq
    positions.  num_splits <= 0 lets the library choose.  Returns (o, lse)."""
    lib = load_library()
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k must be [B, N, H, d]")
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    _check(q, "q", (B, Nq, Hq, d))
    _check(k, "k", (B, Nk, Hkv, d))
    _check(v, "v", (B, Nk, Hkv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    _check(o, "o", (B, Nq, Hq, d))
    _check(lse, "lse", (B, Hq, Nq), torch.float32)
    ws_bytes = fa_fwd_splitkv_workspace_size(B, Hq, Hkv, Nq, Nk, d, causal, num_splits)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    if ws_bytes and workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError("workspace too small")
    _on_device(q.device, k=k, v=v, o=o, lse=lse, workspace=workspace)
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), None if workspace is None else workspace.data_ptr(),
                                B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
                                int(num_splits), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_splitkv")
    return o, lse


def fa_fwd_blocksparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None,
                       o=None, lse=None, stream=None):
    """Block-sparse forward (fa_fwd_blocksparse): block_mask is a CUDA uint8
    (or bool) tensor [H, nb, nb], nb = ceil(N / 128), nonzero = the block is
    computed.  Returns (o, lse); rows with no visible key get o = 0 and
    lse = -inf."""
    lib = load_library()
    B, N, Hq, Hkv, d = _dims(q, k)
    _check(q, "q", (B, N, Hq, d))
    _check(k, "k", (B, N, Hkv, d))
    _check(v, "v", (B, N, Hkv, d))
    nb = (N + 127) // 128
    if block_mask.dtype == torch.bool:
        block_mask = block_mask.to(torch.uint8)
    _check(block_mask, "block_mask", (Hq, nb, nb), torch.uint8)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), device=q.device, dtype=torch.float32)
    _check(o, "o", (B, N, Hq, d))
    _check(lse, "lse", (B, Hq, N), torch.float32)
    _on_device(q.device, k=k, v=v, o=o, lse=lse, block_mask=block_mask)
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_blocksparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), block_mask.data_ptr(), B, Hq, Hkv, N, d,
                                    int(bool(causal)), float(scale), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_blocksparse")
    return o, lse


FA_FP8_ROTATE, FA_FP8_QUANTIZE_ONLY, FA_FP8_ATTEND_ONLY = 1, 2, 4


def fa_fwd_fp8_workspace_size(B: int, H: int, Hkv: int, N: int, d: int) -> int:
    return int(load_library().fa_fwd_fp8_workspace_size(B, H, Hkv, N, d))


def fa_fwd_fp8(q, k, v, causal: bool = False, scale: float | None = None, rotate: bool = True,
               o=None, lse=None, workspace=None, stream=None, stage: int = 0):
    """FP8 (e4m3) forward (fa_fwd_fp8), d = 128: bf16 q, k, v in, bf16 o and
    fp32 lse out; rotate = incoherent processing of q and k; stage 0 = both
    steps, FA_FP8_QUANTIZE_ONLY or FA_FP8_ATTEND_ONLY = one.  Returns (o, lse)."""
    lib = load_library()
    B, N, Hq, Hkv, d = _dims(q, k)
    _check(q, "q", (B, N, Hq, d))
    _check(k, "k", (B, N, Hkv, d))
    _check(v, "v", (B, N, Hkv, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), device=q.device, dtype=torch.float32)
    _check(o, "o", (B, N, Hq, d))
    _check(lse, "lse", (B, Hq, N), torch.float32)
    ws_bytes = fa_fwd_fp8_workspace_size(B, Hq, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), device=q.device, dtype=torch.uint8)
    if workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError("workspace too small")
    _on_device(q.device, k=k, v=v, o=o, lse=lse, workspace=workspace)
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), workspace.data_ptr(), B, Hq, Hkv, N, d,
                            int(bool(causal)), float(scale),
                            (FA_FP8_ROTATE if rotate else 0) | int(stage), _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return o, lse


def fa_get_device_error(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device status."""
    return int(load_library().fa_get_device_error(_stream_handle(stream)))


def fa_debug_watchdog_probe(timeout_ns: int, num_blocks: int = 1, stream=None) -> None:
    """Launches num_blocks blocks whose waits nothing satisfies (limit
    timeout_ns); read the outcome with fa_get_device_error."""
    st = load_library().fa_debug_watchdog_probe(int(timeout_ns), int(num_blocks),
                                                _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_debug_watchdog_probe")
