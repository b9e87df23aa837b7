"""ctypes binding of libfa.so: argument marshalling only.

Every step of the attention computation runs in the CUDA kernels behind the
C-ABI (include/fa.h). This module turns torch tensors into device pointers
and streams, allocates outputs with torch, and raises on a non-zero status.
There is no CPU path: a missing library or a non-CUDA tensor is an error.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")
_lib = None

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_CHECK = range(6)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_U64 = ctypes.c_uint64
_U32 = ctypes.c_uint32

SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_fwd_kpad": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P]),
    "fa_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "fa_bwd_split_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "fa_fwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "fa_fwd_split": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, ctypes.c_size_t, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P,
                    ctypes.c_size_t, _P]),
    "fa_bwd_preprocess": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "fa_bwd_main": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, ctypes.c_size_t,
                         _P]),
    "fa_bwd_dq_convert": (_I, [_P, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "fa_blocksparse_bwd": (_I, [_P] * 9 + [_I, _I, _I, _I, _F, _P, _I, _P, ctypes.c_size_t, _P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P]),
    "fa_blocksparse_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _I, _P]),
    "fa_dropout_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _F, _U64, _U32, _P]),
    "fa_dropout_bwd": (_I, [_P] * 9 + [_I, _I, _I, _I, _I, _F, _P, _F, _U64, _U32, _P,
                                       ctypes.c_size_t, _P]),
    "fa_dropout_mask": (_I, [_I, _I, _I, _F, _U64, _U32, _P, _P]),
    "fa_device_status": (_I, []),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_selftest_wait_timeout": (_I, [ctypes.c_longlong, _P]),
}


class AttentionOptions(ctypes.Structure):
    """fa_attention_options of include/fa.h."""
    _fields_ = [("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
                ("stride_n", ctypes.c_int64), ("causal", ctypes.c_int), ("scale", ctypes.c_float),
                ("kv_len", ctypes.c_void_p), ("block_mask", ctypes.c_void_p),
                ("block_size", ctypes.c_int), ("dropout_p", ctypes.c_float),
                ("dropout_seed", ctypes.c_uint64), ("dropout_offset", ctypes.c_uint32)]


SIGNATURES["fa_attention_fwd"] = (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I,
                                       ctypes.POINTER(AttentionOptions), _P])
SIGNATURES["fa_attention_fwd_split"] = (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I,
                                             ctypes.POINTER(AttentionOptions), _P, ctypes.c_size_t,
                                             _P])
SIGNATURES["fa_attention_bwd"] = (_I, [_P] * 9 + [_I, _I, _I, _I, ctypes.POINTER(AttentionOptions),
                                                  _P, ctypes.c_size_t, _P])


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libfa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "exact_io_aware_11_gb300.build.build() (needs nvcc)")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_qkv(*ts):
    for t in ts:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("exact attention runs on CUDA tensors only")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("expected contiguous bf16 tensors of shape [B, H, N, d]")
        if t.shape != ts[0].shape:
            raise ValueError("q, k, v (and o, dout) must have the same shape")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _raise(rc: int, where: str):
    if rc != FA_OK:
        raise FaError(rc, where)


def fwd_workspace_bytes(B: int, H: int, N: int, d: int, causal: bool = False) -> int:
    """Workspace bytes with which the forward splits its last wave (0: no split)."""
    return int(lib().fa_fwd_workspace_bytes(B, H, N, d, int(bool(causal))))


def bwd_split_workspace_bytes(B: int, H: int, N: int, d: int, causal: bool = False) -> int:
    """Backward workspace bytes that also enable the split of its last wave."""
    return int(lib().fa_bwd_split_workspace_bytes(B, H, N, d, int(bool(causal))))


def _bwd_workspace(q, causal, kv_len, block_mask, split, workspace):
    if workspace is not None:
        return workspace
    B, H, N, d = q.shape
    need = (bwd_split_workspace_bytes(B, H, N, d, causal)
            if split and kv_len is None and block_mask is None else bwd_workspace_bytes(B, H, N, d))
    return torch.empty(need, dtype=torch.uint8, device=q.device)


def _fwd_workspace(q, causal, kv_len, block_mask, split, workspace):
    """(pointer, bytes, tensor) of the forward's split workspace, or (None, 0, None)."""
    if workspace is not None:
        return workspace.data_ptr(), workspace.numel() * workspace.element_size(), workspace
    if not split or kv_len is not None or block_mask is not None:
        return None, 0, None
    B, H, N, d = q.shape
    need = fwd_workspace_bytes(B, H, N, d, causal)
    if need == 0:
        return None, 0, None
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    return ws.data_ptr(), need, ws


def forward(q, k, v, causal: bool = False, scale: float | None = None, kv_len=None,
            out=None, lse=None, stream=None, split: bool = True, workspace=None):
    """O, LSE = exact attention forward (fa_fwd_split: fa_fwd_kpad, with the
    last wave of work spread over every SM when that helps and split=True).
    `workspace`: optional uint8 CUDA tensor of fwd_workspace_bytes(...) bytes."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if kv_len is not None and (kv_len.dtype != torch.int32 or not kv_len.is_cuda):
        raise ValueError("kv_len must be a CUDA int32 tensor of shape [B]")
    wp, wn, _ws = _fwd_workspace(q, causal, kv_len, None, split, workspace)
    rc = lib().fa_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                            B, H, N, d, int(bool(causal)), scale, _ptr(kv_len), wp, wn,
                            _stream_ptr(stream))
    _raise(rc, "fa_fwd_split")
    return o, l


def blocksparse_forward(q, k, v, block_mask, scale: float | None = None, block_size: int = 128,
                        out=None, lse=None, stream=None):
    """O, LSE = block-sparse exact attention forward (fa_blocksparse_fwd)."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if block_mask.dtype != torch.uint8 or not block_mask.is_cuda or not block_mask.is_contiguous():
        raise ValueError("block_mask must be a contiguous CUDA uint8 tensor [nb, nb]")
    nb = (N + block_size - 1) // block_size
    if tuple(block_mask.shape) != (nb, nb):
        raise ValueError(f"block_mask must have shape ({nb}, {nb})")
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    rc = lib().fa_blocksparse_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  l.data_ptr(), B, H, N, d, scale, block_mask.data_ptr(),
                                  int(block_size), _stream_ptr(stream))
    _raise(rc, "fa_blocksparse_fwd")
    return o, l


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, N, d))


def backward(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
             kv_len=None, workspace=None, dq=None, dk=None, dv=None, stream=None,
             split: bool = True):
    """dQ, dK, dV of L = sum(dout * O) (fa_bwd). `workspace` is an optional
    uint8 CUDA tensor of at least bwd_workspace_bytes(...) bytes (with
    bwd_split_workspace_bytes(...) or more the last wave is split over every
    SM); without one, the split size is allocated unless split=False."""
    _check_qkv(q, k, v, o, dout)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws = _bwd_workspace(q, causal, kv_len, None, split, workspace)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if kv_len is not None and (kv_len.dtype != torch.int32 or not kv_len.is_cuda):
        raise ValueError("kv_len must be a CUDA int32 tensor of shape [B]")
    rc = lib().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                      lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                      int(bool(causal)), scale, _ptr(kv_len), ws.data_ptr(), ws.numel(),
                      _stream_ptr(stream))
    _raise(rc, "fa_bwd")
    return dq, dk, dv


def blocksparse_backward(q, k, v, o, dout, lse, block_mask, scale: float | None = None,
                         block_size: int = 128, workspace=None, dq=None, dk=None, dv=None,
                         stream=None):
    """dQ, dK, dV of the block-sparse forward (fa_blocksparse_bwd)."""
    _check_qkv(q, k, v, o, dout)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if block_mask.dtype != torch.uint8 or not block_mask.is_cuda or not block_mask.is_contiguous():
        raise ValueError("block_mask must be a contiguous CUDA uint8 tensor [nb, nb]")
    nb = (N + block_size - 1) // block_size
    if tuple(block_mask.shape) != (nb, nb):
        raise ValueError(f"block_mask must have shape ({nb}, {nb})")
    need = bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device) if workspace is None else workspace
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    rc = lib().fa_blocksparse_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), B, H, N, d, scale, block_mask.data_ptr(),
                                  int(block_size), ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    _raise(rc, "fa_blocksparse_bwd")
    return dq, dk, dv


def _check_dropout(p, seed, offset):
    p = float(p)
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout_p must be in [0, 1)")
    if not (0 <= int(seed) < 2 ** 64) or not (0 <= int(offset) < 2 ** 32):
        raise ValueError("seed must fit in 64 bits and offset in 32 bits")
    return p, int(seed), int(offset)


def dropout_forward(q, k, v, dropout_p: float, seed: int, offset: int = 0, causal: bool = False,
                    scale: float | None = None, kv_len=None, out=None, lse=None, stream=None):
    """O, LSE of attention with fused dropout on P (fa_dropout_fwd)."""
    _check_qkv(q, k, v)
    p, seed, offset = _check_dropout(dropout_p, seed, offset)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if kv_len is not None and (kv_len.dtype != torch.int32 or not kv_len.is_cuda):
        raise ValueError("kv_len must be a CUDA int32 tensor of shape [B]")
    rc = lib().fa_dropout_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              l.data_ptr(), B, H, N, d, int(bool(causal)), scale, _ptr(kv_len), p,
                              seed, offset, _stream_ptr(stream))
    _raise(rc, "fa_dropout_fwd")
    return o, l


def dropout_backward(q, k, v, o, dout, lse, dropout_p: float, seed: int, offset: int = 0,
                     causal: bool = False, scale: float | None = None, kv_len=None,
                     workspace=None, dq=None, dk=None, dv=None, stream=None):
    """dQ, dK, dV of dropout_forward with the same dropout_p, seed and offset
    (fa_dropout_bwd)."""
    _check_qkv(q, k, v, o, dout)
    p, seed, offset = _check_dropout(dropout_p, seed, offset)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws = _bwd_workspace(q, causal, kv_len, None, True, workspace)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if kv_len is not None and (kv_len.dtype != torch.int32 or not kv_len.is_cuda):
        raise ValueError("kv_len must be a CUDA int32 tensor of shape [B]")
    rc = lib().fa_dropout_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, int(bool(causal)), scale, _ptr(kv_len),
                              p, seed, offset, ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    _raise(rc, "fa_dropout_bwd")
    return dq, dk, dv


def dropout_mask(B: int, H: int, N: int, dropout_p: float, seed: int, offset: int = 0,
                 device=None, out=None, stream=None):
    """uint8 [B, H, N, N] keep decisions (1 = kept) of the dropout calls with the
    same arguments (fa_dropout_mask)."""
    p, seed, offset = _check_dropout(dropout_p, seed, offset)
    keep = (torch.empty((B, H, N, N), dtype=torch.uint8, device=device or "cuda")
            if out is None else out)
    if not keep.is_cuda or keep.dtype != torch.uint8 or not keep.is_contiguous():
        raise ValueError("out must be a contiguous CUDA uint8 tensor [B, H, N, N]")
    rc = lib().fa_dropout_mask(B, H, N, p, seed, offset, keep.data_ptr(), _stream_ptr(stream))
    _raise(rc, "fa_dropout_mask")
    return keep


def _check_views(*ts):
    """[B, H, N, d] bf16 CUDA views with a contiguous d axis and one set of strides."""
    for t in ts:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("exact attention runs on CUDA tensors only")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or t.stride(3) != 1:
            raise ValueError("expected bf16 [B, H, N, d] views with a contiguous last axis")
        if t.shape != ts[0].shape or t.stride() != ts[0].stride():
            raise ValueError("all [B, H, N, d] tensors of a call must share shape and strides")


def _options(q, causal, scale, kv_len, block_mask, block_size, dropout_p, seed, offset):
    B, H, N, d = q.shape
    opt = AttentionOptions()
    opt.stride_b, opt.stride_h, opt.stride_n = q.stride(0), q.stride(1), q.stride(2)
    opt.causal = int(bool(causal))
    opt.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if kv_len is not None and (kv_len.dtype != torch.int32 or not kv_len.is_cuda):
        raise ValueError("kv_len must be a CUDA int32 tensor of shape [B]")
    opt.kv_len = _ptr(kv_len)
    if block_mask is not None:
        if block_mask.dtype != torch.uint8 or not block_mask.is_cuda or not block_mask.is_contiguous():
            raise ValueError("block_mask must be a contiguous CUDA uint8 tensor [nb, nb]")
        nb = (N + block_size - 1) // block_size
        if tuple(block_mask.shape) != (nb, nb):
            raise ValueError(f"block_mask must have shape ({nb}, {nb})")
    opt.block_mask = _ptr(block_mask)
    opt.block_size = int(block_size)
    p, seed, offset = _check_dropout(dropout_p, seed, offset)
    opt.dropout_p, opt.dropout_seed, opt.dropout_offset = p, seed, offset
    return opt


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, kv_len=None,
                      block_mask=None, block_size: int = 128, dropout_p: float = 0.0,
                      seed: int = 0, offset: int = 0, out=None, lse=None, stream=None,
                      split: bool = True, workspace=None):
    """O, LSE with every option at once (fa_attention_fwd). q, k, v are
    [B, H, N, d] views sharing one set of strides -- e.g. x.transpose(1, 2) of
    a [B, N, H, d] tensor; O is returned with the same strides."""
    _check_views(q, k, v)
    B, H, N, d = q.shape
    opt = _options(q, causal, scale, kv_len, block_mask, block_size, dropout_p, seed, offset)
    o = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device) if out is None else out
    _check_views(q, o)
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    wp, wn, _ws = _fwd_workspace(q, causal, kv_len, block_mask, split, workspace)
    rc = lib().fa_attention_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      l.data_ptr(), B, H, N, d, ctypes.byref(opt), wp, wn,
                                      _stream_ptr(stream))
    _raise(rc, "fa_attention_fwd_split")
    return o, l


def attention_backward(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
                       kv_len=None, block_mask=None, block_size: int = 128,
                       dropout_p: float = 0.0, seed: int = 0, offset: int = 0, workspace=None,
                       dq=None, dk=None, dv=None, stream=None, split: bool = True):
    """dQ, dK, dV of attention_forward with the same options (fa_attention_bwd);
    the gradients have the inputs' strides."""
    _check_views(q, k, v, o, dout)
    B, H, N, d = q.shape
    opt = _options(q, causal, scale, kv_len, block_mask, block_size, dropout_p, seed, offset)
    ws = _bwd_workspace(q, causal, kv_len, block_mask, split, workspace)

    def like():
        return torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)

    dq = like() if dq is None else dq
    dk = like() if dk is None else dk
    dv = like() if dv is None else dv
    _check_views(q, dq, dk, dv)
    rc = lib().fa_attention_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), B, H, N, d, ctypes.byref(opt), ws.data_ptr(),
                                ws.numel(), _stream_ptr(stream))
    _raise(rc, "fa_attention_bwd")
    return dq, dk, dv


def device_status() -> int:
    """Read-and-clear the device-side status word (call after a synchronize)."""
    return int(lib().fa_device_status())


def selftest_wait_timeout(limit_cycles: int, stream=None) -> int:
    return int(lib().fa_selftest_wait_timeout(int(limit_cycles), _stream_ptr(stream)))
