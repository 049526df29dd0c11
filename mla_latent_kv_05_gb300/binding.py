"""Thin ctypes binding over libmla_gb300.so (the C ABI in include/mla_decode.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their raw pointers and the current CUDA stream are handed to the
library, and every step of the decode runs in the library's kernels.  There
is no fallback: if the library is missing or a call fails, an error is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

MLA_OK = 0
_STATUS = {
    0: "MLA_OK", -1: "MLA_ERR_INVALID_ARG", -2: "MLA_ERR_UNSUPPORTED", -3: "MLA_ERR_WORKSPACE",
    -4: "MLA_ERR_CUDA", -5: "MLA_STATUS_BAD_PAGE", -6: "MLA_STATUS_TIMEOUT", -7: "MLA_STATUS_BAD_SEQ_LEN",
    -8: "MLA_STATUS_BAD_INDEX",
}

# Exported entry points and their C signatures (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "mla_workspace_size": (_I, [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "mla_decode_bf16": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                             ctypes.c_size_t, _P]),
    "mla_decode_bf16_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                                     _P]),
    "mla_decode_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                            ctypes.c_size_t, _P]),
    "mla_decode_fp4": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                            ctypes.c_size_t, _P]),
    "mla_decode_fp8_v41": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                                ctypes.c_size_t, _P]),
    "mla_decode_fp4_v41": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                                ctypes.c_size_t, _P]),
    "mla_workspace_size_sparse": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "mla_decode_sparse_bf16": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                                    ctypes.c_size_t, _P]),
    "mla_up_project_wuv": (_I, [_P, _P, _I, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "mla_combine_splits": (_I, [_P, _P, _P, _I, _I, _P, _P, _P]),
    "mla_get_status": (_I, [_P, _P]),
    "mla_profile_next_decode": (_I, [_P, _P]),
    "mla_status_string": (ctypes.c_char_p, [_I]),
}

_lib = None


class MLAError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built ({p} missing): run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().mla_status_string(int(code)).decode()
    except RuntimeError:
        return _STATUS.get(int(code), "MLA_UNKNOWN_STATUS")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _same_device(tensors: dict, current: int) -> None:
    """Every tensor of a call on one CUDA device, the calling thread's current
    one: the library launches its kernels on the current device, which then
    reads and writes these pointers."""
    devs = {name: t.device for name, t in tensors.items() if t is not None}
    first_name, first = next(iter(devs.items()))
    for name, d in devs.items():
        if d != first:
            raise ValueError(f"{name} is on {d} but {first_name} is on {first}")
    if first.index != current:
        raise ValueError(f"the tensors are on {first} but the current device is cuda:{current}; "
                         f"call under torch.cuda.device({first})")


def mla_workspace_size(batch: int, sq: int, num_heads: int = 128, page_size: int = 64) -> int:
    n = ctypes.c_size_t(0)
    rc = load().mla_workspace_size(int(batch), int(sq), int(num_heads), int(page_size), ctypes.byref(n))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_workspace_size")
    return int(n.value)


def alloc_workspace(batch: int, sq: int, device=None) -> torch.Tensor:
    """A zeroed workspace buffer (uint8) of the size the library asks for."""
    n = mla_workspace_size(batch, sq)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _decode(fn_name, q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out, lse, workspace, stream,
            kv_dtype, row_bytes):
    B, Sq, H, D = q_absorbed.shape
    _check(q_absorbed, "q_absorbed", torch.bfloat16, (B, Sq, H, 512))
    _check(q_rope, "q_rope", torch.bfloat16, (B, Sq, H, 64))
    _check(kv_cache, "kv_cache", kv_dtype)
    if kv_cache.dim() != 3 or kv_cache.shape[2] != row_bytes:
        raise ValueError(f"kv_cache must be [num_pages, page_size, {row_bytes}], got {tuple(kv_cache.shape)}")
    _check(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Sq, H, 512), dtype=torch.bfloat16, device=q_absorbed.device)
    if lse is None:
        lse = torch.empty((B, Sq, H), dtype=torch.float32, device=q_absorbed.device)
    _check(out, "out", torch.bfloat16, (B, Sq, H, 512))
    _check(lse, "lse", torch.float32, (B, Sq, H))
    if workspace is None:
        workspace = alloc_workspace(B, Sq, q_absorbed.device)
    _check(workspace, "workspace", torch.uint8)
    _same_device(dict(q_absorbed=q_absorbed, q_rope=q_rope, kv_cache=kv_cache, block_table=block_table,
                      seq_lens=seq_lens, out=out, lse=lse, workspace=workspace), torch.cuda.current_device())
    rc = getattr(load(), fn_name)(
        _ptr(q_absorbed), _ptr(q_rope), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
        int(B), int(Sq), int(H), int(kv_cache.shape[0]), int(kv_cache.shape[1]), int(block_table.shape[1]),
        ctypes.c_float(float(scale)), _ptr(out), _ptr(lse), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
        _stream(stream))
    if rc != MLA_OK:
        raise MLAError(rc, fn_name)
    return out, lse


def mla_decode_bf16(q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out=None, lse=None,
                    workspace=None, stream=None):
    """MLA decode over a bf16 latent cache [num_pages, 64, 576]; returns (out, lse)."""
    return _decode("mla_decode_bf16", q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out, lse,
                   workspace, stream, torch.bfloat16, 576)


def mla_decode_bf16_noalloc(q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out=None, lse=None,
                            device_status=None, stream=None):
    """mla_decode_bf16 on the library's own static scratch (no workspace
    argument; the library allocates nothing).  At most 8192 query rows;
    calls that can overlap in time race on the shared scratch.
    `device_status`: optional int32 CUDA tensor of one element that receives
    the call's device status.  Returns (out, lse)."""
    B, Sq, H, D = q_absorbed.shape
    _check(q_absorbed, "q_absorbed", torch.bfloat16, (B, Sq, H, 512))
    _check(q_rope, "q_rope", torch.bfloat16, (B, Sq, H, 64))
    _check(kv_cache, "kv_cache", torch.bfloat16)
    if kv_cache.dim() != 3 or kv_cache.shape[2] != 576:
        raise ValueError(f"kv_cache must be [num_pages, page_size, 576], got {tuple(kv_cache.shape)}")
    _check(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Sq, H, 512), dtype=torch.bfloat16, device=q_absorbed.device)
    if lse is None:
        lse = torch.empty((B, Sq, H), dtype=torch.float32, device=q_absorbed.device)
    _check(out, "out", torch.bfloat16, (B, Sq, H, 512))
    _check(lse, "lse", torch.float32, (B, Sq, H))
    if device_status is not None:
        _check(device_status, "device_status", torch.int32, (1,))
    _same_device(dict(q_absorbed=q_absorbed, q_rope=q_rope, kv_cache=kv_cache, block_table=block_table,
                      seq_lens=seq_lens, out=out, lse=lse, device_status=device_status),
                 torch.cuda.current_device())
    rc = load().mla_decode_bf16_noalloc(
        _ptr(q_absorbed), _ptr(q_rope), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
        int(B), int(Sq), int(H), int(kv_cache.shape[0]), int(kv_cache.shape[1]), int(block_table.shape[1]),
        ctypes.c_float(float(scale)), _ptr(out), _ptr(lse), _ptr(device_status), _stream(stream))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_bf16_noalloc")
    return out, lse


def mla_decode_fp8(q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out=None, lse=None,
                   workspace=None, stream=None):
    """MLA decode over an FP8 latent cache [num_pages, 64, 594] (uint8 rows:
    576 e4m3 codes then 18 e8m0 scales); returns (out, lse)."""
    return _decode("mla_decode_fp8", q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out, lse,
                   workspace, stream, torch.uint8, 594)


def mla_decode_fp4(q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out=None, lse=None,
                   workspace=None, stream=None):
    """MLA decode over an FP4 latent cache [num_pages, 64, 324] (uint8 rows:
    576 e2m1 codes, two per byte with the even value in the low nibble, then
    36 e8m0 scales, one per 16 values); returns (out, lse)."""
    return _decode("mla_decode_fp4", q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out, lse,
                   workspace, stream, torch.uint8, 324)


def mla_decode_fp8_v41(q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out=None, lse=None,
                       workspace=None, stream=None):
    """MLA decode over an FP8 latent cache in the V4.1 row layout
    [num_pages, 64, 528] (uint8 rows: 512 e4m3 codes, 448 latent then 64
    RoPE, then 16 e8m0 scales, one per 32 codes); returns (out, lse) with
    out [..., 512] whose dims 448..511 are 0 (q_absorbed dims 448..511 are
    ignored)."""
    return _decode("mla_decode_fp8_v41", q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out, lse,
                   workspace, stream, torch.uint8, 528)


def mla_decode_fp4_v41(q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out=None, lse=None,
                       workspace=None, stream=None):
    """MLA decode over an FP4 latent cache in the 288-byte V4.1 row layout
    [num_pages, 64, 288] (uint8 rows: 512 e2m1 codes, two per byte, 448
    latent then 64 RoPE values, then 32 e8m0 scales, one per 16 values);
    returns (out, lse) as mla_decode_fp8_v41 does."""
    return _decode("mla_decode_fp4_v41", q_absorbed, q_rope, kv_cache, block_table, seq_lens, scale, out, lse,
                   workspace, stream, torch.uint8, 288)


def mla_workspace_size_sparse(batch: int, sq: int, topk: int, num_heads: int = 128, page_size: int = 64) -> int:
    n = ctypes.c_size_t(0)
    rc = load().mla_workspace_size_sparse(int(batch), int(sq), int(topk), int(num_heads), int(page_size),
                                          ctypes.byref(n))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_workspace_size_sparse")
    return int(n.value)


def alloc_workspace_sparse(batch: int, sq: int, topk: int, device=None) -> torch.Tensor:
    """A zeroed workspace buffer (uint8) for the sparse decode."""
    n = mla_workspace_size_sparse(batch, sq, topk)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def mla_decode_sparse_bf16(q_absorbed, q_rope, kv_cache, token_slots, scale, out=None, lse=None,
                           workspace=None, stream=None):
    """Sparse top-k decode over a bf16 latent cache [num_pages, 64, 576]:
    query row (b, i) attends over the cache slots token_slots[b, i, :]
    (int32 [B, Sq, topk], slot = page * 64 + offset, -1 = no token).
    Returns (out, lse)."""
    B, Sq, H, D = q_absorbed.shape
    _check(q_absorbed, "q_absorbed", torch.bfloat16, (B, Sq, H, 512))
    _check(q_rope, "q_rope", torch.bfloat16, (B, Sq, H, 64))
    _check(kv_cache, "kv_cache", torch.bfloat16)
    if kv_cache.dim() != 3 or kv_cache.shape[2] != 576:
        raise ValueError(f"kv_cache must be [num_pages, page_size, 576], got {tuple(kv_cache.shape)}")
    _check(token_slots, "token_slots", torch.int32)
    if token_slots.dim() != 3 or tuple(token_slots.shape[:2]) != (B, Sq):
        raise ValueError("token_slots must be [B, Sq, topk]")
    topk = int(token_slots.shape[2])
    if out is None:
        out = torch.empty((B, Sq, H, 512), dtype=torch.bfloat16, device=q_absorbed.device)
    if lse is None:
        lse = torch.empty((B, Sq, H), dtype=torch.float32, device=q_absorbed.device)
    _check(out, "out", torch.bfloat16, (B, Sq, H, 512))
    _check(lse, "lse", torch.float32, (B, Sq, H))
    if workspace is None:
        workspace = alloc_workspace_sparse(B, Sq, topk, q_absorbed.device)
    _check(workspace, "workspace", torch.uint8)
    _same_device(dict(q_absorbed=q_absorbed, q_rope=q_rope, kv_cache=kv_cache, token_slots=token_slots, out=out,
                      lse=lse, workspace=workspace), torch.cuda.current_device())
    rc = load().mla_decode_sparse_bf16(
        _ptr(q_absorbed), _ptr(q_rope), _ptr(kv_cache), _ptr(token_slots), int(B), int(Sq), topk, int(H),
        int(kv_cache.shape[0]), int(kv_cache.shape[1]), ctypes.c_float(float(scale)), _ptr(out), _ptr(lse),
        _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_decode_sparse_bf16")
    return out, lse


def mla_up_project_wuv(latent, w_uv, out=None, workspace=None, stream=None):
    """out[r, h] = w_uv[h] @ latent[r, h]: latent [..., 128, 512] bf16 (the
    decode's output), w_uv [128, 128, 512] bf16 -> [..., 128, 128] bf16."""
    lead = tuple(latent.shape[:-2])
    _check(latent, "latent", torch.bfloat16)
    if tuple(latent.shape[-2:]) != (128, 512):
        raise ValueError("latent must be [..., 128, 512]")
    _check(w_uv, "w_uv", torch.bfloat16, (128, 128, 512))
    rows = 1
    for x in lead:
        rows *= int(x)
    if out is None:
        out = torch.empty(lead + (128, 128), dtype=torch.bfloat16, device=latent.device)
    _check(out, "out", torch.bfloat16, lead + (128, 128))
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=latent.device)
    _check(workspace, "workspace", torch.uint8)
    _same_device(dict(latent=latent, w_uv=w_uv, out=out, workspace=workspace), torch.cuda.current_device())
    rc = load().mla_up_project_wuv(_ptr(latent), _ptr(w_uv), rows, 128, 128, _ptr(out), _ptr(workspace),
                                   ctypes.c_size_t(workspace.numel()), _stream(stream))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_up_project_wuv")
    return out


def mla_combine_splits(partial_out, partial_lse, split_indptr, out=None, lse=None, stream=None):
    """Merge split partials: partial_out [n, 128, 512] fp32, partial_lse [n, 128] fp32,
    split_indptr [rows+1] int32 -> (out [rows, 128, 512] bf16, lse [rows, 128] fp32)."""
    _check(partial_out, "partial_out", torch.float32)
    if partial_out.dim() != 3 or partial_out.shape[2] != 512:
        raise ValueError(f"partial_out must be [n_parts, num_heads, 512], got {tuple(partial_out.shape)}")
    _check(partial_lse, "partial_lse", torch.float32, tuple(partial_out.shape[:2]))
    _check(split_indptr, "split_indptr", torch.int32)
    if split_indptr.dim() != 1 or split_indptr.numel() < 1:
        raise ValueError("split_indptr must be [rows + 1]")
    rows = split_indptr.numel() - 1
    H = partial_out.shape[1]
    if out is None:
        out = torch.empty((rows, H, 512), dtype=torch.bfloat16, device=partial_out.device)
    if lse is None:
        lse = torch.empty((rows, H), dtype=torch.float32, device=partial_out.device)
    _check(out, "out", torch.bfloat16, (rows, H, 512))
    _check(lse, "lse", torch.float32, (rows, H))
    _same_device(dict(partial_out=partial_out, partial_lse=partial_lse, split_indptr=split_indptr, out=out, lse=lse),
                 torch.cuda.current_device())
    rc = load().mla_combine_splits(_ptr(partial_out), _ptr(partial_lse), _ptr(split_indptr), int(rows), int(H),
                                   _ptr(out), _ptr(lse), _stream(stream))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_combine_splits")
    return out, lse


def mla_profile_next_decode(before: torch.cuda.Event, after: torch.cuda.Event) -> None:
    """Have the next decode call record `before`/`after` around its attention
    kernel (on the call's stream)."""
    before.record() if before.cuda_event == 0 else None
    after.record() if after.cuda_event == 0 else None
    rc = load().mla_profile_next_decode(ctypes.c_void_p(before.cuda_event), ctypes.c_void_p(after.cuda_event))
    if rc != MLA_OK:
        raise MLAError(rc, "mla_profile_next_decode")


def mla_get_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load().mla_get_status(_ptr(workspace), _stream(stream)))
