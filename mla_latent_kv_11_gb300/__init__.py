"""Python binding of libmla.so: weight-absorbed MLA over a paged latent KV cache.

The functions carry the C ABI's names (``include/mla.h``) and only marshal
arguments: a torch tensor becomes an ``mla_tensor`` view (its ``data_ptr()``,
which includes the storage offset, its shape and its element strides), the
stream defaults to torch's current CUDA stream, and a non-OK status raises
:class:`MlaError` with the library's message. Every step of the path runs in
the library's CUDA kernels; there is no other implementation to fall back on,
so a missing ``libmla.so`` raises on first use.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_TIMEOUT, MLA_ERR_DEVICE_DATA = range(6)
MLA_F32, MLA_BF16 = 0, 1


class MlaError(RuntimeError):
    """A call into libmla.so returned a status other than MLA_OK."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class MlaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("rank", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


_lib_handle: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded libmla.so (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m mla_latent_kv_11_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        T = MlaTensor
        sigs = {
            "mla_abi_version": ([], ctypes.c_int),
            "mla_last_error": ([], ctypes.c_char_p),
            "mla_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "mla_absorb_q": ([ctypes.c_int, T, T, T, P], ctypes.c_int),
            "mla_concat_q": ([ctypes.c_int, T, T, T, P], ctypes.c_int),
            "mla_cache_write": ([ctypes.c_int, T, T, T, P, I64, P], ctypes.c_int),
            "mla_decode": ([ctypes.c_int, T, P, T, T, P, I64, I32, P, I32, I32, F32, I32, P, SZ, P],
                           ctypes.c_int),
            "mla_decode_workspace_size": ([I32, I32, I32, I32], SZ),
            "mla_prefill": ([ctypes.c_int, T, P, T, T, P, I64, I32, P, P, I32, I32, I32, I32, F32, P,
                             SZ, P], ctypes.c_int),
            "mla_prefill_workspace_size": ([I32], SZ),
            "mla_v_up": ([ctypes.c_int, T, T, T, P], ctypes.c_int),
            "mla_decode_noalloc": ([ctypes.c_int, T, P, T, T, P, I64, I32, P, I32, I32, F32, I32, P],
                                   ctypes.c_int),
            "mla_cache_write_fp8": ([ctypes.c_int, T, T, T, P, I64, P, P], ctypes.c_int),
            "mla_concat_q_cache_write": ([ctypes.c_int, T, T, T, T, T, T, P, I64, P], ctypes.c_int),
            "mla_absorb_concat_cache_write": ([ctypes.c_int, T, T, T, T, T, T, T, P, I64, P], ctypes.c_int),
            "mla_decode_fp8": ([ctypes.c_int, T, P, T, T, P, I64, I32, P, I32, I32, F32, P, P, I32, P, SZ, P],
                               ctypes.c_int),
            "mla_decode_sparse_fp8": ([ctypes.c_int, T, P, T, T, P, I64, I32, F32, I32, P, SZ, P], ctypes.c_int),
            "mla_decode_sparse_workspace_size": ([I32, I32, I32, I32], SZ),
            "mla_decode_v_up": ([ctypes.c_int, T, P, T, T, P, I64, I32, P, I32, I32, F32, T, I32, P, SZ, P],
                                ctypes.c_int),
            "mla_decode_v_up_workspace_size": ([I32, I32, I32, I32], SZ),
            "mla_device_error": ([P], ctypes.c_int),
            "mla_check_bounded_wait": ([ctypes.c_uint32, P], ctypes.c_int),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(h, name)
            fn.argtypes = args
            fn.restype = res
        _lib_handle = h
    return _lib_handle


def _status_name(status: int) -> str:
    names = ["MLA_OK", "MLA_ERR_INVALID_ARG", "MLA_ERR_UNSUPPORTED", "MLA_ERR_CUDA",
             "MLA_ERR_TIMEOUT", "MLA_ERR_DEVICE_DATA"]
    return names[status] if 0 <= status < len(names) else f"status {status}"


def _check(status: int) -> None:
    if status != MLA_OK:
        raise MlaError(status, lib().mla_last_error().decode(errors="replace"))


def _dtype_code(*tensors) -> int:
    import torch
    dts = {t.dtype for t in tensors if t is not None}
    if len(dts) != 1:
        raise MlaError(MLA_ERR_INVALID_ARG, f"tensors disagree on dtype: {sorted(map(str, dts))}")
    dt = dts.pop()
    if dt == torch.float32:
        return MLA_F32
    if dt == torch.bfloat16:
        return MLA_BF16
    raise MlaError(MLA_ERR_INVALID_ARG, f"unsupported dtype {dt}")


def as_mla_tensor(t) -> MlaTensor:
    """Describe a torch tensor (any strides) as an mla_tensor view."""
    if t.dim() > 4:
        raise MlaError(MLA_ERR_INVALID_ARG, "rank > 4")
    m = MlaTensor()
    m.data = t.data_ptr() if t.numel() > 0 else None
    m.rank = t.dim()
    for i, (n, s) in enumerate(zip(t.shape, t.stride())):
        m.shape[i] = n
        m.stride[i] = s
    return m


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def mla_absorb_q(q_lat_out, q_nope, w_uk, stream=None) -> None:
    """Step 1: q_lat[h,b,:] = q_nope[h,b,:] @ w_uk[h] (views [H,B,L], [H,B,P], [H,P,L])."""
    _check(lib().mla_absorb_q(_dtype_code(q_lat_out, q_nope, w_uk), as_mla_tensor(q_lat_out),
                              as_mla_tensor(q_nope), as_mla_tensor(w_uk), _stream(stream)))


def mla_concat_q(q_cat_out, nope, rope, stream=None) -> None:
    """Step 2: q_cat[t,h,:] = [nope[t,h,:] | rope[t,h or 0,:]], a bit copy."""
    _check(lib().mla_concat_q(_dtype_code(q_cat_out, nope, rope), as_mla_tensor(q_cat_out),
                              as_mla_tensor(nope), as_mla_tensor(rope), _stream(stream)))


def mla_cache_write(cache, kv_c, k_pe, slot_mapping, stream=None) -> None:
    """Step 3: cache[s // page, s % page, :] = [kv_c[i] | k_pe[i]] for s = slot_mapping[i] >= 0."""
    import torch
    if slot_mapping.dtype != torch.int64:
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be int64")
    if slot_mapping.numel() and not slot_mapping.is_contiguous():
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be contiguous")
    _check(lib().mla_cache_write(_dtype_code(cache, kv_c, k_pe), as_mla_tensor(cache),
                                 as_mla_tensor(kv_c), as_mla_tensor(k_pe), _ptr(slot_mapping),
                                 slot_mapping.numel(), _stream(stream)))


def _fp8_cache(cache):
    """An e4m3 cache as a byte view (torch.float8_e4m3fn or uint8 storage of the codes)."""
    import torch
    if cache.dtype == torch.uint8:
        return cache
    if cache.dtype == getattr(torch, "float8_e4m3fn", None):
        return cache.view(torch.uint8)
    raise MlaError(MLA_ERR_INVALID_ARG, "an fp8 cache must be float8_e4m3fn or uint8 codes")


def _f32_scalar(t, name):
    import torch
    if t is None:
        return None
    if t.dtype != torch.float32 or t.numel() != 1 or not t.is_cuda:
        raise MlaError(MLA_ERR_INVALID_ARG, f"{name} must be a device float32 tensor of one element")
    return t.data_ptr()


def mla_cache_write_fp8(cache, kv_c, k_pe, slot_mapping, scale, stream=None) -> None:
    """Step 3 into an e4m3 cache: row s = e4m3([kv_c[i] | k_pe[i]] / scale) for s = slot_mapping[i] >= 0."""
    import torch
    if slot_mapping.dtype != torch.int64:
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be int64")
    if slot_mapping.numel() and not slot_mapping.is_contiguous():
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be contiguous")
    if kv_c.dtype != k_pe.dtype or kv_c.dtype not in (torch.float32, torch.bfloat16):
        raise MlaError(MLA_ERR_INVALID_ARG, "kv_c and k_pe must both be float32 or both bfloat16")
    src = MLA_F32 if kv_c.dtype == torch.float32 else MLA_BF16
    _check(lib().mla_cache_write_fp8(src, as_mla_tensor(_fp8_cache(cache)), as_mla_tensor(kv_c),
                                     as_mla_tensor(k_pe), _ptr(slot_mapping), slot_mapping.numel(),
                                     _f32_scalar(scale, "scale"), _stream(stream)))


def mla_concat_q_cache_write(q_cat_out, nope, rope, cache, kv_c, k_pe, slot_mapping, stream=None) -> None:
    """Steps 2 and 3 in one launch: mla_concat_q(q_cat_out, nope, rope) and
    mla_cache_write(cache, kv_c, k_pe, slot_mapping)."""
    import torch
    if slot_mapping.dtype != torch.int64:
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be int64")
    if slot_mapping.numel() and not slot_mapping.is_contiguous():
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be contiguous")
    _check(lib().mla_concat_q_cache_write(_dtype_code(q_cat_out, nope, rope, cache, kv_c, k_pe),
                                          as_mla_tensor(q_cat_out), as_mla_tensor(nope), as_mla_tensor(rope),
                                          as_mla_tensor(cache), as_mla_tensor(kv_c), as_mla_tensor(k_pe),
                                          _ptr(slot_mapping), slot_mapping.numel(), _stream(stream)))


def mla_absorb_concat_cache_write(q_cat, q_nope, w_uk, q_pe, cache, kv_c, k_pe, slot_mapping, stream=None) -> None:
    """Steps 1 to 3 in one call: mla_absorb_q into q_cat's first L columns (q_nope [H,T,P],
    w_uk [H,P,L]), then the rope columns of q_cat and the cache write of the new rows, the
    copies running alongside the absorb."""
    import torch
    if slot_mapping.dtype != torch.int64:
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be int64")
    if slot_mapping.numel() and not slot_mapping.is_contiguous():
        raise MlaError(MLA_ERR_INVALID_ARG, "slot_mapping must be contiguous")
    _check(lib().mla_absorb_concat_cache_write(_dtype_code(q_cat, q_nope, w_uk, q_pe, cache, kv_c, k_pe),
                                               as_mla_tensor(q_cat), as_mla_tensor(q_nope), as_mla_tensor(w_uk),
                                               as_mla_tensor(q_pe), as_mla_tensor(cache), as_mla_tensor(kv_c),
                                               as_mla_tensor(k_pe), _ptr(slot_mapping), slot_mapping.numel(),
                                               _stream(stream)))


def mla_decode_workspace_size(batch: int, num_heads: int, kv_lora_rank: int, num_splits: int = 0) -> int:
    return int(lib().mla_decode_workspace_size(batch, num_heads, kv_lora_rank, num_splits))


def _check_int32_table(block_table, seq_lens):
    import torch
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise MlaError(MLA_ERR_INVALID_ARG, "block_table and sequence lengths must be int32")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise MlaError(MLA_ERR_INVALID_ARG, "block_table must be [B, max_blocks] with unit column stride")
    if not seq_lens.is_contiguous():
        raise MlaError(MLA_ERR_INVALID_ARG, "sequence lengths must be contiguous")


def mla_decode(o_lat_out, q_cat, cache, block_table, seq_lens, kv_lora_rank: int, rope_dim: int,
               softmax_scale: float, lse_out=None, num_splits: int = 0, workspace=None,
               stream=None) -> None:
    """Step 4: split-KV paged decode; o_lat_out [B,H,L], optional lse_out float32 [B,H]."""
    import torch
    _check_int32_table(block_table, seq_lens)
    if lse_out is not None and (lse_out.dtype != torch.float32 or not lse_out.is_contiguous()):
        raise MlaError(MLA_ERR_INVALID_ARG, "lse_out must be contiguous float32")
    B, H = q_cat.shape[0], q_cat.shape[1]
    need = mla_decode_workspace_size(B, H, kv_lora_rank, num_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_cat.device)
    _check(lib().mla_decode(_dtype_code(o_lat_out, q_cat, cache), as_mla_tensor(o_lat_out),
                            _ptr(lse_out), as_mla_tensor(q_cat), as_mla_tensor(cache),
                            block_table.data_ptr(), block_table.stride(0), block_table.shape[1],
                            seq_lens.data_ptr(), kv_lora_rank, rope_dim, softmax_scale, num_splits,
                            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            _stream(stream)))


def mla_decode_fp8(o_lat_out, q_cat, cache, block_table, seq_lens, kv_lora_rank: int, rope_dim: int,
                   softmax_scale: float, descale_q=None, descale_k=None, lse_out=None, num_splits: int = 0,
                   workspace=None, stream=None) -> None:
    """Step 4 over an e4m3 cache: mla_decode with cache values = code * descale_k and q * descale_q."""
    import torch
    _check_int32_table(block_table, seq_lens)
    if lse_out is not None and (lse_out.dtype != torch.float32 or not lse_out.is_contiguous()):
        raise MlaError(MLA_ERR_INVALID_ARG, "lse_out must be contiguous float32")
    if o_lat_out.dtype != q_cat.dtype:
        raise MlaError(MLA_ERR_INVALID_ARG, "o_lat_out and q_cat must share a dtype")
    code = MLA_F32 if q_cat.dtype == torch.float32 else MLA_BF16
    B, H = q_cat.shape[0], q_cat.shape[1]
    need = mla_decode_workspace_size(B, H, kv_lora_rank, num_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_cat.device)
    _check(lib().mla_decode_fp8(code, as_mla_tensor(o_lat_out), _ptr(lse_out), as_mla_tensor(q_cat),
                                as_mla_tensor(_fp8_cache(cache)), block_table.data_ptr(), block_table.stride(0),
                                block_table.shape[1], seq_lens.data_ptr(), kv_lora_rank, rope_dim, softmax_scale,
                                _f32_scalar(descale_q, "descale_q"), _f32_scalar(descale_k, "descale_k"),
                                num_splits, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream(stream)))


def mla_decode_sparse_workspace_size(batch: int, num_heads: int, topk: int, num_splits: int = 0) -> int:
    return int(lib().mla_decode_sparse_workspace_size(batch, num_heads, topk, num_splits))


def mla_decode_sparse_fp8(o_lat_out, q_cat, cache, indices, softmax_scale: float, lse_out=None,
                          num_splits: int = 0, workspace=None, stream=None) -> None:
    """Sparse top-k decode over an fp8 ds_mla cache: query b attends the slots indices[b]
    (int32 [B, topk] or [B, 1, topk], -1 = padding) of a uint8 [num_blocks, page, 656]
    (or [num_blocks, page, 1, 656]) cache; o_lat_out [B,H,512], q_cat [B,H,576]."""
    import torch
    if cache.dtype != torch.uint8:
        raise MlaError(MLA_ERR_INVALID_ARG, "a ds_mla cache is uint8 bytes")
    if cache.dim() == 4 and cache.shape[2] == 1:
        cache = cache[:, :, 0]
    if indices.dim() == 3 and indices.shape[1] == 1:
        indices = indices[:, 0]
    if indices.dtype != torch.int32 or indices.dim() != 2 or (indices.numel() and indices.stride(1) != 1):
        raise MlaError(MLA_ERR_INVALID_ARG, "indices must be int32 [B, topk] with unit column stride")
    if lse_out is not None and (lse_out.dtype != torch.float32 or not lse_out.is_contiguous()):
        raise MlaError(MLA_ERR_INVALID_ARG, "lse_out must be contiguous float32")
    B, H = q_cat.shape[0], q_cat.shape[1]
    if workspace is None:
        workspace = torch.empty(mla_decode_sparse_workspace_size(B, H, indices.shape[-1], num_splits),
                                dtype=torch.uint8, device=q_cat.device)
    _check(lib().mla_decode_sparse_fp8(_dtype_code(o_lat_out, q_cat), as_mla_tensor(o_lat_out), _ptr(lse_out),
                                       as_mla_tensor(q_cat), as_mla_tensor(cache), _ptr(indices),
                                       indices.stride(0) if indices.dim() == 2 else 0, indices.shape[-1],
                                       softmax_scale, num_splits, workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


def mla_decode_v_up_workspace_size(batch: int, num_heads: int, kv_lora_rank: int, num_splits: int = 0) -> int:
    return int(lib().mla_decode_v_up_workspace_size(batch, num_heads, kv_lora_rank, num_splits))


def mla_decode_v_up(out, q_cat, cache, block_table, seq_lens, kv_lora_rank: int, rope_dim: int,
                    softmax_scale: float, w_uv, lse_out=None, num_splits: int = 0, workspace=None,
                    stream=None) -> None:
    """Steps 4 and 5 as one call: out[b,h,:] = decode(q_cat)[b,h,:] @ w_uv[h]; out [B,H,V], w_uv [H,L,V]."""
    import torch
    _check_int32_table(block_table, seq_lens)
    if lse_out is not None and (lse_out.dtype != torch.float32 or not lse_out.is_contiguous()):
        raise MlaError(MLA_ERR_INVALID_ARG, "lse_out must be contiguous float32")
    B, H = q_cat.shape[0], q_cat.shape[1]
    if workspace is None:
        workspace = torch.empty(mla_decode_v_up_workspace_size(B, H, kv_lora_rank, num_splits), dtype=torch.uint8,
                                device=q_cat.device)
    _check(lib().mla_decode_v_up(_dtype_code(out, q_cat, cache, w_uv), as_mla_tensor(out), _ptr(lse_out),
                                 as_mla_tensor(q_cat), as_mla_tensor(cache), block_table.data_ptr(),
                                 block_table.stride(0), block_table.shape[1], seq_lens.data_ptr(), kv_lora_rank,
                                 rope_dim, softmax_scale, as_mla_tensor(w_uv), num_splits, workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def mla_prefill_workspace_size(batch: int) -> int:
    return int(lib().mla_prefill_workspace_size(batch))


def mla_prefill(o_lat_out, q_cat, cache, block_table, cu_seqlens_q, seq_lens_kv, max_q_len: int,
                kv_lora_rank: int, rope_dim: int, softmax_scale: float, lse_out=None, workspace=None,
                stream=None) -> None:
    """Step 4 (prefill): causal attention of many queries per sequence over the paged cache."""
    import torch
    _check_int32_table(block_table, seq_lens_kv)
    if cu_seqlens_q.dtype != torch.int32 or not cu_seqlens_q.is_contiguous():
        raise MlaError(MLA_ERR_INVALID_ARG, "cu_seqlens_q must be contiguous int32")
    if lse_out is not None and (lse_out.dtype != torch.float32 or not lse_out.is_contiguous()):
        raise MlaError(MLA_ERR_INVALID_ARG, "lse_out must be contiguous float32")
    if workspace is None:
        workspace = torch.empty(mla_prefill_workspace_size(seq_lens_kv.numel()), dtype=torch.uint8,
                                device=q_cat.device)
    _check(lib().mla_prefill(_dtype_code(o_lat_out, q_cat, cache), as_mla_tensor(o_lat_out),
                             _ptr(lse_out), as_mla_tensor(q_cat), as_mla_tensor(cache),
                             block_table.data_ptr(), block_table.stride(0), block_table.shape[1],
                             cu_seqlens_q.data_ptr(), seq_lens_kv.data_ptr(), seq_lens_kv.numel(),
                             max_q_len, kv_lora_rank, rope_dim, softmax_scale, workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream(stream)))


def mla_v_up(out, o_lat, w_uv, stream=None) -> None:
    """Step 5: out[h,b,:] = o_lat[h,b,:] @ w_uv[h] (views [H,B,V], [H,B,L], [H,L,V])."""
    _check(lib().mla_v_up(_dtype_code(out, o_lat, w_uv), as_mla_tensor(out), as_mla_tensor(o_lat),
                          as_mla_tensor(w_uv), _stream(stream)))


def mla_decode_noalloc(o_lat_out, q_cat, cache, block_table, seq_lens, kv_lora_rank: int,
                       rope_dim: int, softmax_scale: float, lse_out=None, num_splits: int = 0,
                       stream=None) -> None:
    """mla_decode for callers that cannot allocate device memory: no workspace, the
    scratch is a fixed array inside the library (shared by all calls; do not overlap
    calls on the GPU)."""
    import torch
    _check_int32_table(block_table, seq_lens)
    if lse_out is not None and (lse_out.dtype != torch.float32 or not lse_out.is_contiguous()):
        raise MlaError(MLA_ERR_INVALID_ARG, "lse_out must be contiguous float32")
    _check(lib().mla_decode_noalloc(_dtype_code(o_lat_out, q_cat, cache), as_mla_tensor(o_lat_out),
                                    _ptr(lse_out), as_mla_tensor(q_cat), as_mla_tensor(cache),
                                    block_table.data_ptr(), block_table.stride(0), block_table.shape[1],
                                    seq_lens.data_ptr(), kv_lora_rank, rope_dim, softmax_scale,
                                    num_splits, _stream(stream)))


def mla_check_bounded_wait(limit_us: int, stream=None) -> None:
    """Run the kernels' bounded wait on an mbarrier nothing arrives on (see include/mla.h)."""
    _check(lib().mla_check_bounded_wait(limit_us, _stream(stream)))


def mla_device_error(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    _check(lib().mla_device_error(_stream(stream)))
