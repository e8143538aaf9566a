"""Thin ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every call checks dtypes, devices, shapes and contiguity of the torch tensors,
then passes raw device pointers, sizes and the current CUDA stream to the C
ABI; all the work runs in the library's CUDA kernels.  PyTorch only supplies
device memory and streams.  There is no fallback: if ``libpkv.so`` has not
been built, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")
_lock = threading.Lock()
_lib = None

PKV_KERNEL_AUTO, PKV_KERNEL_SIMT, PKV_KERNEL_MMA, PKV_KERNEL_TC = 0, 1, 2, 3
DEVERR_NAMES = {0: "none", 1: "slot out of range", 2: "block id out of range",
                3: "context length over max_context_len or the table",
                4: "shared-memory copy timed out"}
_DTYPE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
PKV_FP8_E4M3 = 3

# Every symbol include/pkv.h declares.
EXPORTED = ("pkv_status_string", "pkv_version", "pkv_kv_append", "pkv_attention_plan",
            "pkv_attention_plan_for", "pkv_attention_workspace_size",
            "pkv_paged_decode_attention", "pkv_spec_verify_attention",
            "pkv_read_error_word", "pkv_paged_decode_attention_noalloc",
            "pkv_append_attention", "pkv_tree_verify_attention", "pkv_kv_append_fp8",
            "pkv_paged_attention_fp8", "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_add_sequence",
            "pkv_bm_append", "pkv_bm_fork", "pkv_bm_free", "pkv_bm_sequence",
            "pkv_bm_block_table", "pkv_bm_stats", "pkv_bm_block_info", "pkv_bm_hash",
            "pkv_copy_blocks", "pkv_paged_prefill_attention", "pkv_check_bounded_wait",
            "pkv_host_step_staging_size", "pkv_append_attention_host",
            "pkv_mla_plan", "pkv_mla_workspace_size", "pkv_mla_decode_attention",
            "pkv_mla_append")


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed: {message} (status {status})")
        self.status = status


class Options(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("split_blocks", ctypes.c_int),
                ("stages", ctypes.c_int), ("rows_per_cta", ctypes.c_int),
                ("merge", ctypes.c_int), ("warp_tiles", ctypes.c_int),
                ("blocks_per_iter", ctypes.c_int), ("persistent", ctypes.c_int),
                ("split_waves", ctypes.c_int)]


# Extra launch controls for tuning runs (pkv_options.rows_per_cta / .merge /
# .warp_tiles / .blocks_per_iter / .persistent / .split_waves); module-wide so
# that every binding call passes them.  Empty = planner.
TUNING = {}


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("rows_per_cta", ctypes.c_int),
                ("row_chunks", ctypes.c_int), ("split_blocks", ctypes.c_int),
                ("num_splits", ctypes.c_int), ("grid_x", ctypes.c_int),
                ("grid_y", ctypes.c_int), ("grid_z", ctypes.c_int),
                ("threads_per_cta", ctypes.c_int), ("stages", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int),
                ("smem_bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t),
                ("merge_kernel", ctypes.c_int), ("warp_tiles", ctypes.c_int),
                ("blocks_per_iter", ctypes.c_int), ("split_target", ctypes.c_int),
                ("stream_k", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` "
                    "(there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            f32 = ctypes.c_float
            opt = ctypes.POINTER(Options)
            plan = ctypes.POINTER(Plan)
            L.pkv_status_string.argtypes = [i32]
            L.pkv_status_string.restype = ctypes.c_char_p
            L.pkv_version.argtypes = []
            L.pkv_version.restype = ctypes.c_char_p
            L.pkv_kv_append.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, vp, vp]
            L.pkv_attention_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, opt, plan]
            L.pkv_attention_plan_for.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, opt,
                                                 i32, i32, plan]
            L.pkv_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32,
                                                       opt, ctypes.POINTER(sz)]
            L.pkv_paged_decode_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                                     i32, i32, i32, i64, f32, i32, vp, sz, opt,
                                                     vp, vp]
            L.pkv_spec_verify_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                                    i32, i32, i32, i32, i64, f32, i32, vp, sz,
                                                    opt, vp, vp]
            L.pkv_read_error_word.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
            L.pkv_append_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                               i32, i32, i32, i32, i32, i64, f32, i32, vp, sz,
                                               opt, vp, vp]
            L.pkv_host_step_staging_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32,
                                                     i32, opt, ctypes.POINTER(sz)]
            L.pkv_append_attention_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32,
                                                    i32, i32, i32, i32, i32, i32, i64, f32, i32,
                                                    vp, sz, opt, vp, vp]
            L.pkv_mla_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, opt, plan]
            L.pkv_mla_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, opt,
                                                 ctypes.POINTER(sz)]
            L.pkv_mla_decode_attention.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                   i32, i32, i64, f32, i32, vp, sz, opt, vp, vp]
            L.pkv_mla_append.argtypes = [vp, vp, vp, i64, i32, i32, i64, i32, vp, vp]
            L.pkv_tree_verify_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                                    i32, i32, i32, i32, i64, f32, i32, vp, i64,
                                                    vp, sz, opt, vp, vp]
            L.pkv_kv_append_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, f32,
                                            f32, vp, vp]
            L.pkv_paged_attention_fp8.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                  i32, i32, i32, i64, f32, i32, f32, f32, vp, sz,
                                                  opt, vp, vp]
            L.pkv_paged_decode_attention_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32,
                                                             i32, i32, i32, i32, i32, i64, f32,
                                                             i32, opt, vp, vp]
            pi32, pi64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
            pint, u64 = ctypes.POINTER(ctypes.c_int), ctypes.c_uint64
            L.pkv_bm_create.argtypes = [i64, i32]
            L.pkv_bm_destroy.argtypes = [vp]
            L.pkv_bm_add_sequence.argtypes = [vp, i64, pi32, i32, i32, pint, pi64]
            L.pkv_bm_append.argtypes = [vp, i64, pi32, i32, pi64, pi32, pi32, pint]
            L.pkv_bm_fork.argtypes = [vp, i64, i64]
            L.pkv_bm_free.argtypes = [vp, i64]
            L.pkv_bm_sequence.argtypes = [vp, i64, pi32, i32, pint, pint]
            L.pkv_bm_block_table.argtypes = [vp, pi64, i32, pi32, i32, pi32]
            L.pkv_bm_stats.argtypes = [vp, pi64, pi64, pi64]
            L.pkv_bm_block_info.argtypes = [vp, ctypes.c_int32, pi32, pi32,
                                            ctypes.POINTER(u64)]
            L.pkv_bm_hash.argtypes = [u64, pi32, i32]
            L.pkv_copy_blocks.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, i32, vp, vp]
            L.pkv_check_bounded_wait.argtypes = [vp, ctypes.c_uint32, vp, vp]
            L.pkv_paged_prefill_attention.argtypes = [
                vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, i64,
                ctypes.c_float, i32, ctypes.POINTER(Options), vp, vp]
            for name in EXPORTED:
                if name not in ("pkv_status_string", "pkv_version"):
                    getattr(L, name).restype = i32
            L.pkv_bm_create.restype = vp
            L.pkv_bm_destroy.restype = None
            L.pkv_bm_hash.restype = u64
            _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise PkvError(fn, status, lib().pkv_status_string(status).decode())


def version() -> str:
    return lib().pkv_version().decode()


# The current stream's raw handle, without building a torch.cuda.Stream object
# on every call (that costs several microseconds of host time per call).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor) -> int:
    if _raw_stream is not None:
        return _raw_stream(t.get_device())
    return torch.cuda.current_stream(t.device).cuda_stream


def _opts(kernel: int, split_blocks: int, stages: int = 0, warp_tiles: int = 0):
    rows, merge = TUNING.get("rows_per_cta", 0), TUNING.get("merge", 0)
    warp_tiles = warp_tiles or TUNING.get("warp_tiles", 0)
    kb, pers = TUNING.get("blocks_per_iter", 0), TUNING.get("persistent", 0)
    waves = TUNING.get("split_waves", 0)
    if not any((kernel, split_blocks, stages, rows, merge, warp_tiles, kb, pers, waves)):
        return None
    return ctypes.byref(Options(kernel, split_blocks, stages, rows, merge, warp_tiles, kb, pers,
                                waves))


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _cache_args(k_cache, v_cache):
    _need(k_cache.is_cuda and v_cache.is_cuda, "caches must be CUDA tensors")
    _need(k_cache.dim() == 4 and k_cache.shape == v_cache.shape,
          "k_cache/v_cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    _need(k_cache.dtype == v_cache.dtype and k_cache.dtype in _DTYPE, "cache dtype")
    _need(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")
    return k_cache.shape


def _err_ptr(error_word: Optional[torch.Tensor]):
    if error_word is None:
        return None
    _need(error_word.dtype == torch.int32 and error_word.is_cuda and error_word.numel() >= 1,
          "error_word must be a CUDA int32 tensor")
    return error_word.data_ptr()


def kv_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, slot_mapping: torch.Tensor,
              error_word: Optional[torch.Tensor] = None) -> None:
    """Write k_new/v_new [T, Hkv, D] into slots ``slot_mapping`` [T] (int64,
    negative = skip) of the paged caches, in place (pkv_kv_append)."""
    NB, Hkv, bs, D = _cache_args(k_cache, v_cache)
    T = k_new.shape[0]
    _need(k_new.shape == (T, Hkv, D) and v_new.shape == (T, Hkv, D), "k_new/v_new shape")
    _need(k_new.dtype == k_cache.dtype == v_new.dtype, "dtype mismatch")
    _need(k_new.is_contiguous() and v_new.is_contiguous(), "k_new/v_new must be contiguous")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.shape == (T,)
          and slot_mapping.is_cuda and slot_mapping.is_contiguous(), "slot_mapping int64 [T]")
    _check("pkv_kv_append", lib().pkv_kv_append(
        k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        slot_mapping.data_ptr(), T, Hkv, D, bs, NB, _DTYPE[k_cache.dtype],
        _err_ptr(error_word), _stream(k_cache)))


def _plan_dtype(dtype) -> int:
    """Plan/workspace element type: a torch dtype of q and cache, or
    torch.uint8 / "fp8" for an FP8 E4M3 cache."""
    if dtype in (torch.uint8, "fp8"):
        return PKV_FP8_E4M3
    return _DTYPE[dtype]


def plan(batch: int, num_queries: int, num_heads: int, num_kv_heads: int, head_dim: int,
         max_context_len: int, dtype: torch.dtype, block_size: int = 16, kernel: int = 0,
         split_blocks: int = 0, stages: int = 0) -> dict:
    """The launch an attention call with these sizes makes on the current device."""
    p = Plan()
    _check("pkv_attention_plan", lib().pkv_attention_plan(
        batch, num_queries, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
        _plan_dtype(dtype), _opts(kernel, split_blocks, stages), ctypes.byref(p)))
    return p.as_dict()


def plan_for(batch: int, num_queries: int, num_heads: int, num_kv_heads: int, head_dim: int,
             max_context_len: int, dtype: torch.dtype, num_sms: int, ctas_per_sm: int = 0,
             block_size: int = 16, kernel: int = 0, split_blocks: int = 0, stages: int = 0) -> dict:
    """The plan for a device with ``num_sms`` SMs (no GPU needed)."""
    p = Plan()
    _check("pkv_attention_plan_for", lib().pkv_attention_plan_for(
        batch, num_queries, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
        _plan_dtype(dtype), _opts(kernel, split_blocks, stages), num_sms, ctas_per_sm,
        ctypes.byref(p)))
    return p.as_dict()


def workspace_size(batch: int, num_queries: int, num_heads: int, num_kv_heads: int,
                   head_dim: int, max_context_len: int, dtype: torch.dtype,
                   block_size: int = 16, kernel: int = 0, split_blocks: int = 0, stages: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_attention_workspace_size", lib().pkv_attention_workspace_size(
        batch, num_queries, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
        _plan_dtype(dtype), _opts(kernel, split_blocks, stages), ctypes.byref(n)))
    return int(n.value)


def _attention(q, k_cache, v_cache, block_table, context_lens, scale, max_context_len, out,
               workspace, kernel, split_blocks, error_word, num_queries, stages=0):
    NB, Hkv, bs, D = _cache_args(k_cache, v_cache)
    B = q.shape[0]
    Hq = q.shape[-2]
    _need(q.shape[-1] == D and q.dtype == k_cache.dtype and q.is_cuda and q.is_contiguous(),
          "q must be a contiguous CUDA tensor of the cache dtype and head_dim")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2
          and block_table.shape[0] == B and block_table.is_contiguous() and block_table.is_cuda,
          "block_table must be a contiguous CUDA int32 [batch, max_blocks_per_seq]")
    _need(context_lens.dtype == torch.int32 and context_lens.shape == (B,)
          and context_lens.is_cuda and context_lens.is_contiguous(),
          "context_lens must be a contiguous CUDA int32 [batch]")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0  # device read
    if scale is None:
        scale = 0.0  # the library's default: 1/sqrt(head_dim)
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out")
    need = workspace_size(B, num_queries, Hq, Hkv, D, max_context_len, q.dtype, bs, kernel,
                          split_blocks, stages)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    L = lib()
    args_common = (out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                   block_table.data_ptr(), block_table.shape[1], context_lens.data_ptr(),
                   max_context_len, B)
    if num_queries == 1:
        st = L.pkv_paged_decode_attention(*args_common, Hq, Hkv, D, bs, NB, float(scale),
                                          _DTYPE[q.dtype], ws_ptr, ws_bytes,
                                          _opts(kernel, split_blocks, stages), _err_ptr(error_word),
                                          _stream(q))
        _check("pkv_paged_decode_attention", st)
    else:
        st = L.pkv_spec_verify_attention(*args_common, num_queries, Hq, Hkv, D, bs, NB,
                                         float(scale), _DTYPE[q.dtype], ws_ptr, ws_bytes,
                                         _opts(kernel, split_blocks, stages), _err_ptr(error_word),
                                         _stream(q))
        _check("pkv_spec_verify_attention", st)
    return out


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_table: torch.Tensor, context_lens: torch.Tensor,
                           scale: Optional[float] = None, max_context_len: Optional[int] = None,
                           out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, kernel: int = 0,
                           split_blocks: int = 0,
                           error_word: Optional[torch.Tensor] = None,
                           stages: int = 0) -> torch.Tensor:
    """Decode attention: q [B, Hq, D] -> out [B, Hq, D] over the paged cache
    (pkv_paged_decode_attention).  Pass ``max_context_len`` (a host bound of
    context_lens) to avoid a device read; pass ``workspace`` to avoid an
    allocation when the plan splits."""
    _need(q.dim() == 3, "q must be [batch, num_heads, head_dim]")
    return _attention(q, k_cache, v_cache, block_table, context_lens, scale, max_context_len,
                      out, workspace, kernel, split_blocks, error_word, 1, stages)


def spec_verify_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_table: torch.Tensor, context_lens: torch.Tensor,
                          scale: Optional[float] = None, max_context_len: Optional[int] = None,
                          out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, kernel: int = 0,
                          split_blocks: int = 0,
                          error_word: Optional[torch.Tensor] = None,
                          stages: int = 0) -> torch.Tensor:
    """Speculative verification: q [B, K+1, Hq, D] -> out of the same shape;
    query j sees rows <= L_b - (K+1) + j (pkv_spec_verify_attention)."""
    _need(q.dim() == 4, "q must be [batch, num_queries, num_heads, head_dim]")
    return _attention(q, k_cache, v_cache, block_table, context_lens, scale, max_context_len,
                      out, workspace, kernel, split_blocks, error_word, q.shape[1], stages)


def append_attention(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                     k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                     context_lens: torch.Tensor, scale: Optional[float] = None,
                     max_context_len: Optional[int] = None, out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, kernel: int = 0,
                     split_blocks: int = 0, error_word: Optional[torch.Tensor] = None,
                     stages: int = 0) -> torch.Tensor:
    """Write the new rows and attend in one launch (pkv_append_attention).

    q [B, Q, Hq, D] (or [B, Hq, D] for Q = 1); k_new / v_new [B, Q, Hkv, D]
    (or [B, Hkv, D]): row j of sequence b goes to position L_b - Q + j.
    Returns out with q's shape."""
    NB, Hkv, bs, D = _cache_args(k_cache, v_cache)
    q4 = q if q.dim() == 4 else q.unsqueeze(1)
    B, Q, Hq, _ = q4.shape
    kn = k_new if k_new.dim() == 4 else k_new.unsqueeze(1)
    vn = v_new if v_new.dim() == 4 else v_new.unsqueeze(1)
    _need(kn.shape == (B, Q, Hkv, D) and vn.shape == kn.shape, "k_new/v_new [B, Q, Hkv, D]")
    _need(kn.dtype == vn.dtype == q.dtype == k_cache.dtype, "dtype mismatch")
    _need(kn.is_contiguous() and vn.is_contiguous() and q.is_contiguous(), "contiguity")
    _need(q.shape[-1] == D and q.is_cuda, "q")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2
          and block_table.shape[0] == B and block_table.is_contiguous() and block_table.is_cuda,
          "block_table must be a contiguous CUDA int32 [batch, max_blocks_per_seq]")
    _need(context_lens.dtype == torch.int32 and context_lens.shape == (B,)
          and context_lens.is_cuda and context_lens.is_contiguous(), "context_lens")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0  # device read
    if scale is None:
        scale = 0.0  # the library's default: 1/sqrt(head_dim)
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out")
    need = workspace_size(B, Q, Hq, Hkv, D, max_context_len, q.dtype, bs, kernel, split_blocks,
                          stages)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pkv_append_attention", lib().pkv_append_attention(
        out.data_ptr(), q.data_ptr(), kn.data_ptr(), vn.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), block_table.data_ptr(), block_table.shape[1], context_lens.data_ptr(),
        max_context_len, B, Q, Hq, Hkv, D, bs, NB, float(scale), _DTYPE[q.dtype], ws_ptr,
        ws_bytes, _opts(kernel, split_blocks, stages), _err_ptr(error_word), _stream(q)))
    return out


def host_step_staging_size(batch: int, num_queries: int, num_heads: int, num_kv_heads: int,
                           head_dim: int, max_blocks_per_seq: int, max_context_len: int,
                           dtype: torch.dtype, block_size: int = 16, kernel: int = 0,
                           split_blocks: int = 0, stages: int = 0) -> int:
    """Device staging bytes of append_attention_host (pkv_host_step_staging_size)."""
    n = ctypes.c_size_t(0)
    _check("pkv_host_step_staging_size", lib().pkv_host_step_staging_size(
        batch, num_queries, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
        max_context_len, _DTYPE[dtype], _opts(kernel, split_blocks, stages), ctypes.byref(n)))
    return int(n.value)


def append_attention_host(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                          k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_table: torch.Tensor, context_lens: torch.Tensor,
                          out: torch.Tensor, staging: torch.Tensor, max_context_len: int,
                          scale: Optional[float] = None, kernel: int = 0, split_blocks: int = 0,
                          stages: int = 0, error_word: Optional[torch.Tensor] = None
                          ) -> torch.Tensor:
    """One step with host inputs and output (pkv_append_attention_host).

    q, k_new, v_new, block_table, context_lens and out are CPU tensors in the
    layouts of append_attention; the caches and ``staging`` (uint8,
    host_step_staging_size bytes) live on the GPU.  Pinned tensors are read
    (out: written) by the kernels in place; pageable ones go through
    ``staging``.  Everything is enqueued on the caches' current stream;
    ``out`` holds the result once that stream has been synchronised."""
    NB, Hkv, bs, D = _cache_args(k_cache, v_cache)
    q4 = q if q.dim() == 4 else q.unsqueeze(1)
    B, Q, Hq, _ = q4.shape
    host = (q, k_new, v_new, block_table, context_lens, out)
    _need(not any(t.is_cuda for t in host), "q, k_new, v_new, block_table, context_lens and "
          "out must be host tensors")
    _need(all(t.is_contiguous() for t in host), "contiguity")
    _need(k_new.numel() == B * Q * Hkv * D and v_new.numel() == k_new.numel(),
          "k_new/v_new [B, Q, Hkv, D]")
    _need(k_new.dtype == v_new.dtype == q.dtype == out.dtype == k_cache.dtype, "dtype mismatch")
    _need(q.shape[-1] == D and out.shape == q.shape, "q/out")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2
          and block_table.shape[0] == B, "block_table int32 [batch, max_blocks_per_seq]")
    _need(context_lens.dtype == torch.int32 and context_lens.shape == (B,), "context_lens")
    _need(staging.is_cuda and staging.device == k_cache.device, "staging must be on the caches' GPU")
    if scale is None:
        scale = 0.0  # the library's default: 1/sqrt(head_dim)
    _check("pkv_append_attention_host", lib().pkv_append_attention_host(
        out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), block_table.data_ptr(), block_table.shape[1],
        context_lens.data_ptr(), max_context_len, B, Q, Hq, Hkv, D, bs, NB, float(scale),
        _DTYPE[q.dtype], staging.data_ptr(), staging.numel() * staging.element_size(),
        _opts(kernel, split_blocks, stages), _err_ptr(error_word), _stream(k_cache)))
    return out


MLA_LATENT = 512


def _mla_opts(stages: int, split_blocks: int):
    if not (stages or split_blocks):
        return None
    return ctypes.byref(Options(0, split_blocks, stages, 0, 0, 0, 0, 0))


def mla_plan(batch: int, num_heads: int, rope_dim: int, max_context_len: int,
             dtype: torch.dtype, stages: int = 0, split_blocks: int = 0) -> dict:
    """The launch an MLA decode call with these sizes makes (pkv_mla_plan)."""
    p = Plan()
    _check("pkv_mla_plan", lib().pkv_mla_plan(
        batch, num_heads, MLA_LATENT, rope_dim, 16, max_context_len, _DTYPE[dtype],
        _mla_opts(stages, split_blocks), ctypes.byref(p)))
    return p.as_dict()


def mla_workspace_size(batch: int, num_heads: int, rope_dim: int, max_context_len: int,
                       dtype: torch.dtype, stages: int = 0, split_blocks: int = 0) -> int:
    """Split-K workspace bytes of mla_decode_attention (pkv_mla_workspace_size)."""
    n = ctypes.c_size_t(0)
    _check("pkv_mla_workspace_size", lib().pkv_mla_workspace_size(
        batch, num_heads, MLA_LATENT, rope_dim, 16, max_context_len, _DTYPE[dtype],
        _mla_opts(stages, split_blocks), ctypes.byref(n)))
    return int(n.value)


def mla_append(ckv_new: torch.Tensor, ckv_cache: torch.Tensor, slot_mapping: torch.Tensor,
               error_word: Optional[torch.Tensor] = None) -> None:
    """Write latent rows ckv_new [T, W] into slots ``slot_mapping`` [T] (int64,
    negative = skip) of the latent cache [NB, 16, W] (pkv_mla_append)."""
    _need(ckv_cache.is_cuda and ckv_cache.dim() == 3 and ckv_cache.is_contiguous(),
          "ckv_cache must be a contiguous CUDA [num_blocks, block_size, width] tensor")
    NB, bs, W = ckv_cache.shape
    T = ckv_new.shape[0]
    _need(ckv_new.shape == (T, W) and ckv_new.dtype == ckv_cache.dtype
          and ckv_new.is_contiguous(), "ckv_new [T, width] of the cache's dtype")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.shape == (T,)
          and slot_mapping.is_cuda and slot_mapping.is_contiguous(), "slot_mapping int64 [T]")
    _check("pkv_mla_append", lib().pkv_mla_append(
        ckv_new.data_ptr(), ckv_cache.data_ptr(), slot_mapping.data_ptr(), T, W, bs, NB,
        _DTYPE[ckv_cache.dtype], _err_ptr(error_word), _stream(ckv_cache)))


def mla_decode_attention(q: torch.Tensor, ckv_cache: torch.Tensor, block_table: torch.Tensor,
                         context_lens: torch.Tensor, scale: float,
                         max_context_len: Optional[int] = None,
                         out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, stages: int = 0,
                         split_blocks: int = 0,
                         error_word: Optional[torch.Tensor] = None) -> torch.Tensor:
    """MLA decode over the latent cache (pkv_mla_decode_attention).

    q [B, H, 512 + r] (the absorbed query of each head, r = 0 or 64);
    ckv_cache [NB, 16, 512 + r]; returns the latent output [B, H, 512]."""
    _need(ckv_cache.is_cuda and ckv_cache.dim() == 3 and ckv_cache.is_contiguous()
          and ckv_cache.dtype in _DTYPE, "ckv_cache must be a contiguous CUDA [NB, 16, W] tensor")
    NB, bs, W = ckv_cache.shape
    _need(q.is_cuda and q.dim() == 3 and q.shape[2] == W and q.dtype == ckv_cache.dtype
          and q.is_contiguous(), "q [B, H, width] of the cache's dtype")
    B, H, _ = q.shape
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2
          and block_table.shape[0] == B and block_table.is_contiguous() and block_table.is_cuda,
          "block_table must be a contiguous CUDA int32 [batch, max_blocks_per_seq]")
    _need(context_lens.dtype == torch.int32 and context_lens.shape == (B,)
          and context_lens.is_cuda and context_lens.is_contiguous(), "context_lens")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0  # device read
    rope = W - MLA_LATENT
    if out is None:
        out = torch.empty(B, H, MLA_LATENT, dtype=q.dtype, device=q.device)
    _need(out.shape == (B, H, MLA_LATENT) and out.dtype == q.dtype and out.is_contiguous(),
          "out [B, H, 512]")
    if B == 0:
        return out
    need = mla_workspace_size(B, H, rope, max_context_len, q.dtype, stages, split_blocks)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pkv_mla_decode_attention", lib().pkv_mla_decode_attention(
        out.data_ptr(), q.data_ptr(), ckv_cache.data_ptr(), block_table.data_ptr(),
        block_table.shape[1], context_lens.data_ptr(), max_context_len, B, H, MLA_LATENT, rope,
        bs, NB, float(scale), _DTYPE[q.dtype], ws_ptr, ws_bytes, _mla_opts(stages, split_blocks),
        _err_ptr(error_word), _stream(q)))
    return out


def tree_verify_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_table: torch.Tensor, context_lens: torch.Tensor,
                          tree_mask: torch.Tensor, scale: Optional[float] = None,
                          max_context_len: Optional[int] = None,
                          out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, kernel: int = 0,
                          split_blocks: int = 0, error_word: Optional[torch.Tensor] = None,
                          stages: int = 0) -> torch.Tensor:
    """Tree verification (pkv_tree_verify_attention): q [B, Q, Hq, D]; node j
    of sequence b sees the cached rows and tree row k iff bit k of
    tree_mask[b, j] (or tree_mask[j], shared) is set.  tree_mask: CUDA int64
    (the uint64 bit patterns), [Q] or [B, Q]."""
    NB, Hkv, bs, D = _cache_args(k_cache, v_cache)
    _need(q.dim() == 4 and q.is_cuda and q.is_contiguous() and q.dtype == k_cache.dtype
          and q.shape[-1] == D, "q must be [batch, num_queries, num_heads, head_dim]")
    B, Q, Hq, _ = q.shape
    _need(tree_mask.dtype == torch.int64 and tree_mask.is_cuda and tree_mask.is_contiguous()
          and tree_mask.shape in ((Q,), (B, Q)), "tree_mask: CUDA int64 [Q] or [B, Q]")
    stride = 0 if tree_mask.dim() == 1 else Q
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2
          and block_table.shape[0] == B and block_table.is_contiguous() and block_table.is_cuda,
          "block_table must be a contiguous CUDA int32 [batch, max_blocks_per_seq]")
    _need(context_lens.dtype == torch.int32 and context_lens.shape == (B,)
          and context_lens.is_cuda and context_lens.is_contiguous(), "context_lens")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0  # device read
    if scale is None:
        scale = 0.0  # the library's default: 1/sqrt(head_dim)
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out")
    need = workspace_size(B, Q, Hq, Hkv, D, max_context_len, q.dtype, bs, kernel, split_blocks,
                          stages)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pkv_tree_verify_attention", lib().pkv_tree_verify_attention(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_table.data_ptr(), block_table.shape[1], context_lens.data_ptr(), max_context_len,
        B, Q, Hq, Hkv, D, bs, NB, float(scale), _DTYPE[q.dtype], tree_mask.data_ptr(), stride,
        ws_ptr, ws_bytes, _opts(kernel, split_blocks, stages), _err_ptr(error_word),
        _stream(q)))
    return out


def _fp8_cache_args(k_cache, v_cache):
    _need(k_cache.is_cuda and v_cache.is_cuda and k_cache.dim() == 4
          and k_cache.shape == v_cache.shape and k_cache.dtype == torch.uint8
          and v_cache.dtype == torch.uint8 and k_cache.is_contiguous() and v_cache.is_contiguous(),
          "FP8 caches: contiguous CUDA uint8 [num_blocks, num_kv_heads, block_size, head_dim]")
    return k_cache.shape


def kv_append_fp8(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                  v_scale: float, error_word: Optional[torch.Tensor] = None) -> None:
    """Quantise k_new/v_new [T, Hkv, D] (float32/bf16/f16) to e4m3 codes in the
    uint8 caches at their slots (pkv_kv_append_fp8)."""
    NB, Hkv, bs, D = _fp8_cache_args(k_cache, v_cache)
    T = k_new.shape[0]
    _need(k_new.shape == (T, Hkv, D) and v_new.shape == (T, Hkv, D)
          and k_new.dtype == v_new.dtype and k_new.dtype in _DTYPE
          and k_new.is_contiguous() and v_new.is_contiguous(), "k_new/v_new [T, Hkv, D]")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.shape == (T,)
          and slot_mapping.is_cuda and slot_mapping.is_contiguous(), "slot_mapping int64 [T]")
    _check("pkv_kv_append_fp8", lib().pkv_kv_append_fp8(
        k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        slot_mapping.data_ptr(), T, Hkv, D, bs, NB, _DTYPE[k_new.dtype], float(k_scale),
        float(v_scale), _err_ptr(error_word), _stream(k_cache)))


def paged_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                        block_table: torch.Tensor, context_lens: torch.Tensor, k_scale: float,
                        v_scale: float, scale: Optional[float] = None,
                        max_context_len: Optional[int] = None,
                        out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, kernel: int = 0,
                        split_blocks: int = 0, error_word: Optional[torch.Tensor] = None,
                        stages: int = 0) -> torch.Tensor:
    """Decode (q [B, Hq, D]) or causal verification (q [B, Q, Hq, D]) over
    e4m3 caches (pkv_paged_attention_fp8); out has q's shape and type."""
    NB, Hkv, bs, D = _fp8_cache_args(k_cache, v_cache)
    q4 = q if q.dim() == 4 else q.unsqueeze(1)
    B, Q, Hq, _ = q4.shape
    _need(q.is_cuda and q.is_contiguous() and q.dtype in _DTYPE and q.shape[-1] == D, "q")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2
          and block_table.shape[0] == B and block_table.is_contiguous() and block_table.is_cuda,
          "block_table must be a contiguous CUDA int32 [batch, max_blocks_per_seq]")
    _need(context_lens.dtype == torch.int32 and context_lens.shape == (B,)
          and context_lens.is_cuda and context_lens.is_contiguous(), "context_lens")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0  # device read
    if scale is None:
        scale = 0.0  # the library's default: 1/sqrt(head_dim)
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out")
    n = ctypes.c_size_t(0)
    _check("pkv_attention_workspace_size", lib().pkv_attention_workspace_size(
        B, Q, Hq, Hkv, D, bs, max_context_len, PKV_FP8_E4M3, _opts(kernel, split_blocks, stages),
        ctypes.byref(n)))
    if n.value and workspace is None:
        workspace = torch.empty(n.value, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("pkv_paged_attention_fp8", lib().pkv_paged_attention_fp8(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_table.data_ptr(), block_table.shape[1], context_lens.data_ptr(), max_context_len,
        B, Q, Hq, Hkv, D, bs, NB, float(scale), _DTYPE[q.dtype], float(k_scale), float(v_scale),
        ws_ptr, ws_bytes, _opts(kernel, split_blocks, stages), _err_ptr(error_word), _stream(q)))
    return out


def read_error_word(error_word: torch.Tensor) -> int:
    """Synchronise the current stream and return the device error code."""
    code = ctypes.c_int32(0)
    _check("pkv_read_error_word", lib().pkv_read_error_word(
        error_word.data_ptr(), ctypes.byref(code), _stream(error_word)))
    return int(code.value)


# ---- block manager and copy-on-write ---------------------------------------
def _i32_array(values):
    import numpy as np
    a = np.ascontiguousarray(np.asarray(values, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def bm_hash(parent_hash: int, tokens) -> int:
    """Block hash of the prefix chain (pkv_bm_hash)."""
    a, ptr = _i32_array(tokens)
    return int(lib().pkv_bm_hash(ctypes.c_uint64(parent_hash), ptr, len(a)))


class BlockManager:
    """Physical blocks, reference counts, copy-on-write and the prefix hash
    chain of a paged KV cache (pkv_bm_*): host memory, not thread-safe."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self.block_size = block_size
        self.num_blocks = num_blocks
        self._h = lib().pkv_bm_create(num_blocks, block_size)
        if not self._h:
            raise PkvError("pkv_bm_create", 1, "bad size or out of memory")

    def close(self):
        if getattr(self, "_h", None):
            lib().pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def add_sequence(self, seq_id: int, tokens, prefix_cache: bool = True):
        """New sequence from a prompt -> (cached_tokens, slots of the rest)."""
        import numpy as np
        a, ptr = _i32_array(tokens)
        slots = np.zeros(max(len(a), 1), dtype=np.int64)
        cached = ctypes.c_int(0)
        _check("pkv_bm_add_sequence", lib().pkv_bm_add_sequence(
            self._h, seq_id, ptr, len(a), int(prefix_cache), ctypes.byref(cached),
            slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
        return cached.value, slots[:len(a) - cached.value].copy()

    def append(self, seq_id: int, tokens):
        """Append tokens -> (slots, [(cow_src, cow_dst)])."""
        import numpy as np
        a, ptr = _i32_array(tokens)
        slots = np.zeros(max(len(a), 1), dtype=np.int64)
        src, dst, n = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int(0)
        _check("pkv_bm_append", lib().pkv_bm_append(
            self._h, seq_id, ptr, len(a), slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            ctypes.byref(src), ctypes.byref(dst), ctypes.byref(n)))
        return slots[:len(a)].copy(), [(src.value, dst.value)] if n.value else []

    def fork(self, parent: int, child: int):
        _check("pkv_bm_fork", lib().pkv_bm_fork(self._h, parent, child))

    def free(self, seq_id: int):
        _check("pkv_bm_free", lib().pkv_bm_free(self._h, seq_id))

    def sequence(self, seq_id: int):
        """(block ids, token count) of a sequence."""
        nb, nt = ctypes.c_int(0), ctypes.c_int(0)
        _check("pkv_bm_sequence", lib().pkv_bm_sequence(self._h, seq_id, None, 0,
                                                         ctypes.byref(nb), ctypes.byref(nt)))
        buf = (ctypes.c_int32 * max(nb.value, 1))()
        _check("pkv_bm_sequence", lib().pkv_bm_sequence(self._h, seq_id, buf, nb.value,
                                                         ctypes.byref(nb), ctypes.byref(nt)))
        return list(buf[:nb.value]), nt.value

    def block_table(self, seq_ids, max_blocks: int = 0):
        """(block_table int32 [n, max_blocks], context_lens int32 [n])."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        if max_blocks <= 0:
            max_blocks = max([len(self.sequence(int(i))[0]) for i in ids] + [1])
        table = np.zeros((len(ids), max_blocks), dtype=np.int32)
        lens = np.zeros(len(ids), dtype=np.int32)
        _check("pkv_bm_block_table", lib().pkv_bm_block_table(
            self._h, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(ids),
            table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), max_blocks,
            lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return table, lens

    def stats(self) -> dict:
        f, c, n = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        _check("pkv_bm_stats", lib().pkv_bm_stats(self._h, ctypes.byref(f), ctypes.byref(c),
                                                  ctypes.byref(n)))
        return {"free": f.value, "cached": c.value, "sequences": n.value}

    def block_info(self, block: int):
        """(reference count, cached, hash) of one block."""
        r, c, h = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_uint64(0)
        _check("pkv_bm_block_info", lib().pkv_bm_block_info(self._h, block, ctypes.byref(r),
                                                            ctypes.byref(c), ctypes.byref(h)))
        return r.value, bool(c.value), h.value


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src, dst,
                error_word: Optional[torch.Tensor] = None) -> None:
    """Copy whole blocks src[i] -> dst[i] of both caches (pkv_copy_blocks)."""
    _need(k_cache.is_cuda and k_cache.is_contiguous() and v_cache.shape == k_cache.shape
          and v_cache.dtype == k_cache.dtype and v_cache.is_contiguous() and k_cache.dim() == 4,
          "k_cache / v_cache: contiguous CUDA [num_blocks, num_kv_heads, block_size, head_dim]")
    dev = k_cache.device
    src = torch.as_tensor(src, dtype=torch.int32, device=dev).contiguous()
    dst = torch.as_tensor(dst, dtype=torch.int32, device=dev).contiguous()
    _need(src.shape == dst.shape and src.dim() == 1, "src / dst: equal-length 1-D")
    NB, Hkv, bs, D = k_cache.shape
    dt = PKV_FP8_E4M3 if k_cache.dtype == torch.uint8 else _DTYPE[k_cache.dtype]
    _check("pkv_copy_blocks", lib().pkv_copy_blocks(
        k_cache.data_ptr(), v_cache.data_ptr(), src.data_ptr(), dst.data_ptr(), src.numel(),
        Hkv, D, bs, NB, dt, _err_ptr(error_word), _stream(k_cache)))


# ---- chunked prefill ------------------------------------------------------------
def paged_prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_table: torch.Tensor, context_lens: torch.Tensor,
                            query_start: torch.Tensor, max_query_len: Optional[int] = None,
                            scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                            stages: int = 0,
                            error_word: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Chunked prefill: q [total_q, Hq, D], the rows of sequence b being
    query_start[b] .. query_start[b + 1] - 1, whose K/V rows are already the
    last rows of its cache -> out of q's shape (pkv_paged_prefill_attention).
    Pass ``max_query_len`` (a host bound of the chunk lengths) to avoid a
    device read."""
    NB, Hkv, bs, D = _cache_args(k_cache, v_cache)
    _need(q.dim() == 3 and q.shape[-1] == D and q.dtype == k_cache.dtype and q.is_cuda
          and q.is_contiguous(), "q must be a contiguous CUDA [total_q, Hq, D] of the cache dtype")
    total_q, Hq = q.shape[0], q.shape[1]
    B = context_lens.shape[0]
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2
          and block_table.shape[0] == B and block_table.is_contiguous() and block_table.is_cuda,
          "block_table must be a contiguous CUDA int32 [batch, max_blocks_per_seq]")
    _need(context_lens.dtype == torch.int32 and context_lens.dim() == 1
          and context_lens.is_cuda and context_lens.is_contiguous(),
          "context_lens must be a contiguous CUDA int32 [batch]")
    _need(query_start.dtype == torch.int32 and query_start.shape == (B + 1,)
          and query_start.is_cuda and query_start.is_contiguous(),
          "query_start must be a contiguous CUDA int32 [batch + 1]")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max().item()) if B else 0
    if scale is None:
        scale = 0.0  # the library's default: 1/sqrt(head_dim)
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out")
    _check("pkv_paged_prefill_attention", lib().pkv_paged_prefill_attention(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_table.data_ptr(), block_table.shape[1], context_lens.data_ptr(),
        query_start.data_ptr(), int(max_query_len), B, total_q, Hq, Hkv, D, bs, NB,
        float(scale), _DTYPE[q.dtype], _opts(0, 0, stages), _err_ptr(error_word), _stream(q)))
    return out


def check_bounded_wait(error_word: torch.Tensor, limit_us: int,
                       waited_ns: Optional[torch.Tensor] = None) -> None:
    """Launch a bounded wait on a barrier nothing arrives on
    (pkv_check_bounded_wait): it gives up after limit_us and records
    PKV_DEVERR_TIMEOUT in error_word."""
    _need(error_word.dtype == torch.int32 and error_word.is_cuda, "error_word: CUDA int32")
    ptr = None
    if waited_ns is not None:
        _need(waited_ns.dtype == torch.int64 and waited_ns.is_cuda, "waited_ns: CUDA int64")
        ptr = waited_ns.data_ptr()
    _check("pkv_check_bounded_wait", lib().pkv_check_bounded_wait(
        error_word.data_ptr(), int(limit_us), ptr, _stream(error_word)))
