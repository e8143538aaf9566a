"""Float64 CPU oracle for paged KV-cache decode attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(``paged_kv_cache_18_gb300``) never does, and the two share no code.

Two independent restatements of the same definition live here:

* ``paged_attention`` / ``kv_append`` (O1): plain C loops in float64
  (``pkv_oracle.c``) that walk the block table row by row and use the
  two-pass textbook softmax;
* ``twin.contiguous_attention`` (O2): NumPy float64 that first gathers each
  sequence's rows into a dense array, repeats the KV heads over the query
  group, and applies a dense masked softmax.

Both follow the attention equation of "Inference part 1" (brunomaga,
section "Why attention matters"), the paged layout of its section
"PagedAttention", the grouped-query head sharing of its section "Smaller KV
caches: MQA, GQA and MLA", and the shifted causal mask of its section "KV
cache".  Parity of every function here is pinned in ``tests/test_oracle_*``
against closed forms, library routines and the pages' printed numbers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2}


def compile_library(src: str, out: str) -> str:
    """gcc -O2 -fopenmp shared library from one C source file.

    FP contraction is switched off so that x86 and Arm hosts round alike.
    """
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``liboracle.so`` next to it."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_library(SOURCE, _LIB_PATH)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_storage(a: np.ndarray, dtype: str, name: str) -> None:
    want = np.float32 if dtype == "f32" else np.uint16
    if a.dtype != want or not a.flags["C_CONTIGUOUS"]:
        raise ValueError(f"{name}: expected C-contiguous {np.dtype(want).name}"
                         f" storage for dtype {dtype}, got {a.dtype}")


class Oracle:
    """ctypes view of one compiled copy of ``pkv_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_kv_append.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32,
                                         i32, i64, i32]
        lib.oracle_kv_append.restype = i32
        lib.oracle_paged_attention.argtypes = [
            vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64,
            ctypes.c_double, i32, vp, i64]
        lib.oracle_paged_attention.restype = i32
        lib.oracle_tree_attention.argtypes = [
            vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64,
            ctypes.c_double, i32, vp, i64]
        lib.oracle_tree_attention.restype = i32
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint
        lib.oracle_kv_append_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64,
                                             ctypes.c_float, ctypes.c_float]
        lib.oracle_kv_append_fp8.restype = i32
        lib.oracle_paged_attention_fp8.argtypes = [
            vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64,
            ctypes.c_double, i32, ctypes.c_double, ctypes.c_double]
        lib.oracle_paged_attention_fp8.restype = i32
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        self.lib = lib

    def num_threads(self) -> int:
        """Threads the C oracle's parallel loop uses on this host."""
        return int(self.lib.oracle_num_threads())

    def kv_append(self, k_cache, v_cache, k_new, v_new, slot_mapping,
                  dtype: str) -> None:
        """Write k_new/v_new [T, Hkv, D] into the host caches
        [NB, Hkv, bs, D] in place, slot by slot (negative slots skipped)."""
        for name, a in (("k_cache", k_cache), ("v_cache", v_cache),
                        ("k_new", k_new), ("v_new", v_new)):
            _check_storage(a, dtype, name)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        NB, Hkv, bs, D = k_cache.shape
        T = k_new.shape[0]
        if k_new.shape != (T, Hkv, D) or v_new.shape != (T, Hkv, D) or \
                v_cache.shape != k_cache.shape or slots.shape != (T,):
            raise ValueError("kv_append: inconsistent shapes")
        st = self.lib.oracle_kv_append(_ptr(k_cache), _ptr(v_cache),
                                       _ptr(k_new), _ptr(v_new), _ptr(slots),
                                       T, Hkv, D, bs, NB, DTYPE_CODES[dtype])
        if st != 0:
            raise ValueError(f"oracle_kv_append failed with code {st}")

    def paged_attention(self, q, k_cache, v_cache, block_table, context_lens,
                        scale: float, dtype: str, rows=None) -> np.ndarray:
        """Float64 attention output [B, Q, Hq, D] (NaN where not computed).

        q: [B, Q, Hq, D] (or [B, Hq, D] for Q = 1); caches [NB, Hkv, bs, D];
        block_table [B, max_blocks] int32; context_lens [B] int32.  ``rows``
        optionally restricts the work to flat output rows ((b*Q + j)*Hq + h).
        """
        if q.ndim == 3:
            q = q[:, None]
        q = np.ascontiguousarray(q)
        _check_storage(q, dtype, "q")
        _check_storage(k_cache, dtype, "k_cache")
        _check_storage(v_cache, dtype, "v_cache")
        B, Q, Hq, D = q.shape
        NB, Hkv, bs, D2 = k_cache.shape
        if D2 != D or v_cache.shape != k_cache.shape:
            raise ValueError("paged_attention: inconsistent shapes")
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        if table.ndim != 2 or table.shape[0] != B or lens.shape != (B,):
            raise ValueError("paged_attention: bad block_table/context_lens")
        out = np.full((B, Q, Hq, D), np.nan, dtype=np.float64)
        if rows is None:
            n_rows, rows_ptr = 0, None
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            n_rows, rows_ptr = rows_arr.size, _ptr(rows_arr)
        st = self.lib.oracle_paged_attention(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(table),
            table.shape[1], _ptr(lens), B, Q, Hq, Hkv, D, bs, NB, float(scale),
            DTYPE_CODES[dtype], rows_ptr, n_rows)
        if st != 0:
            raise ValueError(f"oracle_paged_attention failed with code {st}")
        return out


    def tree_attention(self, q, k_cache, v_cache, block_table, context_lens,
                       scale: float, dtype: str, tree_mask) -> np.ndarray:
        """Float64 output [B, Q, Hq, D] of tree verification: node j of
        sequence b sees the cached rows and the tree rows whose bits are set
        in tree_mask [B, Q] (or [Q], shared by every sequence) uint64."""
        q = np.ascontiguousarray(q)
        _check_storage(q, dtype, "q")
        _check_storage(k_cache, dtype, "k_cache")
        _check_storage(v_cache, dtype, "v_cache")
        B, Q, Hq, D = q.shape
        NB, Hkv, bs, _ = k_cache.shape
        mask = np.ascontiguousarray(tree_mask, dtype=np.uint64)
        stride = 0 if mask.ndim == 1 else Q
        if mask.shape not in ((Q,), (B, Q)):
            raise ValueError("tree_mask must be [Q] or [B, Q]")
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.full((B, Q, Hq, D), np.nan, dtype=np.float64)
        st = self.lib.oracle_tree_attention(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(table),
            table.shape[1], _ptr(lens), B, Q, Hq, Hkv, D, bs, NB, float(scale),
            DTYPE_CODES[dtype], _ptr(mask), stride)
        if st != 0:
            raise ValueError(f"oracle_tree_attention failed with code {st}")
        return out


    # ---- FP8 E4M3 cache -------------------------------------------------
    def e4m3_value(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_value(int(code)))

    def e4m3_encode(self, x: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(x)))

    def kv_append_fp8(self, k_cache, v_cache, k_new, v_new, slot_mapping, src_dtype: str,
                      k_scale: float, v_scale: float) -> None:
        """Quantise k_new/v_new [T, Hkv, D] (storage of src_dtype) into the
        e4m3 byte caches [NB, Hkv, bs, D] at their slots."""
        from .twin import widen
        for name, a in (("k_cache", k_cache), ("v_cache", v_cache)):
            if a.dtype != np.uint8 or not a.flags["C_CONTIGUOUS"]:
                raise ValueError(f"{name}: expected C-contiguous uint8 codes")
        kf = np.ascontiguousarray(widen(k_new, src_dtype).astype(np.float32))
        vf = np.ascontiguousarray(widen(v_new, src_dtype).astype(np.float32))
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        NB, Hkv, bs, D = k_cache.shape
        st = self.lib.oracle_kv_append_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(kf), _ptr(vf),
                                           _ptr(slots), kf.shape[0], Hkv, D, bs, NB,
                                           float(k_scale), float(v_scale))
        if st != 0:
            raise ValueError(f"oracle_kv_append_fp8 failed with code {st}")

    def paged_attention_fp8(self, q, k_cache, v_cache, block_table, context_lens,
                            scale: float, q_dtype: str, k_scale: float,
                            v_scale: float) -> np.ndarray:
        """Float64 attention [B, Q, Hq, D] over e4m3 byte caches."""
        if q.ndim == 3:
            q = q[:, None]
        q = np.ascontiguousarray(q)
        _check_storage(q, q_dtype, "q")
        B, Q, Hq, D = q.shape
        NB, Hkv, bs, _ = k_cache.shape
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.full((B, Q, Hq, D), np.nan, dtype=np.float64)
        st = self.lib.oracle_paged_attention_fp8(
            _ptr(out), _ptr(q), _ptr(np.ascontiguousarray(k_cache)),
            _ptr(np.ascontiguousarray(v_cache)), _ptr(table), table.shape[1], _ptr(lens), B, Q,
            Hq, Hkv, D, bs, NB, float(scale), DTYPE_CODES[q_dtype], float(k_scale),
            float(v_scale))
        if st != 0:
            raise ValueError(f"oracle_paged_attention_fp8 failed with code {st}")
        return out


def default() -> Oracle:
    """The oracle built from ``pkv_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def num_threads() -> int:
    return default().num_threads()


def kv_append(*args, **kwargs) -> None:
    default().kv_append(*args, **kwargs)


def paged_attention(*args, **kwargs) -> np.ndarray:
    return default().paged_attention(*args, **kwargs)


def tree_attention(*args, **kwargs) -> np.ndarray:
    return default().tree_attention(*args, **kwargs)


def kv_append_fp8(*args, **kwargs) -> None:
    default().kv_append_fp8(*args, **kwargs)


def paged_attention_fp8(*args, **kwargs) -> np.ndarray:
    return default().paged_attention_fp8(*args, **kwargs)
