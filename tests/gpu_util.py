"""Helpers of the GPU parity tests: move a seeded batch to the device, run one
step (append, then attention) through the C ABI, and compare with the
float64 oracle."""
import contextlib

import numpy as np
import torch

import oracle
import paged_kv_cache_18_gb300 as pkv
from paged_kv_cache_18_gb300 import workloads as W

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}

# Tolerances against the float64 oracle.  bf16/f16: the stated bound of the
# task (max-abs 1e-2, relative L2 2e-3).  f32: an arithmetic bound, see the
# design notes (float32 dot products, ex2.approx and one rounding of the
# output give relative errors of a few 1e-7; the bound leaves a margin of
# about 10x and stays below the 1e-6-scale error the pages print for float32
# attention over 2048 rows only in the max-abs sense).
TOL = {"bf16": (1e-2, 2e-3), "f16": (1e-2, 2e-3), "f32": (1e-5, 2e-6)}


def dev_tensor(a: np.ndarray, dtype: str, device) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(TORCH_DT[dtype])
    return torch.from_numpy(a).to(device)


def host_f64(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return t.float().cpu().numpy().astype(np.float64)
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return W.storage_to_f64(bits, dtype)


def cache_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.float32:
        return t.cpu().numpy().view(np.uint32)
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceBatch:
    def __init__(self, b: W.PagedBatch, device="cuda:0"):
        dt = b.wl.dtype
        self.b = b
        self.k_cache = dev_tensor(b.k_cache, dt, device)
        self.v_cache = dev_tensor(b.v_cache, dt, device)
        self.k_new = dev_tensor(b.k_new, dt, device)
        self.v_new = dev_tensor(b.v_new, dt, device)
        self.q = dev_tensor(b.q, dt, device)
        self.slots = torch.from_numpy(b.slot_mapping).to(device)
        self.table = torch.from_numpy(b.block_table).to(device)
        self.lens = torch.from_numpy(b.context_lens).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def append(self):
        pkv.kv_append(self.k_new, self.v_new, self.k_cache, self.v_cache, self.slots,
                      error_word=self.err)

    def attend(self, kernel=0, split_blocks=0, out=None, workspace=None, stages=0):
        wl = self.b.wl
        if wl.num_queries == 1:
            o = pkv.paged_decode_attention(self.q[:, 0], self.k_cache, self.v_cache, self.table,
                                           self.lens, scale=wl.softmax_scale,
                                           max_context_len=self.b.max_context_len, out=out,
                                           workspace=workspace, kernel=kernel,
                                           split_blocks=split_blocks, error_word=self.err,
                                           stages=stages)
            return o[:, None]
        return pkv.spec_verify_attention(self.q, self.k_cache, self.v_cache, self.table,
                                         self.lens, scale=wl.softmax_scale,
                                         max_context_len=self.b.max_context_len, out=out,
                                         workspace=workspace, kernel=kernel,
                                         split_blocks=split_blocks, error_word=self.err,
                                         stages=stages)


def oracle_after_append(b: W.PagedBatch, rows=None) -> np.ndarray:
    """Append on the host mirror (once) and return the oracle output."""
    if not getattr(b, "_appended", False):
        oracle.kv_append(b.k_cache, b.v_cache, b.k_new, b.v_new, b.slot_mapping, b.wl.dtype)
        b._appended = True
    return oracle.paged_attention(b.q, b.k_cache, b.v_cache, b.block_table, b.context_lens,
                                  b.wl.softmax_scale, b.wl.dtype, rows=rows)


def errors(got: np.ndarray, ref: np.ndarray):
    mask = ~np.isnan(ref)
    d = got[mask] - ref[mask]
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    denom = float(np.linalg.norm(ref[mask]))
    rel = float(np.linalg.norm(d) / denom) if denom > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what=""):
    """The stated bound per element, max-abs tol_abs, except where the output
    type cannot hold it: a bf16 output of |ref| >= 4 is already up to half an
    ulp (2^-6 = 0.0156 > 1e-2) from the exact value when correctly rounded
    (for example 4.07614 -> 4.0625), so there the bound is that half ulp plus
    1e-3 of arithmetic error (below 4, half an ulp is at most 2^-8 and the
    bound stays 1e-2).  Relative L2 over all elements: tol_rel."""
    mask = ~np.isnan(ref)
    assert np.isfinite(got[mask]).all(), f"{what}: non-finite output"
    max_abs, rel = errors(got, ref)
    tol_abs, tol_rel = TOL[dtype]
    d = np.abs(got[mask] - ref[mask])
    bound = np.full(d.shape, tol_abs)
    if dtype != "f32":
        bound = np.maximum(bound, half_ulp(ref[mask], dtype) + 1e-3)
    worst = float((d - bound).max()) if d.size else 0.0
    assert worst <= 0 and rel <= tol_rel, \
        (f"{what}: max-abs {max_abs:.3e} (tol {tol_abs}, or half an output ulp + 1e-3 where "
         f"that is larger), rel-L2 {rel:.3e} (tol {tol_rel})")
    return max_abs, rel


# Output rounding of each type: half a unit in the last place at |x|.
_MANT_BITS = {"bf16": 7, "f16": 10, "f32": 23}
_MIN_EXP = {"bf16": -126, "f16": -14, "f32": -126}


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    e = np.floor(np.log2(np.maximum(np.abs(x), np.finfo(np.float64).tiny)))
    e = np.maximum(e, _MIN_EXP[dtype])
    return np.ldexp(1.0, (e - _MANT_BITS[dtype] - 1).astype(np.int64))


# FP8 caches: an output element is a weighted mean of code * v_scale values,
# which the output type does not hold exactly (a 16-bit V cache gives outputs
# that are often V elements themselves), so the element bound is the output
# rounding plus the arithmetic's own error: for 16-bit q, the f16 rounding
# of the softmax weights (2^-11 relative, at most 2^-11 * max|v| ~ 3.7e-3 for
# |v| <= 448 * 0.0171); float32 q keeps the float32 bound.  The relative L2
# bound stays the stated one.
FP8_EXTRA = {"bf16": 4e-3, "f16": 4e-3, "f32": 1e-5}


def assert_close_fp8(got: np.ndarray, ref: np.ndarray, dtype: str, what=""):
    mask = ~np.isnan(ref)
    assert np.isfinite(got[mask]).all(), f"{what}: non-finite output"
    d = np.abs(got[mask] - ref[mask])
    excess = d - half_ulp(ref[mask], dtype)
    worst = float(excess.max()) if d.size else 0.0
    _, rel = errors(got, ref)
    tol_rel = TOL[dtype][1]
    assert worst <= FP8_EXTRA[dtype] and rel <= tol_rel, \
        (f"{what}: max (|err| - half ulp) {worst:.3e} (tol {FP8_EXTRA[dtype]}), "
         f"rel-L2 {rel:.3e} (tol {tol_rel})")
    return float(d.max()) if d.size else 0.0, rel


@contextlib.contextmanager
def tuning(**kw):
    """Pass extra launch controls (pkv_options fields) to every binding call
    inside the block."""
    saved = dict(pkv.binding.TUNING)
    pkv.binding.TUNING.update(kw)
    try:
        yield
    finally:
        pkv.binding.TUNING.clear()
        pkv.binding.TUNING.update(saved)
