"""Shared test helpers: library loading, tensor upload, attention tolerance checks."""
import os
import re

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Attention gates: max |gpu - oracle| <= 1e-2 and relative RMS <= 2e-3.  For a bf16
# output the final rounding adds at most half a bf16 ulp of the value, which the
# max-abs gate allows on top of 1e-2 (the gate applies to the arithmetic before the
# output cast).  This is the one definition of the gate: the parity tests and the
# smoke run both call assert_attn_close, which also reports the rounding floor of a
# bf16 output, max |bf16(ref) - ref|, beside the errors.
ATOL = 1e-2
RRMS = 2e-3


def header_functions():
    src = open(os.path.join(ROOT, "include", "fa3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa3_[a-z0-9_]+)\s*\(", src)))


def fa3():
    from int8_head_kv_gb300 import build, fa3 as F
    build()
    return F


def bf16_dev(x: np.ndarray) -> torch.Tensor:
    from workloads import bf16_tensor
    return bf16_tensor(x).cuda()


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    _, e = np.frexp(np.abs(x))
    return np.where(x == 0, 0.0, np.ldexp(1.0, e - 9))


def attn_errors(gpu: np.ndarray, ref: np.ndarray, bf16_out: bool = False):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.abs(gpu - ref)
    slack = half_ulp_bf16(ref) if bf16_out else 0.0
    max_abs = float(np.max(diff - slack)) if diff.size else 0.0
    denom = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    rrms = float(np.sqrt(np.mean((gpu - ref) ** 2)) / denom) if denom > 0 else float(np.sqrt(np.mean(gpu ** 2)))
    return max_abs, rrms


def bf16_floor(ref: np.ndarray) -> float:
    """max |bf16(ref) - ref|: the error a bf16 output has even when its arithmetic is exact."""
    import torch as _t
    r = np.asarray(ref, np.float64)
    if r.size == 0:
        return 0.0
    rb = _t.from_numpy(r).to(_t.bfloat16).to(_t.float64).numpy()
    return float(np.max(np.abs(rb - r)))


def assert_attn_close(gpu, ref, bf16_out=False, what=""):
    max_abs, rrms = attn_errors(gpu, ref, bf16_out)
    floor = f", bf16 rounding floor {bf16_floor(ref):.3e}" if bf16_out else ""
    print(f"{what}: max abs error {max_abs:.3e}{' (after the half-ulp output rounding)' if bf16_out else ''}, "
          f"relative RMS {rrms:.3e}{floor}")
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    assert max_abs <= ATOL, f"{what}: max abs error {max_abs:.3e} > {ATOL}{floor}"
    assert rrms <= RRMS, f"{what}: relative RMS {rrms:.3e} > {RRMS}{floor}"
    return max_abs, rrms


def paged_layout(cache: np.ndarray, page_size: int, spare: int, rng) -> tuple:
    """A page pool and block table holding `cache` [B][T][...]: each sequence's
    rows are cut into pages of page_size (the last one zero-padded) and the pages
    are stored in a random order among `spare` extra pages of noise."""
    B, T = cache.shape[:2]
    mp = -(-T // page_size)
    padded = np.zeros((B, mp * page_size) + cache.shape[2:], cache.dtype)
    padded[:, :T] = cache
    n = B * mp + spare
    perm = rng.permutation(n)
    pool = (rng.standard_normal((n, page_size) + cache.shape[2:]) * 3).astype(cache.dtype)
    pool[perm[:B * mp]] = padded.reshape((B * mp, page_size) + cache.shape[2:])
    return pool, perm[:B * mp].reshape(B, mp).astype(np.int32)
