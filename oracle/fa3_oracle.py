"""CPU oracle for the FA3 per-head INT8 attention path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it.  It shares no code, tables or helpers with the
CUDA library; the two meet only in the seeded generators of ``workloads.py``.

Plain, slow and written to be checked by eye against the pages:

* msModelSlim, "FA3量化：Flash Attention 3激活量化算法说明", section 原理 /
  算法流程 -- step 1 (per-head collection), step 2 (Recall Window), step 3
  (cross-batch running min/max), step 4 (symmetric per-head scale).  Cited
  below as "FA3量化 算法流程 step k".
* MindIE, "FA3 quantization", Overview: for MLA only the non-RoPE part of K is
  quantized to 8 bits; the RoPE part of K stays in floating point.
* MindIE, "Attention Quantization", Overview, and MindIE Turbo "Attention量化":
  for GQA models q, k and v are all quantized to 8 bits; ``input_scale``
  quantizes, ``deq_scale`` dequantizes.

Precision: float64 throughout, except where a floating-point value decides an
integer (the INT8 code); there the decision is taken in IEEE float32, the
precision of the kernels (x / scale is one correctly rounded float32 division,
then round-half-to-even).  Readings of points the pages leave open:

* window width = sorted[i+t-1] - sorted[i] as an exact rational number (the
  pages do not fix the subtraction's precision; exact is the plain reading, and
  float64 alone is not exact once the two ends lie more than 45 binades apart),
  ties -> first (smallest) i;
* target_num = int(ratio * N) with the product in float64 and truncation, as
  in Python; clamped to at least 1; ratio must lie in (0, 1];
* -0.0 sorts before +0.0 (IEEE totalOrder), and min/max accumulation uses the
  same order;
* scale = 0 (an all-zero head) quantizes everything to code 0;
* decode attention attends to positions j < lens[b]; lens[b] = 0 gives a zero
  output row.

Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import Iterable, Optional, Tuple

import numpy as np

INT8_MAX = 127


# ---------------------------------------------------------------------------
# FA3量化 算法流程 step 2: Recall Window
# ---------------------------------------------------------------------------
def target_num(ratio: float, n: int) -> int:
    """target_num = int(ratio * N)  (FA3量化 算法流程 step 2), clamped to >= 1."""
    ratio = float(ratio)
    if not (0.0 < ratio <= 1.0):
        raise ValueError("ratio must lie in (0, 1]")
    if n <= 0:
        raise ValueError("a head needs at least one value")
    return max(1, int(ratio * float(n)))


def sort_total_order(values: np.ndarray) -> np.ndarray:
    """Ascending sort of float values; among the zeros, -0.0 comes before +0.0."""
    v = np.asarray(values, dtype=np.float64).ravel()
    if not np.all(np.isfinite(v)):
        raise ValueError("calibration values must be finite")
    s = np.sort(v)
    zeros = np.flatnonzero(s == 0.0)
    if zeros.size:
        n_neg = int(np.count_nonzero((v == 0.0) & np.signbit(v)))
        s[zeros[:n_neg]] = -0.0
        s[zeros[n_neg:]] = 0.0
    return s


def _first_exact_min(lo_vals: np.ndarray, hi_vals: np.ndarray) -> int:
    """Index of the first pair whose exact width hi - lo is smallest.

    Rounding to float64 is monotone, so the exact minimum lies among the pairs
    whose float64 width equals the smallest float64 width; those few are
    compared again as exact rationals (every float is a dyadic rational).
    """
    widths = hi_vals - lo_vals
    cand = np.flatnonzero(widths == widths.min())
    if cand.size == 1 or widths[cand[0]] == 0.0:   # a float64 zero width is exact
        return int(cand[0])
    exact = [Fraction(float(hi_vals[k])) - Fraction(float(lo_vals[k])) for k in cand]
    best = min(range(len(cand)), key=lambda j: (exact[j], j))
    return int(cand[best])


def recall_window(head_values: np.ndarray, ratio: float) -> Tuple[float, float]:
    """Narrowest window of the sorted head holding target_num values.

    FA3量化 算法流程 step 2: sort the N points, target_num = int(ratio*N), slide
    i = 0 .. N - target_num over [sorted[i], sorted[i+target_num-1]], keep the
    window of smallest length (exact length; the first i among equals); output
    (min_val, max_val).
    """
    s = sort_total_order(head_values)
    n = s.size
    t = target_num(ratio, n)
    i = _first_exact_min(s[: n - t + 1], s[t - 1:])   # window_length for i = 0 .. N - t
    return float(s[i]), float(s[i + t - 1])


def recall_window_bruteforce(head_values: np.ndarray, ratio: float) -> Tuple[float, float]:
    """Same answer by exhaustive search over value pairs, without any sort.

    Among all pairs (a, b) of data values with a <= b whose closed interval
    holds at least target_num values, the narrowest one (exact width, every
    candidate width compared as a rational), ties broken by the smallest a and
    then the smallest b.  O(N^2) memory.
    """
    v = np.asarray(head_values, dtype=np.float64).ravel()
    n = v.size
    t = target_num(ratio, n)
    le = np.count_nonzero(v[None, :] <= v[:, None], axis=1)   # #{x <= v[k]}
    lt = np.count_nonzero(v[None, :] < v[:, None], axis=1)    # #{x <  v[k]}
    a = v[:, None]
    b = v[None, :]
    count = le[None, :] - lt[:, None]                          # #{a <= x <= b}
    ok = (a <= b) & (count >= t)
    pairs = np.argwhere(ok)
    best = min(((Fraction(float(v[j])) - Fraction(float(v[i])), v[i], v[j]) for i, j in pairs))
    return float(best[1]), float(best[2])


# ---------------------------------------------------------------------------
# FA3量化 算法流程 steps 1 and 3: per-head collection, cross-batch accumulation
# ---------------------------------------------------------------------------
def _tot_less(a: float, b: float) -> bool:
    return a < b or (a == b and math.copysign(1.0, a) < 0 < math.copysign(1.0, b))


def calibrate_batch(x_bhsd: np.ndarray, ratio: float) -> Tuple[np.ndarray, np.ndarray]:
    """Per-head (min_val, max_val) of one batch x of shape (B, H, S, D).

    Step 1 regroups x per head: N = B*S*D points per head (the order inside a
    head does not matter to step 2).
    """
    x = np.asarray(x_bhsd)
    if x.ndim != 4:
        raise ValueError("x must be (B, H, S, D)")
    H = x.shape[1]
    lo = np.empty(H, np.float32)
    hi = np.empty(H, np.float32)
    for h in range(H):
        a, b = recall_window(x[:, h].reshape(-1), ratio)
        lo[h], hi[h] = a, b
    return lo, hi


def accumulate(min_io: np.ndarray, max_io: np.ndarray, cur_min: np.ndarray, cur_max: np.ndarray) -> None:
    """Step 3: min_values[h] = min(min_values[h], current_min[h]); max likewise."""
    for h in range(min_io.size):
        if _tot_less(float(cur_min[h]), float(min_io[h])):
            min_io[h] = cur_min[h]
        if _tot_less(float(max_io[h]), float(cur_max[h])):
            max_io[h] = cur_max[h]


def init_range(H: int) -> Tuple[np.ndarray, np.ndarray]:
    return np.full(H, np.inf, np.float32), np.full(H, -np.inf, np.float32)


def calibrate(batches: Iterable[np.ndarray], ratio: float,
              min_io: Optional[np.ndarray] = None, max_io: Optional[np.ndarray] = None):
    """Steps 1-3 over a sequence of calibration batches; returns (min, max) per head."""
    for x in batches:
        lo, hi = calibrate_batch(x, ratio)
        if min_io is None:
            min_io, max_io = init_range(lo.size)
        accumulate(min_io, max_io, lo, hi)
    return min_io, max_io


# ---------------------------------------------------------------------------
# FA3量化 算法流程 step 4: symmetric per-head quantization parameters
# ---------------------------------------------------------------------------
def qparams(min_v: np.ndarray, max_v: np.ndarray) -> np.ndarray:
    """abs_max[h] = max(|min[h]|, |max[h]|); scale[h] = abs_max[h] / 127.

    Computed in float64 and rounded once to float32 (equal to one correctly
    rounded float32 division, since float64 carries more than twice float32's
    precision).
    """
    mn = np.asarray(min_v, np.float64)
    mx = np.asarray(max_v, np.float64)
    return (np.maximum(np.abs(mn), np.abs(mx)) / 127.0).astype(np.float32)


# ---------------------------------------------------------------------------
# input_scale: activation -> INT8 code (symmetric, per head)
# ---------------------------------------------------------------------------
def quantize(x: np.ndarray, scale) -> np.ndarray:
    """q = clamp(round_half_even(x / scale), -127, 127); scale = 0 gives 0.

    ``scale`` broadcasts against ``x`` (one value per head).  The division is a
    float32 IEEE division; the rounding decision is taken on that float32.
    """
    x32 = np.asarray(x, np.float32)
    s32 = np.broadcast_to(np.asarray(scale, np.float32), x32.shape)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        r = np.divide(x32, s32, dtype=np.float32)
    r = np.where(s32 == 0, np.float32(0), r)
    r = np.clip(r, -INT8_MAX, INT8_MAX)
    return np.rint(r).astype(np.int8)


def quantize_append(kv: np.ndarray, scale: np.ndarray, cache: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Write quantize(kv[b, t, h, :], scale[h]) at cache[b, pos[b] + t, h, :].

    kv: [B][T_new][H][D] floats, cache: [B][T_max][H][D] int8 (copied, then
    returned).  A row whose destination falls outside the cache is an error.
    """
    out = np.array(cache, copy=True)
    B, T_new, H, D = kv.shape
    for b in range(B):
        p = int(pos[b])
        if p < 0 or p + T_new > out.shape[1]:
            raise ValueError("append position out of range")
        out[b, p:p + T_new] = quantize(kv[b], np.asarray(scale, np.float32)[None, :, None])
    return out


# ---------------------------------------------------------------------------
# Paged cache.  The pages leave the KV cache's storage to the serving runtime
# (MindIE, "FA3 quantization", usage steps: the runtime is told the cache's
# format); the library's paged calls take the block-table layout, defined here
# by the row map alone: token t of sequence b lives in pool page
# block_table[b][t // page_size], row t % page_size.
# ---------------------------------------------------------------------------
def gather_paged(pool: np.ndarray, block_table: np.ndarray, page_size: int, rows: np.ndarray) -> np.ndarray:
    """The contiguous cache [B][max_pages * page_size][...] that a page pool
    [num_pages][page_size][...] and block table [B][max_pages] describe, for the
    first rows[b] tokens of each sequence (later rows are left zero and no entry
    of the table past them is read).  A needed entry outside the pool is an error.
    """
    B, max_pages = block_table.shape
    out = np.zeros((B, max_pages * page_size) + pool.shape[2:], pool.dtype)
    for b in range(B):
        for t in range(int(rows[b])):
            page = int(block_table[b, t // page_size])
            if not 0 <= page < pool.shape[0]:
                raise ValueError("block table entry outside the pool")
            out[b, t] = pool[page, t % page_size]
    return out


def quantize_append_paged(kv: np.ndarray, scale: np.ndarray, pool: np.ndarray, block_table: np.ndarray,
                          pos: np.ndarray) -> np.ndarray:
    """quantize_append into a page pool: quantize(kv[b, t, h, :], scale[h]) goes
    to the pool row of token pos[b] + t of sequence b (pool copied, then
    returned).  Positions past max_pages * page_size, or a page outside the
    pool, are errors.
    """
    out = np.array(pool, copy=True)
    B, T_new, H, D = kv.shape
    page_size = pool.shape[1]
    for b in range(B):
        p = int(pos[b])
        if p < 0 or p + T_new > block_table.shape[1] * page_size:
            raise ValueError("append position out of range")
        for t in range(T_new):
            x = p + t
            page = int(block_table[b, x // page_size])
            if not 0 <= page < pool.shape[0]:
                raise ValueError("block table entry outside the pool")
            out[page, x % page_size] = quantize(kv[b, t], np.asarray(scale, np.float32)[:, None])
    return out


# ---------------------------------------------------------------------------
# Per-channel parameters: MindIE Turbo "Attention量化", 表1 / 表2 -- q/k/v_scale
# and q/k/v_offset of shape [head_num, head_dim].  The Recall Window of FA3量化
# 算法流程 steps 2-3 runs per (head, channel) over the B*S values of that channel.
# ---------------------------------------------------------------------------
def calibrate_channel_batch(x_bhsd: np.ndarray, ratio: float) -> Tuple[np.ndarray, np.ndarray]:
    """Per-(head, channel) (min_val, max_val) of one batch (B, H, S, D): step 2 on
    the N = B*S values x[:, h, :, d] of each channel."""
    x = np.asarray(x_bhsd)
    if x.ndim != 4:
        raise ValueError("x must be (B, H, S, D)")
    _, H, _, D = x.shape
    lo = np.empty((H, D), np.float32)
    hi = np.empty((H, D), np.float32)
    for h in range(H):
        for d in range(D):
            a, b = recall_window(x[:, h, :, d].reshape(-1), ratio)
            lo[h, d], hi[h, d] = a, b
    return lo, hi


def calibrate_channel(batches: Iterable[np.ndarray], ratio: float):
    """Steps 2-3 per (head, channel) over calibration batches; returns ([H][D], [H][D])."""
    mn = mx = None
    for x in batches:
        lo, hi = calibrate_channel_batch(x, ratio)
        if mn is None:
            mn, mx = init_range(lo.size)
            mn, mx = mn.reshape(lo.shape), mx.reshape(lo.shape)
        accumulate(mn.reshape(-1), mx.reshape(-1), lo.reshape(-1), hi.reshape(-1))
    return mn, mx


def qparams_channel(min_v: np.ndarray, max_v: np.ndarray, asymmetric: bool) -> Tuple[np.ndarray, np.ndarray]:
    """scale and offset per (head, channel), float32.

    Symmetric: step 4 per channel, scale = max(|min|, |max|) / 127, offset 0.
    Asymmetric (the pages give the offset tensor's shape, not its formula; the
    plain reading): the range is widened to contain 0, [lo, hi] = [min(min, 0),
    max(max, 0)], so that 0 stays exact, and mapped onto the codes -128 .. 127:
      scale  = (hi - lo) / 255                 (float32 subtraction, then division)
      offset = round_half_even(-lo / scale) - 128   (an integer; 0 when scale = 0)
    """
    mn = np.asarray(min_v, np.float32)
    mx = np.asarray(max_v, np.float32)
    if not asymmetric:
        return qparams(mn, mx), np.zeros(mn.shape, np.float32)
    lo = np.minimum(mn, np.float32(0))
    hi = np.maximum(mx, np.float32(0))
    width = np.subtract(hi, lo, dtype=np.float32)                                    # float32 IEEE subtraction
    scale = np.divide(width, np.float32(255), dtype=np.float32)                      # float32 IEEE division
    with np.errstate(divide="ignore", invalid="ignore"):
        z = np.divide(-lo, scale, dtype=np.float32)                                 # float32 IEEE division
    offset = np.where(scale == 0, np.float32(0), np.rint(z) - np.float32(128)).astype(np.float32)
    return scale, offset


def quantize_channel(x: np.ndarray, scale: np.ndarray, offset: np.ndarray, asymmetric: bool) -> np.ndarray:
    """Codes with per-channel parameters broadcast against x (..., D).

    Symmetric: q = clamp(round_half_even(x / scale), -127, 127).
    Asymmetric: q = clamp(round_half_even(x / scale) + offset, -128, 127).
    x / scale is one float32 division; scale = 0 gives code 0 (symmetric) or
    offset (asymmetric, where offset is then 0)."""
    if not asymmetric:
        return quantize(x, scale)
    x32 = np.asarray(x, np.float32)
    s32 = np.broadcast_to(np.asarray(scale, np.float32), x32.shape)
    o32 = np.broadcast_to(np.asarray(offset, np.float32), x32.shape)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        r = np.divide(x32, s32, dtype=np.float32)
    r = np.where(s32 == 0, np.float32(0), r)
    r = np.clip(r, -1e9, 1e9)                       # +-inf -> large finite before the integer step
    q = np.rint(r).astype(np.float64) + o32.astype(np.float64)
    return np.clip(q, -128, 127).astype(np.int8)


def dequantize_channel(q: np.ndarray, scale: np.ndarray, offset: np.ndarray) -> np.ndarray:
    """deq: (code - offset) * scale, float64."""
    return (np.asarray(q, np.float64) - np.asarray(offset, np.float64)) * np.asarray(scale, np.float64)


def gqa_decode_channel(q8: np.ndarray, k8: np.ndarray, v8: np.ndarray, qs: np.ndarray, qo: np.ndarray,
                       ks: np.ndarray, ko: np.ndarray, vs: np.ndarray, vo: np.ndarray, lens: np.ndarray,
                       softmax_scale: float) -> np.ndarray:
    """GQA decode on per-channel (asymmetric) INT8 q, k, v: every tensor is
    dequantized with its [heads][D] scale and offset, then plain attention.

    q8: [B][Hq][D] (qs, qo: [Hq][D]); k8, v8: [B][T][Hkv][D] (ks, ko, vs, vo: [Hkv][D]).
    Returns float64 [B][Hq][D]."""
    B, Hq, D = q8.shape
    Hkv = k8.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), np.float64)
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        for h in range(Hq):
            g = h // G
            qv = dequantize_channel(q8[b, h], qs[h], qo[h])
            kv = dequantize_channel(k8[b, :n, g], ks[g], ko[g])
            vv = dequantize_channel(v8[b, :n, g], vs[g], vo[g])
            out[b, h] = _softmax_weights((kv @ qv) * float(softmax_scale)) @ vv
    return out


def dequantize(q: np.ndarray, scale) -> np.ndarray:
    """deq_scale: code * scale, in float64."""
    return np.asarray(q, np.float64) * np.asarray(scale, np.float64)


# ---------------------------------------------------------------------------
# Decode attention over the INT8 cache
# ---------------------------------------------------------------------------
def _softmax_weights(s: np.ndarray) -> np.ndarray:
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    return p / p.sum(axis=-1, keepdims=True)


def mla_decode(q: np.ndarray, ckv8: np.ndarray, krope: np.ndarray, q_scale: np.ndarray,
               kv_scale: float, lens: np.ndarray, softmax_scale: float,
               rows: Optional[Iterable[Tuple[int, int]]] = None) -> np.ndarray:
    """Absorbed-MLA decode with an INT8 latent cache and a bf16 RoPE key.

    q: [B][H][Dl+Dr] (latent part first), ckv8: [B][T][Dl] int8 codes (the
    shared K-nope / V latent, one KV head, scale kv_scale), krope: [B][T][Dr].
    The latent query is quantized per head with the static q_scale[h]; the RoPE
    part of K is not quantized ("FA3 quantization", Overview).

      acc[h, j] = sum_c q8[h, c] * ckv8[j, c]                 (exact integer)
      s[h, j]   = (acc * q_scale[h] * kv_scale + q_rope[h] . k_rope[j]) * softmax_scale
      o[h, :]   = kv_scale * sum_j softmax(s[h, :])_j * ckv8[j, :]
    Returns float64 [B][H][Dl]; with ``rows`` = [(b, h), ...] only those rows
    are computed (the others stay 0).
    """
    B, H, _ = q.shape
    Dl = ckv8.shape[2]
    q = np.asarray(q, np.float32)
    q_scale = np.asarray(q_scale, np.float32)
    out = np.zeros((B, H, Dl), np.float64)
    want = None if rows is None else {}
    if rows is not None:
        for b, h in rows:
            want.setdefault(int(b), []).append(int(h))
    for b in range(B):
        n = int(lens[b])
        if n <= 0 or (want is not None and b not in want):
            continue
        hs = list(range(H)) if want is None else want[b]
        q8 = quantize(q[b, hs, :Dl], q_scale[hs, None]).astype(np.int64)
        qr = q[b, hs, Dl:].astype(np.float64)
        c = ckv8[b, :n].astype(np.int64)
        acc = q8 @ c.T                                             # [h][n] exact
        r = qr @ np.asarray(krope[b, :n], np.float64).T
        s = (acc.astype(np.float64) * (q_scale[hs].astype(np.float64)[:, None] * float(kv_scale)) + r) \
            * float(softmax_scale)
        p = _softmax_weights(s)
        out[b, hs] = float(kv_scale) * (p @ c.astype(np.float64))
    return out


def mla_decode_float(q: np.ndarray, ckv: np.ndarray, krope: np.ndarray, lens: np.ndarray,
                     softmax_scale: float) -> np.ndarray:
    """Same attention on the unquantized float latent (the quantization-error reference)."""
    B, H, _ = q.shape
    Dl = ckv.shape[2]
    out = np.zeros((B, H, Dl), np.float64)
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        k = np.concatenate([ckv[b, :n], krope[b, :n]], axis=1).astype(np.float64)
        s = (np.asarray(q[b], np.float64) @ k.T) * float(softmax_scale)
        out[b] = _softmax_weights(s) @ np.asarray(ckv[b, :n], np.float64)
    return out


def gqa_decode(q8: np.ndarray, k8: np.ndarray, v8: np.ndarray, q_scale: np.ndarray, k_scale: np.ndarray,
               v_scale: np.ndarray, lens: np.ndarray, softmax_scale: float) -> np.ndarray:
    """GQA decode with INT8 q, k, v and per-head scales.

    q8: [B][Hq][D], k8, v8: [B][T][Hkv][D]; query head h reads KV head
    g = h // (Hq // Hkv).
      s[h, j] = (q8[h] . k8[j, g]) * q_scale[h] * k_scale[g] * softmax_scale
      o[h]    = v_scale[g] * sum_j softmax(s[h])_j * v8[j, g]
    Returns float64 [B][Hq][D].
    """
    B, Hq, D = q8.shape
    Hkv = k8.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), np.float64)
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        for h in range(Hq):
            g = h // G
            kk = k8[b, :n, g].astype(np.int64)
            acc = kk @ q8[b, h].astype(np.int64)                    # [n] exact
            s = acc.astype(np.float64) * (float(q_scale[h]) * float(k_scale[g])) * float(softmax_scale)
            p = _softmax_weights(s)
            out[b, h] = float(v_scale[g]) * (p @ v8[b, :n, g].astype(np.float64))
    return out


def gqa_prefill(q8: np.ndarray, k8: np.ndarray, v8: np.ndarray, q_scale: np.ndarray, k_scale: np.ndarray,
                v_scale: np.ndarray, q_lens: np.ndarray, kv_lens: np.ndarray, softmax_scale: float,
                rows: Optional[Iterable[Tuple[int, int]]] = None) -> np.ndarray:
    """Prefill-phase attention with INT8 q, k, v (MindIE "Attention Quantization",
    Overview: q, k and v quantized to 8 bits), the same per-head scales as
    gqa_decode.  Reading where the pages are silent: the q_lens[b] new rows of
    sequence b are the last tokens of its kv_lens[b]-token context (a cached
    prefix of kv_lens - q_lens tokens, then the new rows), and new row i, at
    position kv_lens - q_lens + i, attends causally to positions 0 .. that
    position.

    q8: [B][S][Hq][D] (rows i >= q_lens[b] ignored), k8, v8: [B][T][Hkv][D].
    Returns float64 [B][S][Hq][D]; ignored rows are zero.  With ``rows`` =
    [(b, i), ...] only those rows (all heads) are computed.
    """
    B, S, Hq, D = q8.shape
    Hkv = k8.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    out = np.zeros((B, S, Hq, D), np.float64)
    want = None
    if rows is not None:
        want = {}
        for b, i in rows:
            want.setdefault(int(b), set()).add(int(i))
    for b in range(B):
        nq, nkv = int(q_lens[b]), int(kv_lens[b])
        if nq < 0 or nq > S or nkv < nq or nkv > k8.shape[1]:
            raise ValueError("bad q_lens / kv_lens")
        for i in range(nq):
            if want is not None and i not in want.get(b, ()):
                continue
            n = nkv - nq + i + 1                                   # keys 0 .. position of row i
            for h in range(Hq):
                g = h // G
                acc = k8[b, :n, g].astype(np.int64) @ q8[b, i, h].astype(np.int64)    # [n] exact
                s_ = acc.astype(np.float64) * (float(q_scale[h]) * float(k_scale[g])) * float(softmax_scale)
                p_ = _softmax_weights(s_)
                out[b, i, h] = float(v_scale[g]) * (p_ @ v8[b, :n, g].astype(np.float64))
    return out


def gqa_decode_float(q: np.ndarray, k: np.ndarray, v: np.ndarray, lens: np.ndarray,
                     softmax_scale: float) -> np.ndarray:
    """Same attention on unquantized float q, k, v (the quantization-error reference)."""
    B, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), np.float64)
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        for h in range(Hq):
            g = h // G
            s = (np.asarray(k[b, :n, g], np.float64) @ np.asarray(q[b, h], np.float64)) * float(softmax_scale)
            out[b, h] = _softmax_weights(s) @ np.asarray(v[b, :n, g], np.float64)
    return out
