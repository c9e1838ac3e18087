"""Seeded synthetic workloads for the FA3 per-head INT8 attention path.

This module only draws random numbers and casts them to bf16; it holds none
of the method's arithmetic (no sorting, windowing, scaling, quantization or
attention).  Both the CPU oracle tests and the GPU path use it, so the two
sides always see identical inputs.

Recipe (shared by every workload below):
  * generator: ``numpy.random.default_rng([seed, tag, k, ...])``: every tensor
    (and every calibration batch k, and every head of the large calibration
    workload) has its own stream, so any piece can be regenerated alone;
  * log-uniform sigma: ``exp(U(ln a, ln b))``, one draw per head;
  * "outliers x m at rate p": each position independently, with probability p,
    is multiplied by m (Bernoulli mask);
  * every activation is rounded to bf16 (round-to-nearest-even) before use,
    and kept here as float32 arrays whose values are exactly bf16.

The shapes and distributions stand in for the pages' real-model activations
(DeepSeek-V3/R1 absorbed MLA, Llama-3.1-70B GQA) and their BoolQ calibration
text, neither of which is available; only shapes and value laws are imitated.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

# Stream tags so that every tensor of a workload has its own random stream.
TAG_Q, TAG_CKV, TAG_KROPE, TAG_K, TAG_V, TAG_LENS, TAG_SIGMA, TAG_CALIB_Q, TAG_CALIB_KV, \
    TAG_CALIB_K, TAG_CALIB_V, TAG_POS, TAG_APPEND, TAG_PREFILL = range(14)


def rng_for(seed: int, tag: int, k: int = 0, *more: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tag), int(k)] + [int(m) for m in more])


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def bf16_tensor(x: np.ndarray) -> torch.Tensor:
    """bf16 CPU tensor holding the bf16-exact float32 values of ``x``."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    out = t.to(torch.bfloat16)
    if not torch.equal(out.to(torch.float32), t):
        raise ValueError("values are not bf16-exact")
    return out


def log_uniform(rng: np.random.Generator, lo: float, hi: float, size) -> np.ndarray:
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=size))


def with_outliers(rng: np.random.Generator, x: np.ndarray, rate: float, mult: float) -> np.ndarray:
    if rate <= 0:
        return x
    mask = rng.random(x.shape, dtype=np.float32) < rate
    return np.where(mask, x * np.float32(mult), x).astype(np.float32)


def normal(rng, shape, sigma) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.asarray(sigma, np.float32)).astype(np.float32)


def student_t(rng, shape, nu, sigma) -> np.ndarray:
    return (rng.standard_t(nu, size=shape).astype(np.float32) * np.asarray(sigma, np.float32)).astype(np.float32)


def mixed_magnitude_head(rng: np.random.Generator, n: int) -> np.ndarray:
    """A calibration head whose values span about 130 binades: integers in [-3, 3]
    (many windows of equal integer length), 15 % of them replaced by values of
    magnitude 2^-133 .. 2^-100, so that window lengths differ only far below
    float64's precision.  bf16-exact float32 [n]."""
    v = rng.integers(-3, 4, n).astype(np.float64)
    tiny = np.ldexp(rng.integers(1, 256, n).astype(np.float64), rng.integers(-133, -107, n))
    v = np.where(rng.random(n) < 0.15, np.where(rng.random(n) < 0.5, -tiny, tiny), v)
    return bf16_round(v.astype(np.float32))


# ----------------------------------------------------------------------------
# Absorbed-MLA decode workloads
# ----------------------------------------------------------------------------
@dataclass
class MLAWorkload:
    name: str
    B: int
    H: int
    Dl: int
    Dr: int
    T_max: int
    softmax_scale: float
    lens: Optional[Sequence[int]] = None        # fixed lengths, or None -> drawn
    lens_range: Optional[Tuple[int, int]] = None  # inclusive uniform range for drawn lengths
    ckv_sigma: Tuple[float, float] = (0.1, 10.0)  # log-uniform law of the latent sigma
    ckv_outlier_rate: float = 1e-3
    ckv_outlier_mult: float = 20.0
    calib_batches: int = 3
    calib_q_shape: Tuple[int, int, int, int] = (2, 4, 128, 64)     # (B, H, S, D) per batch
    calib_q_sigma: Optional[Tuple[float, float]] = None  # per-head log-uniform law, None -> N(0,1)
    calib_kv_shape: Tuple[int, int, int, int] = (2, 1, 128, 64)
    ratio: float = 0.9999
    seed: int = 0


def mla_tiny() -> MLAWorkload:
    """Tiny MLA decode + calibration (batch 2, 4 heads, latent 64, RoPE 16, lens 37/128)."""
    return MLAWorkload(name="tiny-mla b2 h4 dl64 dr16 lens[37,128]", B=2, H=4, Dl=64, Dr=16, T_max=128,
                       softmax_scale=1.0 / math.sqrt(80.0), lens=[37, 128],
                       calib_q_shape=(2, 4, 128, 64), calib_q_sigma=(0.1, 10.0),
                       calib_kv_shape=(2, 1, 128, 64))


def mla_dsv3(B: int = 32, T: int = 8192, lens: Optional[Sequence[int]] = None) -> MLAWorkload:
    """DeepSeek-V3-shaped absorbed MLA decode (128 heads, latent 512 INT8, RoPE 64 bf16)."""
    return MLAWorkload(name=f"dsv3-mla b{B} h128 dl512 dr64 ctx{T}", B=B, H=128, Dl=512, Dr=64, T_max=T,
                       softmax_scale=1.0 / math.sqrt(192.0), lens=list(lens) if lens is not None else [T] * B,
                       calib_q_shape=(32, 128, 1, 512), calib_q_sigma=None,
                       calib_kv_shape=(1, 1, 8192, 512))


def mla_long(B: int = 8, lo: int = 1024, hi: int = 32768) -> MLAWorkload:
    """Long-context MLA decode with seeded variable lengths and 0.01% x50 outliers."""
    return MLAWorkload(name=f"long-mla b{B} h128 dl512 dr64 ctx U[{lo},{hi}]", B=B, H=128, Dl=512, Dr=64,
                       T_max=hi, softmax_scale=1.0 / math.sqrt(192.0), lens=None, lens_range=(lo, hi),
                       ckv_outlier_rate=1e-4, ckv_outlier_mult=50.0,
                       calib_q_shape=(8, 128, 1, 512), calib_q_sigma=None,
                       calib_kv_shape=(1, 1, 8192, 512))


@dataclass
class MLAInputs:
    q: np.ndarray        # [B][H][Dl+Dr] bf16-exact float32, latent first then RoPE
    ckv: np.ndarray      # [B][T_max][Dl] unquantized latent (bf16-exact float32)
    krope: np.ndarray    # [B][T_max][Dr] bf16-exact float32
    lens: np.ndarray     # [B] int32
    calib_q: List[np.ndarray]   # calibration batches (B, H, S, Dl) for the per-head query scale
    calib_kv: List[np.ndarray]  # calibration batches (B, 1, S, Dl) for the latent cache scale


def mla_lens(w: MLAWorkload) -> np.ndarray:
    if w.lens is not None:
        return np.asarray(w.lens, dtype=np.int32)
    lo, hi = w.lens_range
    return rng_for(w.seed, TAG_LENS).integers(lo, hi + 1, size=w.B).astype(np.int32)


def mla_inputs(w: MLAWorkload, with_calib: bool = True) -> MLAInputs:
    s = w.seed
    sig_kv = float(log_uniform(rng_for(s, TAG_SIGMA), *w.ckv_sigma, size=1)[0])
    q = bf16_round(normal(rng_for(s, TAG_Q), (w.B, w.H, w.Dl + w.Dr), 1.0))
    r = rng_for(s, TAG_CKV)
    ckv = with_outliers(r, normal(r, (w.B, w.T_max, w.Dl), sig_kv), w.ckv_outlier_rate, w.ckv_outlier_mult)
    ckv = bf16_round(ckv)
    krope = bf16_round(normal(rng_for(s, TAG_KROPE), (w.B, w.T_max, w.Dr), 1.0))
    calib_q, calib_kv = [], []
    if with_calib:
        Hc = w.calib_q_shape[1]
        if w.calib_q_sigma is not None:
            sig_q = log_uniform(rng_for(s, TAG_SIGMA, 1), *w.calib_q_sigma, size=Hc).astype(np.float32)
        else:
            sig_q = np.ones(Hc, np.float32)
        for k in range(w.calib_batches):
            rq = rng_for(s, TAG_CALIB_Q, k)
            xq = normal(rq, w.calib_q_shape, sig_q[None, :, None, None])
            if w.calib_q_sigma is not None:
                xq = with_outliers(rq, xq, w.ckv_outlier_rate, w.ckv_outlier_mult)
            calib_q.append(bf16_round(xq))
            rk = rng_for(s, TAG_CALIB_KV, k)
            xk = with_outliers(rk, normal(rk, w.calib_kv_shape, sig_kv), w.ckv_outlier_rate, w.ckv_outlier_mult)
            calib_kv.append(bf16_round(xk))
    return MLAInputs(q=q, ckv=ckv, krope=krope, lens=mla_lens(w), calib_q=calib_q, calib_kv=calib_kv)


# ----------------------------------------------------------------------------
# GQA decode workloads
# ----------------------------------------------------------------------------
@dataclass
class GQAWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    T_max: int
    softmax_scale: float
    lens: Optional[Sequence[int]] = None
    nu: float = 4.0
    sigma: Tuple[float, float] = (0.05, 5.0)
    calib_batches: int = 1
    calib_S: int = 512
    ratio: float = 0.9999
    seed: int = 0


def gqa_llama70b(B: int = 16, T: int = 4096, lens: Optional[Sequence[int]] = None) -> GQAWorkload:
    """Llama-3.1-70B-shaped GQA decode layer: 64 query heads, 8 KV heads, head_dim 128."""
    return GQAWorkload(name=f"llama70b-gqa b{B} hq64 hkv8 d128 ctx{T}", B=B, Hq=64, Hkv=8, D=128, T_max=T,
                       softmax_scale=1.0 / math.sqrt(128.0),
                       lens=list(lens) if lens is not None else [T] * B)


@dataclass
class GQAInputs:
    q: np.ndarray   # [B][Hq][D] bf16-exact float32
    k: np.ndarray   # [B][T_max][Hkv][D]
    v: np.ndarray   # [B][T_max][Hkv][D]
    lens: np.ndarray
    calib_q: List[np.ndarray]   # (1, Hq, S, D) batches
    calib_k: List[np.ndarray]   # (1, Hkv, S, D)
    calib_v: List[np.ndarray]


def gqa_inputs(w: GQAWorkload, with_calib: bool = True) -> GQAInputs:
    s = w.seed
    sq = log_uniform(rng_for(s, TAG_SIGMA, 0), *w.sigma, size=w.Hq).astype(np.float32)
    sk = log_uniform(rng_for(s, TAG_SIGMA, 1), *w.sigma, size=w.Hkv).astype(np.float32)
    sv = log_uniform(rng_for(s, TAG_SIGMA, 2), *w.sigma, size=w.Hkv).astype(np.float32)
    q = bf16_round(student_t(rng_for(s, TAG_Q), (w.B, w.Hq, w.D), w.nu, sq[None, :, None]))
    k = bf16_round(student_t(rng_for(s, TAG_K), (w.B, w.T_max, w.Hkv, w.D), w.nu, sk[None, None, :, None]))
    v = bf16_round(student_t(rng_for(s, TAG_V), (w.B, w.T_max, w.Hkv, w.D), w.nu, sv[None, None, :, None]))
    lens = np.asarray(w.lens if w.lens is not None else [w.T_max] * w.B, dtype=np.int32)
    cq, ck, cv = [], [], []
    if with_calib:
        for kk in range(w.calib_batches):
            cq.append(bf16_round(student_t(rng_for(s, TAG_CALIB_Q, kk), (1, w.Hq, w.calib_S, w.D), w.nu,
                                           sq[None, :, None, None])))
            ck.append(bf16_round(student_t(rng_for(s, TAG_CALIB_K, kk), (1, w.Hkv, w.calib_S, w.D), w.nu,
                                           sk[None, :, None, None])))
            cv.append(bf16_round(student_t(rng_for(s, TAG_CALIB_V, kk), (1, w.Hkv, w.calib_S, w.D), w.nu,
                                           sv[None, :, None, None])))
    return GQAInputs(q=q, k=k, v=v, lens=lens, calib_q=cq, calib_k=ck, calib_v=cv)


# ----------------------------------------------------------------------------
# GQA prefill workloads (the Llama-3.1-70B GQA law over S new rows)
# ----------------------------------------------------------------------------
@dataclass
class PrefillWorkload:
    name: str
    B: int
    S: int                      # rows of the q / out arrays
    T: int                      # rows of the k / v arrays
    Hq: int
    Hkv: int
    D: int
    softmax_scale: float
    q_lens: Sequence[int]
    kv_lens: Sequence[int]
    nu: float = 4.0
    sigma: Tuple[float, float] = (0.05, 5.0)
    calib_S: int = 512
    ratio: float = 0.9999
    seed: int = 0


def prefill_llama70b(B: int = 1, S: int = 4096, T: int = 4096, Hq: int = 64, Hkv: int = 8,
                     q_lens: Optional[Sequence[int]] = None, kv_lens: Optional[Sequence[int]] = None,
                     seed: int = 0) -> PrefillWorkload:
    """Llama-3.1-70B-shaped prefill (64 query heads, 8 KV heads, head_dim 128): by
    default every sequence attends S new rows over a T-token context."""
    ql = list(q_lens) if q_lens is not None else [S] * B
    kl = list(kv_lens) if kv_lens is not None else [T] * B
    return PrefillWorkload(name=f"llama70b-prefill b{B} s{S} t{T} hq{Hq} hkv{Hkv} d128", B=B, S=S, T=T, Hq=Hq,
                           Hkv=Hkv, D=128, softmax_scale=1.0 / math.sqrt(128.0), q_lens=ql, kv_lens=kl, seed=seed)


@dataclass
class PrefillInputs:
    q: np.ndarray   # [B][S][Hq][D] bf16-exact float32
    k: np.ndarray   # [B][T][Hkv][D]
    v: np.ndarray   # [B][T][Hkv][D]
    calib_q: List[np.ndarray]   # (1, Hq, calib_S, D)
    calib_k: List[np.ndarray]   # (1, Hkv, calib_S, D)
    calib_v: List[np.ndarray]


def prefill_inputs(w: PrefillWorkload) -> PrefillInputs:
    """Student-t (nu) activations, each head scaled by its own log-uniform sigma;
    one calibration batch per tensor drawn from the same law."""
    s = w.seed
    sq = log_uniform(rng_for(s, TAG_PREFILL, 0), *w.sigma, size=w.Hq).astype(np.float32)
    sk = log_uniform(rng_for(s, TAG_PREFILL, 1), *w.sigma, size=w.Hkv).astype(np.float32)
    sv = log_uniform(rng_for(s, TAG_PREFILL, 2), *w.sigma, size=w.Hkv).astype(np.float32)
    q = bf16_round(student_t(rng_for(s, TAG_PREFILL, 3), (w.B, w.S, w.Hq, w.D), w.nu, sq[None, None, :, None]))
    k = bf16_round(student_t(rng_for(s, TAG_PREFILL, 4), (w.B, w.T, w.Hkv, w.D), w.nu, sk[None, None, :, None]))
    v = bf16_round(student_t(rng_for(s, TAG_PREFILL, 5), (w.B, w.T, w.Hkv, w.D), w.nu, sv[None, None, :, None]))
    cq = [bf16_round(student_t(rng_for(s, TAG_PREFILL, 6), (1, w.Hq, w.calib_S, w.D), w.nu, sq[None, :, None, None]))]
    ck = [bf16_round(student_t(rng_for(s, TAG_PREFILL, 7), (1, w.Hkv, w.calib_S, w.D), w.nu,
                               sk[None, :, None, None]))]
    cv = [bf16_round(student_t(rng_for(s, TAG_PREFILL, 8), (1, w.Hkv, w.calib_S, w.D), w.nu,
                               sv[None, :, None, None]))]
    return PrefillInputs(q=q, k=k, v=v, calib_q=cq, calib_k=ck, calib_v=cv)


# ----------------------------------------------------------------------------
# Calibration-at-scale + quantize-append workload
# ----------------------------------------------------------------------------
@dataclass
class CalibWorkload:
    name: str
    B: int = 4
    H: int = 128
    S: int = 2048
    D: int = 192
    nu: float = 3.0
    sigma: Tuple[float, float] = (0.1, 10.0)
    batches: int = 4
    ratio: float = 0.9999
    # quantize-append part: new latent rows into a 512-wide INT8 cache
    app_B: int = 32
    app_T_new: int = 64
    app_D: int = 512
    app_T_max: int = 1024
    seed: int = 0


def calib_scale() -> CalibWorkload:
    return CalibWorkload(name="calib b4 h128 s2048 d192 x4 + append b32 t64 d512")


def calib_sigmas(w: CalibWorkload) -> np.ndarray:
    return log_uniform(rng_for(w.seed, TAG_SIGMA), *w.sigma, size=w.H).astype(np.float32)


def calib_head(w: CalibWorkload, k: int, h: int) -> np.ndarray:
    """Head h of calibration batch k, shape (B, S, D); each head has its own stream."""
    sig = calib_sigmas(w)[h]
    r = rng_for(w.seed, TAG_CALIB_Q, k, h)
    return bf16_round(student_t(r, (w.B, w.S, w.D), w.nu, sig))


def calib_batch(w: CalibWorkload, k: int, heads: Optional[Sequence[int]] = None) -> np.ndarray:
    """Calibration batch k laid out (B, H, S, D), restricted to ``heads`` if given."""
    hs = list(range(w.H)) if heads is None else list(heads)
    out = np.empty((w.B, len(hs), w.S, w.D), np.float32)
    for j, h in enumerate(hs):
        out[:, j] = calib_head(w, k, h)
    return out


def append_inputs(w: CalibWorkload) -> Tuple[np.ndarray, np.ndarray]:
    """New latent rows [B][T_new][1][D] (bf16-exact) and write positions pos[B]."""
    sig = float(log_uniform(rng_for(w.seed, TAG_SIGMA, 7), *w.sigma, size=1)[0])
    kv = bf16_round(student_t(rng_for(w.seed, TAG_APPEND), (w.app_B, w.app_T_new, 1, w.app_D), w.nu, sig))
    pos = rng_for(w.seed, TAG_POS).integers(0, w.app_T_max - w.app_T_new + 1, size=w.app_B).astype(np.int32)
    return kv, pos
