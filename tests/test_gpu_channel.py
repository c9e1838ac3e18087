"""GPU parity of the per-channel (symmetric and asymmetric) parameters and
quantize-append: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import bf16_dev, fa3
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu


def _bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def _ranges(rng, H, D):
    mn = W.bf16_round((-np.abs(rng.standard_t(3, (H, D))) * rng.uniform(0.01, 8, (H, 1))).astype(np.float32))
    mx = W.bf16_round((np.abs(rng.standard_t(3, (H, D))) * rng.uniform(0.01, 8, (H, 1))).astype(np.float32))
    mn[0, :4] = [2.0, 0.0, -0.0, -3.0]        # a positive minimum, zeros
    mx[0, :4] = [5.0, 0.0, 0.0, -1.0]         # an all-zero channel, a negative maximum
    return mn, mx


@pytest.mark.parametrize("asym", [False, True])
def test_qparams_channel_bit_exact(asym):
    F = fa3()
    mn, mx = _ranges(np.random.default_rng(40), 8, 128)
    sc, of = F.qparams_channel(torch.from_numpy(mn).cuda(), torch.from_numpy(mx).cuda(), asym)
    osc, oof = O.qparams_channel(mn, mx, asym)
    assert np.array_equal(_bits(sc.cpu().numpy()), _bits(osc))
    assert np.array_equal(of.cpu().numpy(), oof)


@pytest.mark.parametrize("asym", [False, True])
def test_quantize_append_channel_bit_exact(asym):
    F = fa3()
    rng = np.random.default_rng(41)
    B, T_new, H, D, T_max = 5, 7, 8, 128, 40
    mn, mx = _ranges(rng, H, D)
    sc, of = O.qparams_channel(mn, mx, asym)
    x = W.bf16_round((rng.standard_normal((B, T_new, H, D)) * np.maximum(np.abs(mx), np.abs(mn))[None, None] * 0.6)
                     .astype(np.float32))
    # near-ties: values whose quotient lies at (or next to) a half-integer step
    k = rng.integers(-120, 120, (B, T_new, H, D)).astype(np.float32) + 0.5
    ties = W.bf16_round((k * sc[None, None]).astype(np.float32))
    x = np.where(rng.random(x.shape) < 0.3, ties, x)
    x[0, 0, 0, :8] = [2.0 ** 100, -2.0 ** 100, 0.0, -0.0, 3.0, -2.0, 2.0 ** -100, 7.0]     # clamps, zeros, the zero channel
    pos = np.array([0, 3, 33, 10, 40], np.int32)                          # the last one is out of range
    cache = rng.integers(-128, 128, (B, T_max, H, D)).astype(np.int8)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    c = t(cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.quantize_append_channel(bf16_dev(x), t(sc), t(of), asym, c, t(pos), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & F.FA3_DEVERR_POS
    want = cache.copy()
    for b in range(B - 1):
        want[b, pos[b]:pos[b] + T_new] = O.quantize_channel(x[b], sc, of, asym)
    assert np.array_equal(c.cpu().numpy(), want)


@pytest.mark.parametrize("ratio", [1.0, 0.9999, 0.999, 0.99])
def test_calibrate_perchannel_bit_exact(ratio):
    # (B, H, S, D) = (3, 4, 1000, 40): 3000 values per channel, 1 .. 31 window starts;
    # channels with duplicates, signed zeros, one constant channel; a strided view.
    F = fa3()
    rng = np.random.default_rng(42)
    B, H, S, D = 3, 4, 1000, 40
    x = (rng.standard_t(3, (B, H, S, D)) * rng.uniform(0.05, 10, (1, H, 1, D))).astype(np.float32)
    x[:, 0, :, 0] = rng.integers(-2, 3, (B, S))
    x[:, 0, :, 1] = np.where(rng.random((B, S)) < 0.5, 0.0, -0.0)
    x[:, 0, :, 2] = 0.375
    x = W.bf16_round(x)
    big = torch.zeros(B, H + 1, S, D + 8, dtype=torch.bfloat16, device="cuda")
    big[:, 1:, :, :D] = bf16_dev(x)
    view = big[:, 1:, :, :D]
    omn, omx = O.calibrate_channel([x, x[::-1].copy() * 0.5], ratio)
    mn = torch.full((H, D), float("inf"), device="cuda")
    mx = torch.full((H, D), float("-inf"), device="cuda")
    F.calibrate_perchannel(view, ratio, mn, mx)
    F.calibrate_perchannel(bf16_dev(x[::-1].copy() * 0.5), ratio, mn, mx)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn))
    assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx))


def test_channel_pipeline_calibrate_params_append():
    # calibration -> asymmetric parameters -> quantize-append, all on the GPU, bit-exact
    F = fa3()
    rng = np.random.default_rng(43)
    B, H, S, D = 2, 8, 512, 128
    calib = [W.bf16_round((rng.standard_t(4, (B, H, S, D)) * rng.uniform(0.05, 5, (1, H, 1, D)) +
                           rng.uniform(-2, 2, (1, H, 1, D))).astype(np.float32)) for _ in range(2)]
    mn = torch.full((H, D), float("inf"), device="cuda")
    mx = torch.full((H, D), float("-inf"), device="cuda")
    for c in calib:
        F.calibrate_perchannel(bf16_dev(c), 0.9999, mn, mx)
    sc, of = F.qparams_channel(mn, mx, True)
    omn, omx = O.calibrate_channel(calib, 0.9999)
    osc, oof = O.qparams_channel(omn, omx, True)
    assert np.array_equal(_bits(sc.cpu().numpy()), _bits(osc)) and np.array_equal(of.cpu().numpy(), oof)
    new = W.bf16_round((rng.standard_t(4, (4, 16, H, D)) * 2).astype(np.float32))
    cache = torch.zeros(4, 64, H, D, dtype=torch.int8, device="cuda")
    pos = torch.tensor([0, 5, 48, 20], dtype=torch.int32, device="cuda")
    F.quantize_append_channel(bf16_dev(new), sc, of, True, cache, pos)
    want = np.zeros((4, 64, H, D), np.int8)
    for b, p0 in enumerate([0, 5, 48, 20]):
        want[b, p0:p0 + 16] = O.quantize_channel(new[b], osc, oof, True)
    assert np.array_equal(cache.cpu().numpy(), want)


@pytest.mark.parametrize("B,T,lens", [(4, 300, [300, 1, 129, 0]), (16, 4096, None)])
def test_gqa_decode_channel_against_oracle(B, T, lens):
    # per-channel asymmetric q, k, v calibrated and quantized by the oracle; the
    # Llama-70B shape (16 x 4096, split over several CTAs per sequence) included
    F = fa3()
    w = W.gqa_llama70b(B=B, T=T, lens=lens)
    inp = W.gqa_inputs(w)
    qs, qo = O.qparams_channel(*O.calibrate_channel(inp.calib_q, 0.9999), True)
    ks, ko = O.qparams_channel(*O.calibrate_channel(inp.calib_k, 0.9999), True)
    vs, vo = O.qparams_channel(*O.calibrate_channel(inp.calib_v, 0.9999), True)
    q8 = O.quantize_channel(inp.q, qs, qo, True)
    k8 = O.quantize_channel(inp.k, ks, ko, True)
    v8 = O.quantize_channel(inp.v, vs, vo, True)
    ln = np.asarray(w.lens, np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    got = F.decode_attn_gqa_channel(t(q8), t(k8), t(v8), t(qs), t(qo), t(ks), t(ko), t(vs), t(vo), t(ln),
                                    w.softmax_scale).float().cpu().numpy()
    ref = O.gqa_decode_channel(q8, k8, v8, qs, qo, ks, ko, vs, vo, ln, w.softmax_scale)
    from helpers import assert_attn_close
    assert_attn_close(got, ref, bf16_out=True, what=f"gqa channel B={B} T={T}")
    assert not got[ln == 0].any()
