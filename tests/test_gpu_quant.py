"""GPU parity of qparams and quantize-append: bit-exact codes and scales."""
import json
import os

import numpy as np
import pytest
import torch

import workloads as W
from helpers import bf16_dev, fa3
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_qparams_bit_exact():
    F = fa3()
    rng = np.random.default_rng(1)
    mn = (-np.abs(rng.standard_t(2, 333)) * 9).astype(np.float32)
    mx = (np.abs(rng.standard_t(2, 333)) * 9).astype(np.float32)
    mn[:5] = 0.0
    mx[:3] = 0.0
    got = F.qparams(torch.from_numpy(mn).cuda(), torch.from_numpy(mx).cuda()).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), O.qparams(mn, mx).view(np.uint32))


def test_quantize_golden_codes():
    F = fa3()
    g = json.load(open(os.path.join(GOLDEN, "quantize_hand.json")))
    x = np.asarray(g["x"], np.float32)
    n = x.size + (-x.size) % 8
    kv = np.zeros((1, 1, 1, n), np.float32)
    kv[0, 0, 0, :x.size] = x
    cache = torch.zeros(1, 1, 1, n, dtype=torch.int8, device="cuda")
    F.quantize_append(bf16_dev(kv), torch.tensor([g["scale"]], device="cuda"), cache,
                      torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert cache.cpu().numpy()[0, 0, 0, :x.size].tolist() == g["code"]


def test_append_large_with_rope_bit_exact():
    F = fa3()
    w = W.calib_scale()
    kv, pos = W.append_inputs(w)
    sc = O.qparams(*O.calibrate([kv.transpose(0, 2, 1, 3)], w.ratio))     # (B, H=1, T, D)
    rng = np.random.default_rng(3)
    cache0 = rng.integers(-127, 128, (w.app_B, w.app_T_max, 1, w.app_D)).astype(np.int8)
    rope = W.bf16_round(rng.standard_normal((w.app_B, w.app_T_new, 64)).astype(np.float32))
    cache = torch.from_numpy(cache0).cuda()
    rope_cache = torch.zeros(w.app_B, w.app_T_max, 64, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.quantize_append(bf16_dev(kv), torch.from_numpy(sc).cuda(), cache, torch.from_numpy(pos).cuda(),
                      bf16_dev(rope), rope_cache, err)
    want = O.quantize_append(kv, sc, cache0, pos)
    assert np.array_equal(cache.cpu().numpy(), want)
    rc = rope_cache.float().cpu().numpy()
    for b in range(w.app_B):
        assert np.array_equal(rc[b, pos[b]:pos[b] + w.app_T_new], rope[b])
    assert int(err.item()) == 0


def test_append_gqa_heads_and_scalar_path():
    F = fa3()
    rng = np.random.default_rng(4)
    for D in (128, 20):                          # 20: rows not 16-byte multiples -> scalar kernel
        kv = W.bf16_round((rng.standard_t(4, (3, 5, 8, D)) * rng.uniform(0.1, 4, (1, 1, 8, 1))).astype(np.float32))
        sc = (np.abs(kv).max(axis=(0, 1, 3)) / 127 * 0.8).astype(np.float32)   # forces clamping
        sc[2] = 0.0                              # a zero scale quantizes to 0
        cache0 = np.zeros((3, 9, 8, D), np.int8)
        pos = np.array([0, 4, 2], np.int32)
        cache = torch.from_numpy(cache0).cuda()
        F.quantize_append(bf16_dev(kv), torch.from_numpy(sc).cuda(), cache, torch.from_numpy(pos).cuda())
        assert np.array_equal(cache.cpu().numpy(), O.quantize_append(kv, sc, cache0, pos)), D


def test_append_bad_position_sets_error_and_skips():
    F = fa3()
    kv = W.bf16_round(np.ones((2, 4, 1, 16), np.float32))
    cache = torch.zeros(2, 8, 1, 16, dtype=torch.int8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.tensor([5, 2], dtype=torch.int32, device="cuda")    # 5 + 4 > 8
    F.quantize_append(bf16_dev(kv), torch.tensor([0.5], device="cuda"), cache, pos, dev_err=err)
    c = cache.cpu().numpy()
    assert int(err.item()) & F.FA3_DEVERR_POS
    assert np.all(c[0] == 0)
    assert np.all(c[1, 2:6] == 2) and np.all(c[1, :2] == 0) and np.all(c[1, 6:] == 0)


def test_query_quantization_as_append():
    # A GQA query: T_new = T_max = 1, pos = 0.
    F = fa3()
    w = W.gqa_llama70b(B=4, T=64)
    inp = W.gqa_inputs(w)
    qs = O.qparams(*O.calibrate(inp.calib_q, w.ratio))
    q8 = torch.zeros(w.B, 1, w.Hq, w.D, dtype=torch.int8, device="cuda")
    F.quantize_append(bf16_dev(inp.q[:, None]), torch.from_numpy(qs).cuda(), q8,
                      torch.zeros(w.B, dtype=torch.int32, device="cuda"))
    assert np.array_equal(q8.cpu().numpy()[:, 0], O.quantize(inp.q, qs[None, :, None]))


def test_codes_near_rounding_boundaries():
    # Quotients x/scale on or next to half-integers (exact ties for power-of-two
    # scales, near-ties otherwise): codes must equal the IEEE float32 division's.
    F = fa3()
    rng = np.random.default_rng(11)
    scales = np.array([1.0 / 64, 0.25, 2.0, 0.0173, 0.31, 1.0 / 3.0, 2.5e-3, 7.7], np.float32)
    for s in scales:
        k = rng.integers(-130, 131, 4096).astype(np.float32)
        x = ((k + 0.5) * s).astype(np.float32)
        x = np.concatenate([x, np.nextafter(x, np.float32(np.inf)), np.nextafter(x, np.float32(-np.inf)),
                            (k * s).astype(np.float32)])
        x = W.bf16_round(x)[None, None, None, :]                          # [B=1][T_new=1][H=1][D]
        cache = torch.zeros(1, 1, 1, x.shape[-1], dtype=torch.int8, device="cuda")
        F.quantize_append(bf16_dev(x), torch.tensor([s], device="cuda"), cache,
                          torch.zeros(1, dtype=torch.int32, device="cuda"))
        assert np.array_equal(cache.cpu().numpy()[0, 0, 0], O.quantize(x[0, 0, 0], s)), s
