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
    # D = 128: two groups per thread within a head; D = 24: pairs of groups that
    # straddle two heads (three groups per row); (H, D) = (3, 24): rows of 72 bytes,
    # one group per thread; D = 20: rows not 16-byte multiples -> scalar kernel.
    for H, D in ((8, 128), (8, 24), (3, 24), (8, 20)):
        kv = W.bf16_round((rng.standard_t(4, (3, 5, H, D)) * rng.uniform(0.1, 4, (1, 1, H, 1))).astype(np.float32))
        sc = (np.abs(kv).max(axis=(0, 1, 3)) / 127 * 0.8).astype(np.float32)   # forces clamping
        sc[2] = 0.0                              # a zero scale quantizes to 0
        cache0 = np.zeros((3, 9, H, D), np.int8)
        pos = np.array([0, 4, 2], np.int32)
        cache = torch.from_numpy(cache0).cuda()
        F.quantize_append(bf16_dev(kv), torch.from_numpy(sc).cuda(), cache, torch.from_numpy(pos).cuda())
        assert np.array_equal(cache.cpu().numpy(), O.quantize_append(kv, sc, cache0, pos)), (H, D)


def test_append_grid_stride_passes_and_sequence_loop():
    # 16 sequences of 512 new rows x 2 heads x 512 plus a 64-wide RoPE row: more
    # 16-byte groups per sequence than one wave of blocks covers, so threads take
    # several passes and passes mix latent and RoPE groups.
    F = fa3()
    rng = np.random.default_rng(6)
    B, T_new, H, D, Dr, T_max = 16, 512, 2, 512, 64, 640
    kv = W.bf16_round((rng.standard_normal((B, T_new, H, D)) * np.array([0.5, 3.0])[None, None, :, None]).astype(np.float32))
    sc = (np.abs(kv).max(axis=(0, 1, 3)) / 127).astype(np.float32)
    rope = W.bf16_round(rng.standard_normal((B, T_new, Dr)).astype(np.float32))
    pos = rng.integers(0, T_max - T_new + 1, B).astype(np.int32)
    cache0 = rng.integers(-127, 128, (B, T_max, H, D)).astype(np.int8)
    cache = torch.from_numpy(cache0).cuda()
    rope_cache = torch.zeros(B, T_max, Dr, dtype=torch.bfloat16, device="cuda")
    F.quantize_append(bf16_dev(kv), torch.from_numpy(sc).cuda(), cache, torch.from_numpy(pos).cuda(),
                      bf16_dev(rope), rope_cache)
    assert np.array_equal(cache.cpu().numpy(), O.quantize_append(kv, sc, cache0, pos))
    rc = rope_cache.float().cpu().numpy()
    for b in range(B):
        assert np.array_equal(rc[b, pos[b]:pos[b] + T_new], rope[b])
        assert not rc[b, :pos[b]].any() and not rc[b, pos[b] + T_new:].any()
    # More sequences than one grid dimension holds (65535): the blocks loop over them.
    B = 70001
    kv = W.bf16_round(rng.standard_normal((B, 1, 1, 8)).astype(np.float32))
    pos = rng.integers(0, 2, B).astype(np.int32)
    cache0 = np.zeros((B, 2, 1, 8), np.int8)
    cache = torch.from_numpy(cache0).cuda()
    F.quantize_append(bf16_dev(kv), torch.tensor([0.02], device="cuda"), cache, torch.from_numpy(pos).cuda())
    assert np.array_equal(cache.cpu().numpy(), O.quantize_append(kv, np.array([0.02], np.float32), cache0, pos))


def test_append_every_bf16_value():
    # Every finite bf16 bit pattern (and +-inf) against scales that take each branch of
    # the group conversion: power-of-two and decimal scales (many exact and near ties),
    # a calibrated-looking one, the smallest and largest scales decided without a
    # division, scales outside that range, a subnormal, zero and a negative scale.
    F = fa3()
    bits = np.arange(65536, dtype=np.uint32)
    finite = (bits & 0x7F80) != 0x7F80
    inf = (bits & 0x7FFF) == 0x7F80
    x = ((bits[finite | inf] << 16).astype(np.uint32)).view(np.float32)
    x = np.concatenate([x, np.zeros((-len(x)) % 16, np.float32)])
    scales = np.array([0.02, 0.1, 1.0 / 127.0, 4.5 / 127.0, 0.25, 1.0 / 3.0, 7.7, 3.7e-3, 2.0 ** -100,
                       2.0 ** 100, 2.0 ** -101, 1.5e30, 1e-39, 0.0, -0.5], np.float32)
    H = len(scales)
    kv = np.broadcast_to(x, (1, 1, H, len(x))).copy()
    cache = torch.zeros(1, 1, H, len(x), dtype=torch.int8, device="cuda")
    F.quantize_append(bf16_dev(kv), torch.from_numpy(scales).cuda(), cache, torch.zeros(1, dtype=torch.int32, device="cuda"))
    got = cache.cpu().numpy()[0, 0]
    for h, s in enumerate(scales):
        want = O.quantize(x, s)
        bad = np.flatnonzero(got[h] != want)
        assert bad.size == 0, (float(s), x[bad[:5]], got[h][bad[:5]], want[bad[:5]])


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
