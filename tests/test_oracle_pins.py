"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- a hand-worked example, brute force, a closed form, an invariant, or
an independent library routine (torch) -- chosen so that a dropped term, a
wrong sign or index, or a transposed operand fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import fa3_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return W.bf16_round(np.asarray(x, np.float32))


# ---------------------------------------------------------------- calibration
def test_recall_window_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "recall_window_hand.json")))
    v = np.asarray(g["values"], np.float32)
    assert O.target_num(g["ratio"], v.size) == g["target_num"]
    lo, hi = O.recall_window(v, g["ratio"])
    assert (lo, hi) == (g["min_val"], g["max_val"])
    assert O.recall_window_bruteforce(v, g["ratio"]) == (lo, hi)
    sc = O.qparams(np.array([lo], np.float32), np.array([hi], np.float32))
    assert sc[0] == np.float32(g["abs_max"]) / np.float32(127)


def test_recall_window_exact_width_hand_example():
    # Two windows whose lengths differ by 2^-120 but round to the same float64.
    g = json.load(open(os.path.join(GOLDEN, "recall_window_exact_width.json")))
    v = np.array([float.fromhex(x) for x in g["values_hex"]], np.float32)
    assert O.target_num(g["ratio"], v.size) == g["target_num"]
    want = (float.fromhex(g["min_val_hex"]), float.fromhex(g["max_val_hex"]))
    assert O.recall_window(v, g["ratio"]) == want
    assert O.recall_window_bruteforce(v, g["ratio"]) == want
    # the float64 lengths do tie, so the example separates the two readings
    s = np.sort(v.astype(np.float64))
    w = s[2:] - s[:2]
    assert w[0] == w[1] and (s[0], s[2]) == tuple(float.fromhex(x) for x in g["float64_first_min_hex"])


@pytest.mark.parametrize("seed", range(8))
def test_recall_window_exact_widths_match_bruteforce_mixed_magnitudes(seed):
    rng = np.random.default_rng(100 + seed)
    v = W.mixed_magnitude_head(rng, int(rng.integers(20, 250)))
    ties = 0
    for ratio in (1.0, 0.9999, 0.95, 0.9, 0.75, 0.5, 0.2):
        got = O.recall_window(v, ratio)
        assert got == O.recall_window_bruteforce(v, ratio), (seed, ratio)
        t = O.target_num(ratio, v.size)
        s = O.sort_total_order(v)
        w = s[t - 1:] - s[: v.size - t + 1]
        ties += int(np.count_nonzero(w == w.min()) > 1)
    assert ties > 0          # float64 lengths tied somewhere: the exact comparison decided


def test_target_num_values():
    # The two calibration sizes of the workloads: 0.9999 * 16384 and 0.9999 * 1572864.
    assert O.target_num(0.9999, 2 * 128 * 64) == 16382
    assert O.target_num(0.9999, 4 * 2048 * 192) == 1572706
    assert O.target_num(1.0, 7) == 7
    assert O.target_num(1e-9, 10) == 1          # clamped to one element
    for bad in (0.0, -0.5, 1.0000001, float("nan")):
        with pytest.raises(ValueError):
            O.target_num(bad, 10)


@pytest.mark.parametrize("seed", range(12))
def test_recall_window_matches_bruteforce_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    kind = seed % 4
    if kind == 0:
        v = rng.standard_normal(n)
    elif kind == 1:
        v = rng.standard_t(3, n) * 5.0
    elif kind == 2:
        v = rng.integers(-3, 4, n).astype(np.float64)       # heavy duplicates
    else:
        v = np.concatenate([rng.standard_normal(n), [40.0, -55.0]])
    v = _bf16(v)
    for ratio in (1.0, 0.9999, 0.99, 0.9, 0.75, 0.5, 0.1, 1.0 / v.size):
        assert O.recall_window(v, ratio) == O.recall_window_bruteforce(v, ratio), (seed, ratio)


def test_recall_window_all_equal_and_single():
    v = np.full(50, 0.375, np.float32)
    for ratio in (1.0, 0.5, 0.01):
        assert O.recall_window(v, ratio) == (0.375, 0.375)
    assert O.recall_window(np.array([-3.0], np.float32), 0.9999) == (-3.0, -3.0)


def test_recall_window_ratio_one_is_min_max():
    rng = np.random.default_rng(5)
    v = _bf16(rng.standard_t(2, 5000) * 3)
    lo, hi = O.recall_window(v, 1.0)
    mn, mx = torch.aminmax(torch.from_numpy(v))
    assert (lo, hi) == (float(mn), float(mx))


def test_recall_window_invariants():
    rng = np.random.default_rng(11)
    v = _bf16(np.concatenate([rng.standard_normal(4000), rng.standard_normal(3) * 60]))
    for ratio in (0.9999, 0.999, 0.95, 0.6):
        t = O.target_num(ratio, v.size)
        lo, hi = O.recall_window(v, ratio)
        # the window holds at least target_num values
        assert np.count_nonzero((v >= lo) & (v <= hi)) >= t
        # both ends are data values
        assert lo in v and hi in v
        # no other window of target_num consecutive sorted values is narrower
        s = np.sort(v.astype(np.float64))
        assert np.all(s[t - 1:] - s[: v.size - t + 1] >= hi - lo)
        # independent of the order of the values inside the head
        assert O.recall_window(rng.permutation(v), ratio) == (lo, hi)
        # scaling by a power of two scales the result exactly
        assert O.recall_window(v * 4.0, ratio) == (lo * 4.0, hi * 4.0)


def test_signed_zero_order():
    v = np.array([0.0, -0.0, -0.0, 1.0, 2.0], np.float32)
    s = O.sort_total_order(v)
    assert [math.copysign(1, x) for x in s[:3]] == [-1, -1, 1]
    lo, hi = O.recall_window(v, 0.6)       # t = 3: [-0, +0] has width 0
    assert lo == 0.0 and math.copysign(1, lo) < 0 and hi == 0.0 and math.copysign(1, hi) > 0
    mn, mx = O.init_range(1)
    O.accumulate(mn, mx, np.array([0.0], np.float32), np.array([-0.0], np.float32))
    O.accumulate(mn, mx, np.array([-0.0], np.float32), np.array([0.0], np.float32))
    assert math.copysign(1, mn[0]) < 0 and math.copysign(1, mx[0]) > 0


def test_accumulation_order_independent_and_covering():
    w = W.mla_tiny()
    inp = W.mla_inputs(w)
    batches = inp.calib_q
    mn, mx = O.calibrate(batches, w.ratio)
    mn2, mx2 = O.calibrate(list(reversed(batches)), w.ratio)
    assert np.array_equal(mn, mn2) and np.array_equal(mx, mx2)
    per = [O.calibrate_batch(x, w.ratio) for x in batches]
    assert np.array_equal(mn, np.min([p[0] for p in per], axis=0))
    assert np.array_equal(mx, np.max([p[1] for p in per], axis=0))
    for lo, hi in per:
        assert np.all(mn <= lo) and np.all(mx >= hi)
    # resuming from saved state equals one pass
    a, b = O.calibrate(batches[:1], w.ratio)
    a, b = O.calibrate(batches[1:], w.ratio, a.copy(), b.copy())
    assert np.array_equal(a, mn) and np.array_equal(b, mx)


def test_calibrate_batch_groups_by_head():
    # Each head sees only its own B*S*D values: a head made of a shifted copy moves alone.
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((2, 3, 16, 8)))
    x[:, 1] = _bf16(x[:, 1] * 8.0)
    lo, hi = O.calibrate_batch(x, 0.9)
    for h in range(3):
        assert (lo[h], hi[h]) == O.recall_window(x[:, h].reshape(-1), 0.9)
    assert lo.shape == (3,)


# ------------------------------------------------------------------ qparams
def test_qparams_matches_float32_division():
    rng = np.random.default_rng(2)
    mn = (-np.abs(rng.standard_t(2, 1000)) * 7).astype(np.float32)
    mx = (np.abs(rng.standard_t(2, 1000)) * 7).astype(np.float32)
    want = np.maximum(np.abs(mn), np.abs(mx)).astype(np.float32) / np.float32(127)
    got = O.qparams(mn, mx)
    assert got.dtype == np.float32 and np.array_equal(got, want)
    # sign of the range does not matter; abs_max picks the larger side
    assert O.qparams(np.array([-5.0]), np.array([1.0]))[0] == np.float32(5) / np.float32(127)
    assert O.qparams(np.array([-1.0]), np.array([5.0]))[0] == np.float32(5) / np.float32(127)
    assert O.qparams(np.array([0.0]), np.array([0.0]))[0] == 0.0


# ----------------------------------------------------------------- quantize
def test_quantize_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "quantize_hand.json")))
    x = np.asarray(g["x"], np.float32)
    assert O.quantize(x, g["scale"]).tolist() == g["code"]
    assert O.quantize(-x, g["scale"]).tolist() == [-c for c in g["code"]]


def test_quantize_matches_torch_round_half_even():
    rng = np.random.default_rng(4)
    x = _bf16(rng.standard_t(3, (64, 257)) * 4)
    scale = O.qparams(x.min(axis=1) * 0.7, x.max(axis=1) * 0.7)      # forces clamping too
    got = O.quantize(x, scale[:, None])
    xt = torch.from_numpy(x)
    st = torch.from_numpy(scale)[:, None]
    want = torch.clamp(torch.round(xt / st), -127, 127).to(torch.int8).numpy()
    assert np.array_equal(got, want)
    # error bound for unclamped values: |x - q*s| <= s/2 (plus one float32 rounding)
    unclamped = np.abs(x / scale[:, None]) < 126.5
    err = np.abs(x.astype(np.float64) - got.astype(np.float64) * scale[:, None].astype(np.float64))
    assert np.all(err[unclamped] <= scale[:, None].repeat(x.shape[1], 1)[unclamped] * (0.5 + 1e-6))


def test_quantize_zero_scale_and_range():
    x = np.array([1.0, -3.0, 0.0], np.float32)
    assert O.quantize(x, 0.0).tolist() == [0, 0, 0]
    big = O.quantize(np.array([1e30, -1e30], np.float32), 1e-30)
    assert big.tolist() == [127, -127]
    assert O.quantize(np.linspace(-1000, 1000, 2001).astype(np.float32), 0.01).min() == -127


def test_quantize_append_writes_only_target_rows():
    rng = np.random.default_rng(6)
    kv = _bf16(rng.standard_normal((3, 4, 2, 16)))
    scale = np.array([0.02, 0.05], np.float32)
    cache = rng.integers(-127, 128, (3, 10, 2, 16)).astype(np.int8)
    pos = np.array([0, 6, 3], np.int32)
    out = O.quantize_append(kv, scale, cache, pos)
    for b in range(3):
        p = pos[b]
        for t in range(10):
            if p <= t < p + 4:
                assert np.array_equal(out[b, t], O.quantize(kv[b, t - p], scale[:, None]))
            else:
                assert np.array_equal(out[b, t], cache[b, t])
    with pytest.raises(ValueError):
        O.quantize_append(kv, scale, cache, np.array([0, 7, 3], np.int32))


# ----------------------------------------------------------------- paged cache
def _pages_of(cache, page_size, perm):
    """Pool and block table holding `cache` [B][T][...] (T a multiple of
    page_size): page k of the natural order is stored at pool page perm[k]."""
    B, T = cache.shape[:2]
    mp = T // page_size
    natural = cache.reshape((B * mp, page_size) + cache.shape[2:])
    pool = np.zeros((len(perm),) + natural.shape[1:], cache.dtype)
    pool[perm[:B * mp]] = natural
    bt = perm[:B * mp].reshape(B, mp).astype(np.int32)
    return pool, bt


def test_gather_paged_identity_permutation_and_hand_rows():
    rng = np.random.default_rng(21)
    cache = rng.integers(-127, 128, (3, 12, 2, 4)).astype(np.int8)
    full = np.full(3, 12)
    ident = np.arange(9)
    pool, bt = _pages_of(cache, 4, ident)
    assert np.array_equal(O.gather_paged(pool, bt, 4, full), cache)
    perm = rng.permutation(11)                          # two spare pages
    pool, bt = _pages_of(cache, 4, perm)
    assert np.array_equal(O.gather_paged(pool, bt, 4, full), cache)
    # By hand: token 5 of sequence 1 is row 1 of natural page 1 * 3 + 1 = 4.
    assert np.array_equal(pool[perm[4], 1], cache[1, 5])
    assert np.array_equal(O.gather_paged(pool, bt, 4, full)[1, 5], pool[perm[4], 1])
    # Rows past rows[b] are zero and their table entries are not read.
    bt2 = bt.copy()
    bt2[2, 1:] = -1
    g = O.gather_paged(pool, bt2, 4, np.array([12, 12, 3]))
    assert np.array_equal(g[2, :3], cache[2, :3]) and not g[2, 3:].any()
    with pytest.raises(ValueError):
        O.gather_paged(pool, bt2, 4, np.array([12, 12, 5]))


def test_quantize_append_paged_matches_contiguous_append():
    rng = np.random.default_rng(22)
    B, T_new, H, D, P, mp = 3, 5, 2, 8, 4, 4
    kv = _bf16(rng.standard_normal((B, T_new, H, D)))
    scale = np.array([0.02, 0.05], np.float32)
    cache = rng.integers(-127, 128, (B, mp * P, H, D)).astype(np.int8)
    perm = rng.permutation(B * mp + 2)
    pool, bt = _pages_of(cache, P, perm)
    pos = np.array([0, 3, 11], np.int32)              # sequence 1 spans pages 0-2, sequence 2 ends the last
    out = O.quantize_append_paged(kv, scale, pool, bt, pos)
    full = np.full(B, mp * P)
    assert np.array_equal(O.gather_paged(out, bt, P, full), O.quantize_append(kv, scale, cache, pos))
    spare = perm[B * mp:]
    assert np.array_equal(out[spare], pool[spare])     # pages no sequence owns stay untouched
    # By hand: token 3 + 2 = 5 of sequence 1 is row 1 of its page 1.
    assert np.array_equal(out[bt[1, 1], 1], O.quantize(kv[1, 2], scale[:, None]))
    with pytest.raises(ValueError):
        O.quantize_append_paged(kv, scale, pool, bt, np.array([0, 3, 12], np.int32))
    bad = bt.copy()
    bad[0, 1] = len(pool)
    with pytest.raises(ValueError):
        O.quantize_append_paged(kv, scale, pool, bad, pos)


# ---------------------------------------------------------- decode attention
def _sdpa64(q, k, v, scale):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None], scale=scale)[0].numpy()


def _mla_case(seed=0, B=3, H=5, Dl=32, Dr=8, T=50, lens=(50, 1, 17)):
    rng = np.random.default_rng(seed)
    q = _bf16(rng.standard_normal((B, H, Dl + Dr)))
    ckv8 = rng.integers(-127, 128, (B, T, Dl)).astype(np.int8)
    krope = _bf16(rng.standard_normal((B, T, Dr)))
    q_scale = (rng.uniform(0.005, 0.05, H)).astype(np.float32)
    kv_scale = np.float32(0.03)
    return q, ckv8, krope, q_scale, kv_scale, np.asarray(lens, np.int32)


def test_mla_decode_matches_sdpa_on_dequantized():
    q, ckv8, krope, q_scale, kv_scale, lens = _mla_case()
    sm = 1 / math.sqrt(40)
    out = O.mla_decode(q, ckv8, krope, q_scale, kv_scale, lens, sm)
    Dl = ckv8.shape[2]
    qd = np.concatenate([O.dequantize(O.quantize(q[:, :, :Dl], q_scale[None, :, None]), q_scale[None, :, None]),
                         q[:, :, Dl:].astype(np.float64)], axis=2)
    for b in range(q.shape[0]):
        n = lens[b]
        cd = O.dequantize(ckv8[b, :n], kv_scale)
        k = np.concatenate([cd, krope[b, :n].astype(np.float64)], axis=1)
        ref = _sdpa64(qd[b], k, cd, sm)
        assert np.max(np.abs(out[b] - ref)) < 1e-9


def test_mla_decode_closed_forms():
    q, ckv8, krope, q_scale, kv_scale, lens = _mla_case(seed=1)
    sm = 0.1
    out = O.mla_decode(q, ckv8, krope, q_scale, kv_scale, lens, sm)
    # one cached token: output is that token's dequantized latent
    assert np.array_equal(out[1], np.broadcast_to(ckv8[1, 0].astype(np.float64) * float(kv_scale), out[1].shape))
    # all tokens identical: output is that row for any scores
    c2 = ckv8.copy(); c2[2, :] = c2[2, 0]
    k2 = krope.copy(); k2[2, :] = k2[2, 0]
    o2 = O.mla_decode(q, c2, k2, q_scale, kv_scale, lens, sm)
    assert np.allclose(o2[2], ckv8[2, 0].astype(np.float64) * float(kv_scale), rtol=0, atol=1e-12)
    # zero length: zero row
    o0 = O.mla_decode(q, ckv8, krope, q_scale, kv_scale, np.array([0, 1, 17], np.int32), sm)
    assert np.all(o0[0] == 0)
    # token order inside the context does not matter
    perm = np.random.default_rng(0).permutation(lens[0])
    c3 = ckv8.copy(); c3[0, :lens[0]] = ckv8[0, perm]
    k3 = krope.copy(); k3[0, :lens[0]] = krope[0, perm]
    o3 = O.mla_decode(q, c3, k3, q_scale, kv_scale, lens, sm)
    assert np.allclose(o3[0], out[0], rtol=1e-12, atol=1e-12)
    # a dominant score picks that token: give token 5 a huge RoPE match
    k4 = krope.copy(); k4[0, 5] = _bf16(q[0, 0, -8:] * 64)
    o4 = O.mla_decode(q, ckv8, k4, q_scale, kv_scale, lens, 1.0)
    assert np.allclose(o4[0, 0], ckv8[0, 5] * float(kv_scale), atol=1e-6)


def test_mla_without_rope_is_gqa_with_one_kv_head():
    q, ckv8, krope, q_scale, kv_scale, lens = _mla_case(seed=2, Dr=0)
    sm = 0.2
    out = O.mla_decode(q, ckv8, krope, q_scale, kv_scale, lens, sm)
    q8 = O.quantize(q, q_scale[None, :, None])
    kv = ckv8[:, :, None, :]
    ref = O.gqa_decode(q8, kv, kv, q_scale, np.array([kv_scale]), np.array([kv_scale]), lens, sm)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_mla_rows_subset_equals_full():
    q, ckv8, krope, q_scale, kv_scale, lens = _mla_case(seed=3)
    full = O.mla_decode(q, ckv8, krope, q_scale, kv_scale, lens, 0.3)
    part = O.mla_decode(q, ckv8, krope, q_scale, kv_scale, lens, 0.3, rows=[(0, 4), (2, 1)])
    # (BLAS may sum in another order for a subset, hence the 1e-12 slack)
    assert np.allclose(part[0, 4], full[0, 4], rtol=1e-12, atol=1e-12)
    assert np.allclose(part[2, 1], full[2, 1], rtol=1e-12, atol=1e-12)
    assert np.all(part[1] == 0)


def test_mla_float_reference_matches_sdpa():
    q, ckv8, krope, q_scale, kv_scale, lens = _mla_case(seed=4)
    ckv = _bf16(ckv8.astype(np.float32) * 0.01)
    out = O.mla_decode_float(q, ckv, krope, lens, 0.25)
    for b in range(q.shape[0]):
        n = lens[b]
        k = np.concatenate([ckv[b, :n], krope[b, :n]], axis=1).astype(np.float64)
        ref = _sdpa64(q[b].astype(np.float64), k, ckv[b, :n].astype(np.float64), 0.25)
        assert np.max(np.abs(out[b] - ref)) < 1e-12


def _gqa_case(seed=0, B=2, Hq=8, Hkv=2, D=16, T=40, lens=(40, 9)):
    rng = np.random.default_rng(seed)
    q8 = rng.integers(-127, 128, (B, Hq, D)).astype(np.int8)
    k8 = rng.integers(-127, 128, (B, T, Hkv, D)).astype(np.int8)
    v8 = rng.integers(-127, 128, (B, T, Hkv, D)).astype(np.int8)
    qs = rng.uniform(0.001, 0.01, Hq).astype(np.float32)
    ks = rng.uniform(0.001, 0.01, Hkv).astype(np.float32)
    vs = rng.uniform(0.01, 0.1, Hkv).astype(np.float32)
    return q8, k8, v8, qs, ks, vs, np.asarray(lens, np.int32)


def test_gqa_decode_matches_sdpa_on_dequantized():
    q8, k8, v8, qs, ks, vs, lens = _gqa_case()
    sm = 1 / 4
    out = O.gqa_decode(q8, k8, v8, qs, ks, vs, lens, sm)
    G = q8.shape[1] // k8.shape[2]
    for b in range(q8.shape[0]):
        n = lens[b]
        qd = O.dequantize(q8[b], qs[:, None])
        kd = np.repeat(O.dequantize(k8[b, :n], ks[None, :, None]), G, axis=1)   # [n][Hq][D]
        vd = np.repeat(O.dequantize(v8[b, :n], vs[None, :, None]), G, axis=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qd)[:, None], torch.from_numpy(kd).transpose(0, 1),
            torch.from_numpy(vd).transpose(0, 1), scale=sm)[:, 0].numpy()
        assert np.max(np.abs(out[b] - ref)) < 1e-12


def test_gqa_group_mapping_and_closed_forms():
    q8, k8, v8, qs, ks, vs, lens = _gqa_case(seed=1)
    out = O.gqa_decode(q8, k8, v8, qs, ks, vs, np.array([1, 0], np.int32), 0.5)
    G = 4
    for h in range(8):
        assert np.array_equal(out[0, h], v8[0, 0, h // G].astype(np.float64) * float(vs[h // G]))
    assert np.all(out[1] == 0)
    # changing KV head 1 changes only query heads 4..7
    base = O.gqa_decode(q8, k8, v8, qs, ks, vs, lens, 0.5)
    v2 = v8.copy(); v2[:, :, 1] = -v2[:, :, 1]
    o2 = O.gqa_decode(q8, k8, v2, qs, ks, vs, lens, 0.5)
    assert np.array_equal(o2[:, :4], base[:, :4]) and np.allclose(o2[:, 4:], -base[:, 4:])


def test_gqa_float_reference_matches_sdpa():
    w = W.gqa_llama70b(B=1, T=64)
    w.Hq, w.Hkv, w.D = 8, 2, 32
    inp = W.gqa_inputs(w, with_calib=False)
    out = O.gqa_decode_float(inp.q, inp.k, inp.v, inp.lens, w.softmax_scale)
    qd, kd, vd = (x.astype(np.float64) for x in (inp.q[0], inp.k[0], inp.v[0]))
    kd = np.repeat(kd, 4, axis=1).transpose(1, 0, 2)
    vd = np.repeat(vd, 4, axis=1).transpose(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qd)[:, None], torch.from_numpy(kd), torch.from_numpy(vd), scale=w.softmax_scale)[:, 0]
    assert np.max(np.abs(out[0] - ref.numpy())) < 1e-12


# ------------------------------------------------------ prefill (GQA, INT8 q/k/v)
def _prefill_case(seed=0, B=2, S=9, Hq=4, Hkv=2, D=16, T=14):
    rng = np.random.default_rng(seed)
    q8 = rng.integers(-127, 128, (B, S, Hq, D)).astype(np.int8)
    k8 = rng.integers(-127, 128, (B, T, Hkv, D)).astype(np.int8)
    v8 = rng.integers(-127, 128, (B, T, Hkv, D)).astype(np.int8)
    qs = rng.uniform(0.002, 0.01, Hq).astype(np.float32)
    ks = rng.uniform(0.002, 0.01, Hkv).astype(np.float32)
    vs = rng.uniform(0.01, 0.05, Hkv).astype(np.float32)
    return q8, k8, v8, qs, ks, vs


def test_prefill_rows_are_decodes_at_their_positions():
    q8, k8, v8, qs, ks, vs = _prefill_case()
    q_lens, kv_lens = np.array([9, 4]), np.array([14, 6])        # prefixes of 5 and 2 cached tokens
    out = O.gqa_prefill(q8, k8, v8, qs, ks, vs, q_lens, kv_lens, 0.25)
    for b in range(2):
        for i in range(9):
            if i >= q_lens[b]:
                assert not out[b, i].any()
                continue
            pos = kv_lens[b] - q_lens[b] + i
            one = O.gqa_decode(q8[b:b + 1, i], k8[b:b + 1], v8[b:b + 1], qs, ks, vs, np.array([pos + 1]), 0.25)
            assert np.allclose(out[b, i], one[0], rtol=0, atol=1e-12)


def test_prefill_matches_causal_sdpa_on_dequantized():
    q8, k8, v8, qs, ks, vs = _prefill_case(seed=1, B=1, S=12, T=12)
    out = O.gqa_prefill(q8, k8, v8, qs, ks, vs, np.array([12]), np.array([12]), 0.2)
    G = 2
    q = q8[0].astype(np.float64) * qs[None, :, None]              # [S][Hq][D]
    k = np.repeat(k8[0].astype(np.float64) * ks[None, :, None], G, axis=1)
    v = np.repeat(v8[0].astype(np.float64) * vs[None, :, None], G, axis=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.transpose(1, 0, 2)), torch.from_numpy(k.transpose(1, 0, 2)),
        torch.from_numpy(v.transpose(1, 0, 2)), is_causal=True, scale=0.2).numpy().transpose(1, 0, 2)
    assert np.allclose(out[0], ref, rtol=1e-9, atol=1e-12)


def test_prefill_first_row_and_validation():
    q8, k8, v8, qs, ks, vs = _prefill_case(seed=2)
    out = O.gqa_prefill(q8, k8, v8, qs, ks, vs, np.array([9, 0]), np.array([9, 3]), 0.3)
    # a plain prefill's first row sees only token 0: its output is that token's value row
    for h in range(4):
        assert np.allclose(out[0, 0, h], v8[0, 0, h // 2] * float(vs[h // 2]), rtol=0, atol=1e-12)
    assert not out[1].any()                                       # no new rows
    with pytest.raises(ValueError):
        O.gqa_prefill(q8, k8, v8, qs, ks, vs, np.array([9, 4]), np.array([8, 6]), 0.3)   # kv_lens < q_lens



def test_prefill_row_selection_equals_full_rows():
    q8, k8, v8, qs, ks, vs = _prefill_case(seed=3)
    q_lens, kv_lens = np.array([9, 4]), np.array([14, 6])
    full = O.gqa_prefill(q8, k8, v8, qs, ks, vs, q_lens, kv_lens, 0.25)
    rows = [(0, 0), (0, 8), (1, 3)]
    part = O.gqa_prefill(q8, k8, v8, qs, ks, vs, q_lens, kv_lens, 0.25, rows=rows)
    for b, i in rows:
        assert np.array_equal(part[b, i], full[b, i])
    mask = np.zeros(part.shape[:2], bool)
    for b, i in rows:
        mask[b, i] = True
    assert not part[~mask].any()


# ------------------------------------------------------------ per-channel / asymmetric
def test_qparams_channel_hand_example():
    # channel 0: [-1, 3] -> width 4, scale 4/255, offset RNE(1 / (4/255)) - 128 = RNE(63.75) - 128 = -64
    # channel 1: [2, 5]  -> widened to [0, 5]: scale 5/255, offset 0 - 128 = -128
    # channel 2: [-6, -2] -> widened to [-6, 0]: scale 6/255, offset 255 - 128 = 127
    # channel 3: all zero -> scale 0, offset 0
    mn = np.array([-1.0, 2.0, -6.0, 0.0], np.float32)
    mx = np.array([3.0, 5.0, -2.0, 0.0], np.float32)
    sc, of = O.qparams_channel(mn, mx, asymmetric=True)
    assert np.array_equal(sc, np.array([4, 5, 6, 0], np.float32) / np.float32(255))
    assert of.tolist() == [-64.0, -128.0, 127.0, 0.0]
    ssc, sof = O.qparams_channel(mn, mx, asymmetric=False)
    assert np.array_equal(ssc, np.array([3, 5, 6, 0], np.float32) / np.float32(127)) and not sof.any()
    # the ends of the range land on (or next to) the extreme codes, and 0 is exact
    q = O.quantize_channel(np.stack([np.minimum(mn, 0), np.maximum(mx, 0), np.zeros(4, np.float32)]), sc, of, True)
    assert q[0, :3].tolist() == [-128, -128, -128] and q[1, :3].tolist() == [127, 127, 127]
    assert np.all(O.dequantize_channel(q[2], sc, of) == 0.0)


def test_quantize_channel_matches_torch_affine_quantizer():
    # torch's per-channel affine quantizer computes clamp(round(x * (1 / scale)) +
    # zero_point) with half-to-even rounding: an independent implementation of the
    # rule, which multiplies by a rounded reciprocal instead of dividing, so the two
    # may differ where x / scale lies within a hair of a half-integer (checked rare).
    rng = np.random.default_rng(12)
    H, D = 3, 16
    x = _bf16(rng.standard_normal((50, H, D)) * rng.uniform(0.1, 4, (1, H, D)))
    mn = x.min(axis=0) * 1.2
    mx = x.max(axis=0) * 0.9
    sc, of = O.qparams_channel(mn, mx, asymmetric=True)
    q = O.quantize_channel(x, sc, of, True)
    ref = torch.quantize_per_channel(torch.from_numpy(x.reshape(50, H * D)), torch.from_numpy(sc.reshape(-1)).double(),
                                     torch.from_numpy(of.reshape(-1).astype(np.int64)), 1, torch.qint8).int_repr()
    r = x.reshape(50, H * D).astype(np.float64) / sc.reshape(-1).astype(np.float64)
    near_tie = np.abs(r - np.floor(r) - 0.5) < 1e-3
    diff = q.reshape(50, H * D) != ref.numpy()
    assert not np.any(diff & ~near_tie) and np.count_nonzero(near_tie) < 0.01 * r.size
    # dequantization error inside the range is at most half a step
    inside = (x >= np.minimum(mn, 0)) & (x <= np.maximum(mx, 0))
    err = np.abs(O.dequantize_channel(q, sc, of) - x.astype(np.float64))
    assert np.all(err[inside] <= 0.5 * sc.astype(np.float64)[None].repeat(50, 0)[inside] * (1 + 1e-6))


def test_channel_calibration_is_per_head_on_each_channel():
    rng = np.random.default_rng(13)
    x = _bf16(rng.standard_t(3, (2, 3, 40, 5)) * rng.uniform(0.1, 3, (1, 3, 1, 5)))
    lo, hi = O.calibrate_channel_batch(x, 0.95)
    for h in range(3):
        for d in range(5):
            col = x[:, h, :, d].reshape(-1)
            assert (lo[h, d], hi[h, d]) == O.recall_window_bruteforce(col, 0.95)
    # a channel-constant layout reduces to the per-head calibration of that channel
    x2 = np.repeat(x[..., :1], 4, axis=-1)
    lo2, hi2 = O.calibrate_channel_batch(x2, 0.95)
    plo, phi = O.calibrate_batch(x[..., :1], 0.95)
    assert np.array_equal(lo2, np.repeat(plo[:, None], 4, 1)) and np.array_equal(hi2, np.repeat(phi[:, None], 4, 1))
    # accumulation over batches
    b2 = _bf16(rng.standard_normal((2, 3, 40, 5)) * 9)
    mn, mx = O.calibrate_channel([x, b2], 0.95)
    l2, h2 = O.calibrate_channel_batch(b2, 0.95)
    assert np.array_equal(mn, np.minimum(lo, l2)) and np.array_equal(mx, np.maximum(hi, h2))


def test_gqa_decode_channel_reduces_and_matches_sdpa():
    rng = np.random.default_rng(14)
    B, Hq, Hkv, T, D = 2, 4, 2, 9, 8
    q8 = rng.integers(-128, 128, (B, Hq, D)).astype(np.int8)
    k8 = rng.integers(-128, 128, (B, T, Hkv, D)).astype(np.int8)
    v8 = rng.integers(-128, 128, (B, T, Hkv, D)).astype(np.int8)
    qs, ks, vs = (rng.uniform(0.005, 0.02, (n, D)).astype(np.float32) for n in (Hq, Hkv, Hkv))
    qo, ko, vo = (rng.integers(-20, 20, (n, D)).astype(np.float32) for n in (Hq, Hkv, Hkv))
    lens = np.array([9, 4])
    out = O.gqa_decode_channel(q8, k8, v8, qs, qo, ks, ko, vs, vo, lens, 0.3)
    for b in range(B):
        n = lens[b]
        q = O.dequantize_channel(q8[b], qs, qo)                                     # [Hq][D]
        k = np.repeat(O.dequantize_channel(k8[b, :n], ks, ko), 2, axis=1)          # [n][Hq][D]
        v = np.repeat(O.dequantize_channel(v8[b, :n], vs, vo), 2, axis=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[:, None, :]), torch.from_numpy(k.transpose(1, 0, 2)),
            torch.from_numpy(v.transpose(1, 0, 2)), scale=0.3).numpy()[:, 0]
        assert np.allclose(out[b], ref, rtol=1e-9, atol=1e-12)
    # per-head scales broadcast along D with zero offsets: the per-head decode
    qh, kh, vh = qs[:, :1], ks[:, :1], vs[:, :1]
    z = lambda a: np.zeros_like(a)
    a = O.gqa_decode_channel(np.clip(q8, -127, 127), np.clip(k8, -127, 127), np.clip(v8, -127, 127),
                             np.repeat(qh, D, 1), z(qo), np.repeat(kh, D, 1), z(ko), np.repeat(vh, D, 1), z(vo),
                             lens, 0.3)
    bb = O.gqa_decode(np.clip(q8, -127, 127), np.clip(k8, -127, 127), np.clip(v8, -127, 127), qh[:, 0], kh[:, 0],
                      vh[:, 0], lens, 0.3)
    assert np.allclose(a, bb, rtol=1e-12, atol=1e-12)
