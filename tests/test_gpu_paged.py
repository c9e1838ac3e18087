"""GPU parity of the paged-cache calls: quantize-append into a page pool and MLA / GQA
decode through a block table, against the oracle on the gathered (contiguous) cache."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_attn_close, bf16_dev, fa3, paged_layout
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _mla_case(B, T, lens):
    w = W.mla_dsv3(B=B, T=T)
    inp = W.mla_inputs(w)
    q_scale = O.qparams(*O.calibrate(inp.calib_q, w.ratio))
    kv_scale = O.qparams(*O.calibrate(inp.calib_kv, w.ratio))
    return w, inp, q_scale, kv_scale, O.quantize(inp.ckv, kv_scale[0]), np.asarray(lens, np.int32)


def _mla_paged(F, w, inp, q_scale, kv_scale, ckv_pool, kr_pool, bt, lens, err=None):
    out = F.decode_attn_mla_paged(bf16_dev(inp.q), _t(ckv_pool), bf16_dev(kr_pool), _t(q_scale), _t(kv_scale),
                                  _t(lens), _t(bt), w.softmax_scale, dev_err=err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _mla_oracle(w, inp, q_scale, kv_scale, ckv_pool, kr_pool, bt, lens):
    P = ckv_pool.shape[1]
    ckv = O.gather_paged(ckv_pool, bt, P, lens)
    kr = O.gather_paged(kr_pool, bt, P, lens)
    return O.mla_decode(inp.q, ckv, kr, q_scale, float(kv_scale[0]), lens, w.softmax_scale)


@pytest.mark.parametrize("page_size", [64, 128, 256])
def test_mla_paged_ragged(page_size):
    F = fa3()
    w, inp, qs, kvs, ckv8, lens = _mla_case(3, 700, [700, 333, 64])
    rng = np.random.default_rng(page_size)
    ckv_pool, bt = paged_layout(ckv8, page_size, 5, rng)
    kr_pool, _ = paged_layout(inp.krope, page_size, 5, np.random.default_rng(page_size))   # same permutation
    ckv_pool = np.clip(ckv_pool, -127, 127).astype(np.int8)
    kr_pool = W.bf16_round(kr_pool)
    if page_size == 64:
        bt[1, 0] = bt[0, 0]                 # a shared first page (sequence 1 reads sequence 0's)
        bt[2, 1:] = -1                      # entries past lens[2] = 64 are never read
    got = _mla_paged(F, w, inp, qs, kvs, ckv_pool, kr_pool, bt, lens)
    ref = _mla_oracle(w, inp, qs, kvs, ckv_pool, kr_pool, bt, lens)
    assert_attn_close(got, ref, what=f"mla paged {page_size}")


def test_mla_paged_bad_entry_sets_error():
    F = fa3()
    w, inp, qs, kvs, ckv8, lens = _mla_case(3, 300, [300, 200, 129])
    rng = np.random.default_rng(5)
    ckv_pool, bt = paged_layout(ckv8, 64, 2, rng)
    kr_pool, _ = paged_layout(inp.krope, 64, 2, np.random.default_rng(5))
    kr_pool = W.bf16_round(kr_pool)
    bt[1, 2] = len(ckv_pool) + 7            # inside lens[1]: read as zeros, error flagged
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _mla_paged(F, w, inp, qs, kvs, ckv_pool, kr_pool, bt, lens, err)
    assert int(err.item()) & F.FA3_DEVERR_PAGE
    assert np.all(np.isfinite(got))
    keep = np.array([0, 2])
    ref = O.mla_decode(inp.q[keep], O.gather_paged(ckv_pool, bt[keep], 64, lens[keep]),
                       O.gather_paged(kr_pool, bt[keep], 64, lens[keep]), qs, float(kvs[0]), lens[keep],
                       w.softmax_scale)
    assert_attn_close(got[keep], ref, what="mla paged, other sequences")


def test_mla_paged_equals_contiguous_at_bench_size():
    # 32 sequences x 8192 tokens, pages of 64 in shuffled order: the same tiles in the
    # same schedule, so the outputs must agree bit for bit with the contiguous call.
    F = fa3()
    B, T, H, Dl, Dr, P = 32, 8192, 128, 512, 64, 64
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    ckv = torch.randint(-127, 128, (B, T, Dl), dtype=torch.int8, device="cuda", generator=g)
    kr = torch.randn(B, T, Dr, device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn(B, H, Dl + Dr, device="cuda", generator=g).to(torch.bfloat16)
    qs, kvs = torch.full((H,), 0.03, device="cuda"), torch.full((1,), 0.02, device="cuda")
    lens = torch.randint(1, T + 1, (B,), dtype=torch.int32, device="cuda", generator=g)
    mp = T // P
    perm = torch.randperm(B * mp, device="cuda", generator=g)
    ckv_pool = torch.empty(B * mp, P, Dl, dtype=torch.int8, device="cuda")
    kr_pool = torch.empty(B * mp, P, Dr, dtype=torch.bfloat16, device="cuda")
    ckv_pool[perm] = ckv.reshape(B * mp, P, Dl)
    kr_pool[perm] = kr.reshape(B * mp, P, Dr)
    bt = perm.reshape(B, mp).to(torch.int32).contiguous()
    a = F.decode_attn_mla(q, ckv, kr, qs, kvs, lens, 0.0721)
    b = F.decode_attn_mla_paged(q, ckv_pool, kr_pool, qs, kvs, lens, bt, 0.0721)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def _gqa_case(B, T, lens):
    w = W.gqa_llama70b(B=B, T=T)
    inp = W.gqa_inputs(w)
    qs = O.qparams(*O.calibrate(inp.calib_q, w.ratio))
    ks = O.qparams(*O.calibrate(inp.calib_k, w.ratio))
    vs = O.qparams(*O.calibrate(inp.calib_v, w.ratio))
    q8 = O.quantize(inp.q, qs[None, :, None])
    k8 = O.quantize(inp.k, ks[None, None, :, None])
    v8 = O.quantize(inp.v, vs[None, None, :, None])
    return w, q8, k8, v8, qs, ks, vs, np.asarray(lens, np.int32)


@pytest.mark.parametrize("page_size", [16, 32, 48, 64, 96, 128])
def test_gqa_paged_ragged(page_size):
    F = fa3()
    w, q8, k8, v8, qs, ks, vs, lens = _gqa_case(4, 300, [1, 37, 300, 129])
    k_pool, bt = paged_layout(k8, page_size, 3, np.random.default_rng(page_size))
    v_pool, _ = paged_layout(v8, page_size, 3, np.random.default_rng(page_size))
    k_pool = np.clip(k_pool, -127, 127).astype(np.int8)
    v_pool = np.clip(v_pool, -127, 127).astype(np.int8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = F.decode_attn_gqa_paged(_t(q8), _t(k_pool), _t(v_pool), _t(qs), _t(ks), _t(vs), _t(lens), _t(bt),
                                  w.softmax_scale, dev_err=err)
    torch.cuda.synchronize()
    got = got.float().cpu().numpy()
    ref = O.gqa_decode(q8, O.gather_paged(k_pool, bt, page_size, lens), O.gather_paged(v_pool, bt, page_size, lens),
                       qs, ks, vs, lens, w.softmax_scale)
    assert_attn_close(got, ref, bf16_out=True, what=f"gqa paged {page_size}")
    assert int(err.item()) == 0
    bt[2, min(3, (int(lens[2]) - 1) // page_size)] = -1     # a page inside lens[2]
    got = F.decode_attn_gqa_paged(_t(q8), _t(k_pool), _t(v_pool), _t(qs), _t(ks), _t(vs), _t(lens), _t(bt),
                                  w.softmax_scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & F.FA3_DEVERR_PAGE
    keep = np.array([0, 1, 3])
    assert_attn_close(got.float().cpu().numpy()[keep], ref[keep], bf16_out=True, what="gqa paged, others")


@pytest.mark.parametrize("B,T_new,H,D,Dr,P,mp", [
    (4, 37, 1, 512, 64, 16, 8),    # MLA latent + RoPE key, rows spanning pages
    (5, 1, 8, 128, 0, 64, 3),      # GQA decode step: one token per sequence
    (3, 9, 3, 24, 0, 7, 5),        # odd page size; 72-byte rows (one group per thread)
    (64, 300, 2, 512, 0, 32, 12),  # several grid-stride passes per sequence
])
def test_append_paged(B, T_new, H, D, Dr, P, mp):
    F = fa3()
    rng = np.random.default_rng(B * 1000 + T_new)
    kv = W.bf16_round((rng.standard_normal((B, T_new, H, D)) * rng.uniform(0.2, 3, (1, 1, H, 1))).astype(np.float32))
    sc = (np.abs(kv).max(axis=(0, 1, 3)) / 127 * 0.9).astype(np.float32)
    n = B * mp + 3
    bt = rng.permutation(n)[:B * mp].reshape(B, mp).astype(np.int32)
    pos = rng.integers(0, mp * P - T_new + 1, B).astype(np.int32)
    pool0 = rng.integers(-127, 128, (n, P, H, D)).astype(np.int8)
    pool = _t(pool0)
    rope = rope_pool = None
    if Dr:
        rope = W.bf16_round(rng.standard_normal((B, T_new, Dr)).astype(np.float32))
        rope_pool = torch.zeros(n, P, Dr, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.quantize_append_paged(bf16_dev(kv), _t(sc), pool, _t(bt), _t(pos), None if rope is None else bf16_dev(rope),
                            rope_pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(pool.cpu().numpy(), O.quantize_append_paged(kv, sc, pool0, bt, pos))
    if Dr:
        rp = rope_pool.float().cpu().numpy()
        for b in range(B):
            for t in range(T_new):
                x = pos[b] + t
                assert np.array_equal(rp[bt[b, x // P], x % P], rope[b, t])
        assert np.count_nonzero(np.abs(rp).sum(axis=-1)) <= B * T_new


def test_append_paged_bad_entry_skips_row():
    F = fa3()
    rng = np.random.default_rng(9)
    B, T_new, H, D, P, mp = 3, 6, 1, 64, 4, 4
    kv = W.bf16_round(rng.standard_normal((B, T_new, H, D)).astype(np.float32))
    sc = np.array([0.02], np.float32)
    bt = rng.permutation(B * mp).reshape(B, mp).astype(np.int32)
    pos = np.array([0, 2, 5], np.int32)
    pool0 = np.zeros((B * mp, P, H, D), np.int8)
    bad = bt.copy()
    bad[1, 1] = 999                        # positions 4..7 of sequence 1
    pool = _t(pool0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    F.quantize_append_paged(bf16_dev(kv), _t(sc), pool, _t(bad), _t(pos), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & F.FA3_DEVERR_PAGE
    want = O.quantize_append_paged(kv[[0, 2]], sc, pool0, bt[[0, 2]], pos[[0, 2]])
    # sequence 1: positions 2, 3 land in its valid page 0; positions 4..7 are skipped
    want[bt[1, 0], 2:4] = O.quantize(kv[1, 0:2], sc[:, None])
    assert np.array_equal(pool.cpu().numpy(), want)
