"""GPU parity of GQA decode attention (INT8 q/k/v, bf16 output) against the float64 oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_attn_close, fa3
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu


def _case(w, lens=None):
    inp = W.gqa_inputs(w)
    qs = O.qparams(*O.calibrate(inp.calib_q, w.ratio))
    ks = O.qparams(*O.calibrate(inp.calib_k, w.ratio))
    vs = O.qparams(*O.calibrate(inp.calib_v, w.ratio))
    q8 = O.quantize(inp.q, qs[None, :, None])
    k8 = O.quantize(inp.k, ks[None, None, :, None])
    v8 = O.quantize(inp.v, vs[None, None, :, None])
    lens = inp.lens if lens is None else np.asarray(lens, np.int32)
    return inp, (q8, k8, v8, qs, ks, vs, lens)


def _run(F, w, args, err=None):
    q8, k8, v8, qs, ks, vs, lens = args
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = F.decode_attn_gqa(t(q8), t(k8), t(v8), t(qs), t(ks), t(vs), t(lens), w.softmax_scale, dev_err=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def test_ragged_small():
    F = fa3()
    w = W.gqa_llama70b(B=4, T=300)
    inp, args = _case(w, lens=[1, 37, 300, 129])
    got = _run(F, w, args)
    ref = O.gqa_decode(*args[:6], args[6], w.softmax_scale)
    assert_attn_close(got, ref, bf16_out=True, what="gqa ragged")


def test_edge_lengths_and_errors():
    F = fa3()
    w = W.gqa_llama70b(B=5, T=96)
    inp, args = _case(w, lens=[0, 16, 15, 17, 96])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(F, w, args, err)
    ref = O.gqa_decode(*args[:6], args[6], w.softmax_scale)
    assert_attn_close(got, ref, bf16_out=True, what="gqa edges")
    assert np.all(got[0] == 0) and int(err.item()) == 0
    bad = list(args)
    bad[6] = np.array([97, 16, -1, 17, 96], np.int32)
    got = _run(F, w, bad, err)
    assert int(err.item()) & F.FA3_DEVERR_LENS
    assert np.all(got[0] == 0) and np.all(got[2] == 0)


def test_fewer_query_heads_per_group():
    F = fa3()
    w = W.gqa_llama70b(B=2, T=200)
    w.Hq, w.Hkv = 12, 4                   # 3 query heads per KV head
    inp, args = _case(w, lens=[200, 77])
    got = _run(F, w, args)
    ref = O.gqa_decode(*args[:6], args[6], w.softmax_scale)
    assert_attn_close(got, ref, bf16_out=True, what="gqa G=3")


def test_split_plans_and_workspace_reuse():
    # Split-K plans of several shapes (one split with several pairs per wave,
    # many splits of few tokens, a single split; lengths past a split's start,
    # zero and one) through one explicit workspace reused across all of them.
    F = fa3()
    cases = [
        (3, 64, 8, 4096, [4096, 70, 2500]),
        (40, 16, 2, 300, None),
        (600, 8, 1, 64, None),
        (7, 24, 8, 1000, [1000, 1, 999, 64, 65, 0, 513]),
        (40, 64, 8, 2048, None),
    ]
    need = max(F.gqa_workspace_size(B, Hq, Hkv, 128, T) for B, Hq, Hkv, T, _ in cases)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for B, Hq, Hkv, T, lens in cases:
        w = W.gqa_llama70b(B=B, T=T)
        w.Hq, w.Hkv = Hq, Hkv
        if lens is None:
            lens = np.random.default_rng(B).integers(1, T + 1, B)
        inp, args = _case(w, lens=lens)
        q8, k8, v8, qs, ks, vs, ln = args
        out = F.decode_attn_gqa(t(q8), t(k8), t(v8), t(qs), t(ks), t(vs), t(ln), w.softmax_scale, workspace=ws)
        torch.cuda.synchronize()
        ref = O.gqa_decode(*args[:6], ln, w.softmax_scale)
        assert_attn_close(out.float().cpu().numpy(), ref, bf16_out=True, what=f"gqa split B={B} Hkv={Hkv} T={T}")


@pytest.mark.slow
def test_llama70b_full_size():
    F = fa3()
    w = W.gqa_llama70b()
    inp, args = _case(w)
    got = _run(F, w, args)
    ref = O.gqa_decode(*args[:6], args[6], w.softmax_scale)
    max_abs, rrms = assert_attn_close(got, ref, bf16_out=True, what="gqa llama70b")
    print(f"gqa full: max_abs(after bf16 slack)={max_abs:.3e} rel_rms={rrms:.3e}")


def test_stream_order_with_other_kernels_between_calls():
    # Programmatic dependent launches: each call must see the query and lengths that
    # ordinary device copies wrote just before it; the clone after it must see its output.
    F = fa3()
    w = W.gqa_llama70b(B=3, T=640)
    inp, args = _case(w, lens=[640, 300, 17])
    q8, k8, v8, qs, ks, vs, _ = args
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    variants = [(q8, np.array([640, 300, 17], np.int32)),
                (np.ascontiguousarray(-q8), np.array([5, 640, 211], np.int32)),
                (np.ascontiguousarray(q8[:, ::-1]), np.array([129, 1, 640], np.int32))]
    dq = torch.empty(q8.shape, dtype=torch.int8, device="cuda")
    dl = torch.empty(w.B, dtype=torch.int32, device="cuda")
    srcs = [(t(q), t(ls)) for q, ls in variants]
    dk, dv, dqs, dks, dvs = t(k8), t(v8), t(qs), t(ks), t(vs)
    keep = []
    torch.cuda.synchronize()
    for sq, sl in srcs:
        dq.copy_(sq)
        dl.copy_(sl)
        out = F.decode_attn_gqa(dq, dk, dv, dqs, dks, dvs, dl, w.softmax_scale)
        keep.append(out.clone())
    torch.cuda.synchronize()
    for (q, ls), got in zip(variants, keep):
        ref = O.gqa_decode(q, k8, v8, qs, ks, vs, ls, w.softmax_scale)
        assert_attn_close(got.float().cpu().numpy(), ref, bf16_out=True, what=f"gqa ordered {ls.tolist()}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 1), (40, 5)])
def test_group_sizes(Hq, Hkv):
    # G = 1 (one query head per KV head), G = 8 with a single KV head, G = 8 over 5 KV heads
    F = fa3()
    w = W.gqa_llama70b(B=2, T=300)
    w.Hq, w.Hkv = Hq, Hkv
    inp, args = _case(w, lens=[300, 65])
    got = _run(F, w, args)
    ref = O.gqa_decode(*args[:6], args[6], w.softmax_scale)
    assert_attn_close(got, ref, bf16_out=True, what=f"gqa Hq={Hq} Hkv={Hkv}")
