"""GPU parity of absorbed-MLA decode attention (INT8 latent, bf16 RoPE key) against the float64 oracle."""
import os

import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_attn_close, bf16_dev, fa3
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu


def _prepare(w, lens=None):
    inp = W.mla_inputs(w)
    q_scale = O.qparams(*O.calibrate(inp.calib_q, w.ratio))
    if q_scale.size != w.H:                       # calibration head count == query heads
        raise AssertionError("calibration heads")
    kv_scale = O.qparams(*O.calibrate(inp.calib_kv, w.ratio))
    ckv8 = O.quantize(inp.ckv, kv_scale[0])
    lens = inp.lens if lens is None else np.asarray(lens, np.int32)
    return inp, q_scale, kv_scale, ckv8, lens


def _run(F, w, inp, q_scale, kv_scale, ckv8, lens, err=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = F.decode_attn_mla(bf16_dev(inp.q), t(ckv8), bf16_dev(inp.krope), t(q_scale), t(kv_scale), t(lens),
                            w.softmax_scale, dev_err=err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _oracle(w, inp, q_scale, kv_scale, ckv8, lens, rows=None):
    return O.mla_decode(inp.q, ckv8, inp.krope, q_scale, float(kv_scale[0]), lens, w.softmax_scale, rows=rows)


def test_tiny_mla_full():
    F = fa3()
    w = W.mla_tiny()
    args = _prepare(w)
    got = _run(F, w, *args)
    ref = _oracle(w, *args)
    assert_attn_close(got, ref, what="tiny mla")


def test_dsv3_shape_ragged():
    F = fa3()
    w = W.mla_dsv3(B=3, T=700)
    args = _prepare(w, lens=[700, 333, 64])
    got = _run(F, w, *args)
    ref = _oracle(w, *args)
    assert_attn_close(got, ref, what="dsv3 ragged")


def test_edge_lengths_errors_and_small_shapes():
    F = fa3()
    w = W.mla_dsv3(B=6, T=130)
    args = list(_prepare(w, lens=[0, 1, 63, 64, 65, 130]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(F, w, *args, err=err)
    assert_attn_close(got, _oracle(w, *args), what="mla edges")
    assert np.all(got[0] == 0) and int(err.item()) == 0
    args[4] = np.array([131, 1, -5, 64, 65, 130], np.int32)
    got = _run(F, w, *args, err=err)
    assert int(err.item()) & F.FA3_DEVERR_LENS
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    # fewer heads, narrower latent, no RoPE
    w2 = W.MLAWorkload(name="h16 dl128 dr0", B=2, H=16, Dl=128, Dr=0, T_max=300, softmax_scale=0.1, lens=[300, 200],
                       calib_q_shape=(2, 16, 16, 128), calib_kv_shape=(1, 1, 256, 128))
    a2 = _prepare(w2)
    assert_attn_close(_run(F, w2, *a2), _oracle(w2, *a2), what="h16 dl128 dr0")
    w3 = W.MLAWorkload(name="h128 dl256 dr32", B=2, H=128, Dl=256, Dr=32, T_max=200, softmax_scale=0.1,
                       lens=[200, 129], calib_q_shape=(2, 128, 4, 256), calib_kv_shape=(1, 1, 256, 256))
    a3 = _prepare(w3)
    assert_attn_close(_run(F, w3, *a3), _oracle(w3, *a3), what="h128 dl256 dr32")
    # Dr = 48: three 16-wide RoPE chunks, split 2 / 1 over the pair; the second CTA's
    # RoPE key box reaches past Dr and is zero-filled there
    w4 = W.MLAWorkload(name="h64 dl512 dr48", B=2, H=64, Dl=512, Dr=48, T_max=260, softmax_scale=0.08,
                       lens=[260, 77], calib_q_shape=(2, 64, 4, 512), calib_kv_shape=(1, 1, 256, 512))
    a4 = _prepare(w4)
    assert_attn_close(_run(F, w4, *a4), _oracle(w4, *a4), what="h64 dl512 dr48")


def _oracle_all_rows(w, inp, q_scale, kv_scale, ckv8, lens):
    """Every row of the oracle, one thread per sequence (numpy's matmuls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    def one(b):
        return O.mla_decode(inp.q[b:b + 1], ckv8[b:b + 1], inp.krope[b:b + 1], q_scale, float(kv_scale[0]),
                            lens[b:b + 1], w.softmax_scale)[0]

    with ThreadPoolExecutor(max_workers=max(1, min(w.B, os.cpu_count() or 1))) as ex:
        return np.stack(list(ex.map(one, range(w.B))))


@pytest.mark.slow
def test_dsv3_full_size_all_rows():
    # 32 sequences x 8192 tokens x 128 heads: every output row against the oracle.
    F = fa3()
    w = W.mla_dsv3()
    args = _prepare(w)
    got = _run(F, w, *args)
    ref = _oracle_all_rows(w, *args)
    max_abs, rrms = assert_attn_close(got, ref, what="dsv3 full")
    print(f"mla dsv3 full: max_abs={max_abs:.3e} rel_rms={rrms:.3e}")


@pytest.mark.slow
def test_long_context_variable_lengths_all_rows():
    # 8 sequences of seeded lengths in [1024, 32768], split over many clusters.
    F = fa3()
    w = W.mla_long()
    args = _prepare(w)
    got = _run(F, w, *args)
    ref = _oracle_all_rows(w, *args)
    max_abs, rrms = assert_attn_close(got, ref, what="long mla")
    print(f"mla long full: max_abs={max_abs:.3e} rel_rms={rrms:.3e} lens={args[4].tolist()}")


def test_poisoned_workspace_few_tiles():
    # Fewer tiles than clusters: some clusters own nothing and must not be read back.
    F = fa3()
    w = W.mla_dsv3(B=2, T=256)
    inp, q_scale, kv_scale, ckv8, lens = _prepare(w, lens=[256, 128])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ws = torch.full((F.mla_workspace_size(w.B, w.H, w.Dl, w.T_max),), 0xFF, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        out = F.decode_attn_mla(bf16_dev(inp.q), t(ckv8), bf16_dev(inp.krope), t(q_scale), t(kv_scale), t(lens),
                                w.softmax_scale, workspace=ws)
        assert_attn_close(out.cpu().numpy(), _oracle(w, inp, q_scale, kv_scale, ckv8, lens), what="poisoned ws")


def test_multi_tile_segments():
    # 256 tiles: every cluster walks several tiles, crosses a sequence boundary and
    # hands split sequences to the combine kernel.
    F = fa3()
    w = W.mla_dsv3(B=2, T=8192)
    args = _prepare(w, lens=[8192, 5000])
    got = _run(F, w, *args)
    assert_attn_close(got, _oracle(w, *args), what="multi-tile")


def test_forced_rescales():
    # RoPE keys aligned with each head's RoPE query and growing along the context:
    # the running maximum jumps by more than the lazy-rescale threshold tile after tile.
    F = fa3()
    w = W.mla_dsv3(B=2, T=4096)
    inp, q_scale, kv_scale, ckv8, lens = _prepare(w, lens=[4096, 3000])
    qr = inp.q[:, :, w.Dl:]
    ramp = (np.arange(w.T_max, dtype=np.float32) / 64.0) * 150.0          # about +10 (log2) per tile
    k = qr.mean(axis=1, keepdims=True) / (np.linalg.norm(qr.mean(axis=1), axis=-1)[:, None, None] + 1e-6)
    krope = W.bf16_round((k * ramp[None, :, None] + inp.krope * 0.1).astype(np.float32))
    inp.krope = krope
    got = _run(F, w, inp, q_scale, kv_scale, ckv8, lens)
    assert_attn_close(got, _oracle(w, inp, q_scale, kv_scale, ckv8, lens), what="forced rescales")


def test_stream_order_with_other_kernels_between_calls():
    # The library's kernels are programmatic dependents of the kernel before them:
    # each call must still see the query and lengths that ordinary device copies wrote
    # just before it, and the copies after it must see its finished output.
    F = fa3()
    w = W.mla_dsv3(B=2, T=2048)
    inp, q_scale, kv_scale, ckv8, _ = _prepare(w)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    variants = [(W.bf16_round(inp.q * s), np.array(ls, np.int32))
                for s, ls in ((1.0, [2048, 1500]), (-0.7, [900, 2048]), (1.3, [64, 1]))]
    dq = torch.empty(inp.q.shape, dtype=torch.bfloat16, device="cuda")
    dl = torch.empty(w.B, dtype=torch.int32, device="cuda")
    out = torch.empty(w.B, w.H, w.Dl, dtype=torch.float32, device="cuda")
    ws = torch.empty(F.mla_workspace_size(w.B, w.H, w.Dl, w.T_max), dtype=torch.uint8, device="cuda")
    srcs = [(bf16_dev(q), t(ls)) for q, ls in variants]
    ck, kr, qs, kvs = t(ckv8), bf16_dev(inp.krope), t(q_scale), t(kv_scale)
    keep = []
    torch.cuda.synchronize()
    for (sq, sl) in srcs:
        dq.copy_(sq)
        dl.copy_(sl)
        F.decode_attn_mla(dq, ck, kr, qs, kvs, dl, w.softmax_scale, out=out, workspace=ws)
        keep.append(out.clone())
    torch.cuda.synchronize()
    for (q, ls), got in zip(variants, keep):
        inp.q = q
        assert_attn_close(got.cpu().numpy(), _oracle(w, inp, q_scale, kv_scale, ckv8, ls), what=f"ordered {ls}")


@pytest.mark.parametrize("H", [1, 37, 100])
def test_head_counts_not_a_multiple_of_the_lane_quarter(H):
    # heads >= H are padding rows of the 128-lane tiles: zero query codes, never written out
    F = fa3()
    w = W.MLAWorkload(name=f"h{H} dl512 dr64", B=2, H=H, Dl=512, Dr=64, T_max=333, softmax_scale=0.07,
                      lens=[333, 70], calib_q_shape=(2, H, 4, 512), calib_kv_shape=(1, 1, 256, 512))
    args = _prepare(w)
    assert_attn_close(_run(F, w, *args), _oracle(w, *args), what=f"mla H={H}")
