"""GPU parity of prefill-phase GQA attention (INT8 q/k/v, causal, bf16 output) against the float64 oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_attn_close, fa3
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu


def _case(w):
    inp = W.prefill_inputs(w)
    qs = O.qparams(*O.calibrate(inp.calib_q, w.ratio))
    ks = O.qparams(*O.calibrate(inp.calib_k, w.ratio))
    vs = O.qparams(*O.calibrate(inp.calib_v, w.ratio))
    q8 = O.quantize(inp.q, qs[None, None, :, None])
    k8 = O.quantize(inp.k, ks[None, None, :, None])
    v8 = O.quantize(inp.v, vs[None, None, :, None])
    return q8, k8, v8, qs, ks, vs, np.asarray(w.q_lens, np.int32), np.asarray(w.kv_lens, np.int32)


def _run(F, w, args, err=None, out=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q8, k8, v8, qs, ks, vs, ql, kl = args
    o = F.prefill_attn_gqa(t(q8), t(k8), t(v8), t(qs), t(ks), t(vs), t(ql), t(kl), w.softmax_scale, out=out,
                           dev_err=err)
    torch.cuda.synchronize()
    return o.float().cpu().numpy()


def _check_rows(got, ref, ql, what):
    for b in range(len(ql)):
        if ql[b]:
            assert_attn_close(got[b, :ql[b]], ref[b, :ql[b]], bf16_out=True, what=f"{what} b{b}")
        assert not got[b, ql[b]:].any(), f"{what}: rows past q_lens written"


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (4, 4), (16, 8), (32, 8), (128, 8), (64, 1)])
def test_ragged_with_cached_prefix(Hq, Hkv):
    # group sizes 8, 1, 2, 4, 16, 64; cached prefixes, a sequence with no new rows, ragged tile tails
    F = fa3()
    w = W.prefill_llama70b(B=4, S=200, T=333, Hq=Hq, Hkv=Hkv, q_lens=[200, 37, 0, 129], kv_lens=[333, 37, 5, 300])
    args = _case(w)
    got = _run(F, w, args)
    ref = O.gqa_prefill(*args[:6], args[6], args[7], w.softmax_scale)
    _check_rows(got, ref, args[6], f"prefill G={Hq // Hkv}")


def test_single_row_and_tile_edges():
    F = fa3()
    w = W.prefill_llama70b(B=5, S=130, T=257, q_lens=[1, 1, 128, 129, 130], kv_lens=[1, 257, 128, 256, 257])
    args = _case(w)
    got = _run(F, w, args)
    ref = O.gqa_prefill(*args[:6], args[6], args[7], w.softmax_scale)
    _check_rows(got, ref, args[6], "prefill edges")


def test_bad_lengths_set_the_error_bit_and_skip_the_sequence():
    F = fa3()
    w = W.prefill_llama70b(B=3, S=64, T=64, q_lens=[64, 10, 5], kv_lens=[64, 64, 64])
    args = list(_case(w))
    args[6] = np.array([64, 65, 9], np.int32)       # q_lens > S
    args[7] = np.array([64, 64, 4], np.int32)       # kv_lens < q_lens
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(F, w, args, err=err)
    assert int(err.item()) & F.FA3_DEVERR_LENS
    assert not got[1].any() and not got[2].any()
    ref = O.gqa_prefill(*args[:6], np.array([64, 0, 0]), np.array([64, 64, 64]), w.softmax_scale)
    assert_attn_close(got[0], ref[0], bf16_out=True, what="prefill good sequence")


def test_growing_scores_force_rescales():
    # keys aligned with the queries and growing along the context: the running
    # maximum of late rows jumps by more than the lazy-rescale threshold tile after tile
    F = fa3()
    w = W.prefill_llama70b(B=1, S=512, T=512, Hq=8, Hkv=1)
    q8, k8, v8, qs, ks, vs, ql, kl = _case(w)
    base = np.sign(q8[0, :, :, :].astype(np.int64).sum(axis=(0, 1)))        # [D]
    ramp = np.clip((np.arange(w.T) / 512.0 * 127), 1, 127).astype(np.int64)
    k8 = np.clip(base[None, None, :] * ramp[:, None, None], -127, 127).astype(np.int8)[None]
    q8 = np.broadcast_to(np.clip(base * 100, -127, 127).astype(np.int8), q8.shape).copy()
    qs = np.full_like(qs, 0.02)
    ks = np.full_like(ks, 0.02)
    args = (q8, k8, v8, qs, ks, vs, ql, kl)
    got = _run(F, w, args)
    ref = O.gqa_prefill(*args[:6], ql, kl, w.softmax_scale)
    _check_rows(got, ref, ql, "prefill rescales")


@pytest.mark.slow
def test_llama70b_4096_sampled_rows():
    # S = T = 4096, 64 query heads / 8 KV heads: every head of 40 sampled rows (the
    # first, the last, tile boundaries and random ones) against the oracle; the
    # whole output is finite and no row is missing.
    F = fa3()
    w = W.prefill_llama70b(B=1, S=4096, T=4096)
    args = _case(w)
    got = _run(F, w, args)
    rng = np.random.default_rng(3)
    rows = sorted({0, 1, 127, 128, 129, 2047, 2048, 4095} | set(int(x) for x in rng.integers(0, 4096, 32)))
    ref = O.gqa_prefill(*args[:6], args[6], args[7], w.softmax_scale, rows=[(0, i) for i in rows])
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got[0]).sum(axis=(1, 2)) > 0)
    assert_attn_close(got[0, rows], ref[0, rows], bf16_out=True, what="prefill 4096 sampled rows")
