"""The allocation-free GQA decode entry point, called through the C ABI.

Callers that cannot allocate device memory while they run attention (inside an
allocator callback, under an ahead-of-time memory plan, or where allocation
after start-up is forbidden) use fa3_decode_attn_gqa_noalloc, whose split-K
scratch is a fixed array inside the library.  Its output must match the
workspace-taking entry point on two calls in a row, and the split plan (at most
one wave of resident CTAs) must keep every size within its fixed scratch.  The
two entry points run the same kernels with the same split plan, so their
outputs must be equal bit for bit; both are also held to the oracle's gate.
This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_attn_close, fa3
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu

STATIC_SCRATCH = 8 << 20
P, I, F32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


def _entry(L):
    fn = L.fa3_decode_attn_gqa_noalloc
    fn.restype = I
    fn.argtypes = [P] * 8 + [I] * 5 + [F32, P, P]
    return fn


def test_noalloc_matches_workspace_entry_point_twice():
    F = fa3()
    fn = _entry(F.lib())
    w = W.gqa_llama70b(B=16, T=4096)
    inp = W.gqa_inputs(w)
    qs = O.qparams(*O.calibrate(inp.calib_q, w.ratio))
    ks = O.qparams(*O.calibrate(inp.calib_k, w.ratio))
    vs = O.qparams(*O.calibrate(inp.calib_v, w.ratio))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q8, k8, v8 = (t(O.quantize(inp.q, qs[None, :, None])), t(O.quantize(inp.k, ks[None, None, :, None])),
                  t(O.quantize(inp.v, vs[None, None, :, None])))
    qs_d, ks_d, vs_d = t(qs), t(ks), t(vs)
    lens = t(np.array([4096, 1, 2049, 4000] * 4, np.int32))
    assert 0 < F.gqa_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.T_max) <= STATIC_SCRATCH   # the scratch is used
    ref = F.decode_attn_gqa(q8, k8, v8, qs_d, ks_d, vs_d, lens, w.softmax_scale)
    oracle = O.gqa_decode(O.quantize(inp.q, qs[None, :, None]), O.quantize(inp.k, ks[None, None, :, None]),
                          O.quantize(inp.v, vs[None, None, :, None]), qs, ks, vs, lens.cpu().numpy(),
                          w.softmax_scale)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.empty(w.B, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
        st = fn(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), qs_d.data_ptr(), ks_d.data_ptr(), vs_d.data_ptr(),
                lens.data_ptr(), out.data_ptr(), w.B, w.Hq, w.Hkv, w.D, w.T_max, w.softmax_scale, None, stream)
        assert st == 0, F.lib().fa3_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert_attn_close(out.float().cpu().numpy(), oracle, bf16_out=True, what="no-alloc gqa")


def test_split_plan_keeps_partials_within_the_fixed_scratch():
    # Partials take one 4 KB block per (sequence, KV head, split); the plan never
    # makes more blocks than one wave of resident CTAs, far below 8 MiB.
    F = fa3()
    for B in (1, 2, 7, 16, 57, 128, 137, 1024):
        for Hkv in (1, 2, 8):
            for T in (64, 1000, 8192, 131072):
                Hq = 8 * Hkv
                assert F.gqa_workspace_size(B, Hq, Hkv, 128, T) <= STATIC_SCRATCH, (B, Hkv, T)
