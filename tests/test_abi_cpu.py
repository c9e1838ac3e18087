"""CPU checks of the C ABI: the library builds, loads, exports every declared symbol,
and its host-side validation rejects bad arguments before touching a GPU."""
import ctypes

import pytest

from helpers import fa3, header_functions

EINVAL, ERANGE, EWORKSPACE = 1, 2, 4
FAKE = ctypes.c_void_p(4096)   # never dereferenced: validation fails first


@pytest.fixture(scope="module")
def L():
    return fa3().lib()


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    assert L.fa3_version() == 100
    for s in range(6):
        assert L.fa3_status_string(s).startswith(b"FA3")


def test_calibrate_validation(L):
    ws = L.fa3_calibrate_workspace_size(4)
    assert ws == 4 * 65536 * 4 + 4 * 16 + 4 * 2 * 16384 * 2   # key counts, tail state, tail-key lists
    args = lambda **k: dict(dict(x=FAKE, B=2, H=4, L=64, sb=256, sh=64, ratio=0.9999, mn=FAKE, mx=FAKE,
                                 ws=FAKE, wsb=ws), **k)
    call = lambda a: L.fa3_calibrate_perhead(a["x"], a["B"], a["H"], a["L"], a["sb"], a["sh"], a["ratio"],
                                             a["mn"], a["mx"], a["ws"], a["wsb"], None)
    assert call(args(x=None)) == EINVAL
    assert call(args(mn=None)) == EINVAL
    for r in (0.0, -1.0, 1.5, float("nan")):
        assert call(args(ratio=r)) == EINVAL
    assert call(args(B=0)) == EINVAL
    assert call(args(L=1 << 31, B=4)) == ERANGE        # N >= 2^32
    assert call(args(wsb=ws - 1)) == EWORKSPACE
    assert call(args(ws=None)) == EWORKSPACE


def test_qparams_and_append_validation(L):
    assert L.fa3_qparams(None, FAKE, FAKE, 4, None) == EINVAL
    assert L.fa3_qparams(FAKE, FAKE, FAKE, 0, None) == EINVAL
    q = lambda **k: L.fa3_quantize_append(k.get("kv", FAKE), FAKE, FAKE, FAKE, k.get("B", 2), k.get("T_new", 4), 1,
                                          512, k.get("T_max", 16), k.get("rs", None), k.get("rc", None),
                                          k.get("Dr", 0), None, None)
    assert q(kv=None) == EINVAL
    assert q(T_new=17) == EINVAL
    assert q(rs=FAKE) == EINVAL                         # source without destination
    assert q(rs=FAKE, rc=FAKE, Dr=0) == EINVAL


def test_mla_validation(L):
    call = lambda H=128, Dl=512, Dr=64, q=FAKE, sc=0.07: L.fa3_decode_attn_mla(
        q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, H, Dl, Dr, 64, sc, FAKE, 1 << 30, None, None)
    assert call(q=None) == EINVAL
    assert call(sc=0.0) == EINVAL
    assert call(H=129) == ERANGE
    assert call(Dl=96) == ERANGE
    assert call(Dr=24) == ERANGE
    assert call(Dr=80) == ERANGE


def test_gqa_validation(L):
    call = lambda Hq=64, Hkv=8, D=128, k=FAKE: L.fa3_decode_attn_gqa(
        FAKE, k, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, Hq, Hkv, D, 64, 0.09, FAKE, 1 << 30, None, None)
    assert call(k=None) == EINVAL
    assert call(Hq=60) == EINVAL          # not a multiple of Hkv
    assert call(D=64) == ERANGE
    assert call(Hq=128, Hkv=8) == ERANGE  # 16 query heads per KV head


def test_range_merge_validation(L):
    call = lambda mins=FAKE, R=2, H=4: L.fa3_range_merge(mins, FAKE, R, H, FAKE, FAKE, None)
    assert call(mins=None) == EINVAL
    assert call(R=0) == EINVAL
    assert call(H=0) == EINVAL


def test_channel_validation(L):
    q = lambda mn=FAKE, n=8: L.fa3_qparams_channel(mn, FAKE, n, 1, FAKE, FAKE, None)
    assert q(mn=None) == EINVAL and q(n=0) == EINVAL
    a = lambda off=FAKE, asym=1, D=128: L.fa3_quantize_append_channel(FAKE, FAKE, off, asym, FAKE, FAKE, 2, 4, 8, D,
                                                                      64, None, None)
    assert a(off=None) == EINVAL             # asymmetric without offsets
    assert a(D=12) == ERANGE                 # not a multiple of 8
    c = lambda ratio=0.9999, S=1000: L.fa3_calibrate_perchannel(FAKE, 3, 4, S, 40, 1, 1, 1, ratio, FAKE, FAKE, None)
    assert c(ratio=0.0) == EINVAL
    assert c(ratio=0.9, S=1000) == ERANGE    # 301 window starts > 32
    g = lambda ko=FAKE, D=128: L.fa3_decode_attn_gqa_channel(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ko, FAKE, FAKE,
                                                             FAKE, FAKE, 2, 64, 8, D, 64, 0.09, FAKE, 1 << 30,
                                                             None, None)
    assert g(ko=None) == EINVAL
    assert g(D=64) == ERANGE


def test_calibrate_f32_validation(L):
    ws = L.fa3_calibrate_f32_workspace_size(4)
    call = lambda ratio=0.9999, N=1000, wsb=ws: L.fa3_calibrate_perhead_f32(FAKE, 1, 4, N, 0, N, ratio, FAKE, FAKE,
                                                                           FAKE, wsb, None, None)
    assert call(ratio=0.0) == EINVAL
    assert call(ratio=0.9, N=100000) == ERANGE     # 10001 window starts > 4096
    assert call(wsb=ws - 1) == EWORKSPACE


def test_prefill_validation(L):
    UNALIGNED = ctypes.c_void_p(4096 + 8)
    call = lambda Hq=64, Hkv=8, D=128, q=FAKE, sc=0.09, out=FAKE, S=64: L.fa3_prefill_attn_gqa(
        q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, out, 2, S, 64, Hq, Hkv, D, sc, None, None)
    assert call(q=None) == EINVAL
    assert call(out=None) == EINVAL
    assert call(S=0) == EINVAL
    assert call(sc=float("nan")) == EINVAL
    assert call(Hq=60) == EINVAL          # not a multiple of Hkv
    assert call(D=64) == ERANGE
    assert call(Hq=24, Hkv=8) == ERANGE   # 3 query heads per KV head do not divide 128 rows
    assert call(q=UNALIGNED) == ERANGE


def test_paged_validation(L):
    mla = lambda bt=FAKE, npg=8, ps=64, mp=4: L.fa3_decode_attn_mla_paged(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, bt, FAKE, 2, 128, 512, 64, npg, ps, mp, 0.07, FAKE, 1 << 30, None, None)
    assert mla(bt=None) == EINVAL
    assert mla(npg=0) == EINVAL
    assert mla(ps=48) == ERANGE            # a 64-token tile would span two pages
    assert mla(npg=1 << 26, ps=64) == ERANGE   # pool rows >= 2^31
    gqa = lambda bt=FAKE, npg=8, ps=16, mp=4: L.fa3_decode_attn_gqa_paged(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, bt, FAKE, 2, 64, 8, 128, npg, ps, mp, 0.09, FAKE, 1 << 30,
        None, None)
    assert gqa(bt=None) == EINVAL
    assert gqa(mp=0) == EINVAL
    assert gqa(ps=24) == ERANGE            # a 16-token step would span two pages
    app = lambda bt=FAKE, ps=16, mp=4, T_new=4: L.fa3_quantize_append_paged(
        FAKE, FAKE, FAKE, bt, FAKE, 2, T_new, 1, 512, 8, ps, mp, None, None, 0, None, None)
    assert app(bt=None) == EINVAL
    assert app(ps=0) == EINVAL
    assert app(T_new=65) == EINVAL         # more new rows than max_pages * page_size


def test_kernel_timing_hook_validation(L):
    # exactly one event is an error; none turns the hook off (no CUDA call either way)
    assert L.fa3_set_kernel_timing(None, FAKE) == EINVAL
    assert L.fa3_set_kernel_timing(FAKE, None) == EINVAL
    assert L.fa3_set_kernel_timing(None, None) == 0


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    # No fallback: with the shared library absent every call raises.
    from int8_head_kv_gb300 import fa3 as F
    monkeypatch.setattr(F, "_lib", None)
    monkeypatch.setattr(F, "library_path", lambda: str(tmp_path / "missing" / "libfa3.so"))
    with pytest.raises(RuntimeError, match="not built"):
        F.lib()
    with pytest.raises(RuntimeError, match="not built"):
        F.mla_workspace_size(1, 1, 64, 64)


def test_product_sources_never_reach_the_oracle():
    # The package (binding, build script, kernels) neither imports nor names the
    # oracle; the oracle is test infrastructure only.
    import glob
    import os
    from helpers import ROOT
    files = glob.glob(os.path.join(ROOT, "int8_head_kv_gb300", "**", "*.*"), recursive=True)
    files = [f for f in files if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp"))]
    assert len(files) >= 6
    for f in files:
        src = open(f, encoding="utf-8").read()
        assert "oracle" not in src, f


def test_workspace_cache_is_per_stream(monkeypatch):
    # One scratch buffer per (call kind, device, stream); a larger request replaces it.
    import contextlib
    import torch
    from int8_head_kv_gb300 import fa3 as F

    class FakeStream:
        def __init__(self, h):
            self.cuda_stream = h

    from collections import OrderedDict
    cur = FakeStream(11)
    monkeypatch.setattr(F, "_ws_cache", OrderedDict())
    monkeypatch.setattr(torch.cuda, "current_stream", lambda dev=None: cur)
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    cpu = torch.device("cpu")
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    assert F._workspace("mla", 0, cpu) is None
    a = F._workspace("mla", 64, cpu)
    assert a is F._workspace("mla", 32, cpu)                      # same stream: reused
    b = F._workspace("mla", 64, cpu, stream=FakeStream(12))
    assert b is not a                                             # another stream: its own buffer
    c = F._workspace("gqa", 64, cpu)
    assert c is not a                                             # another call kind
    d = F._workspace("mla", 128, cpu)
    assert d is not a and d.numel() == 128 and F._workspace("mla", 100, cpu) is d
    z = F._workspace("calib", 16, cpu, zero=True)
    assert not z.any()
    # at most _WS_PER_KIND streams per (call kind, device): the least recently used goes
    for h in range(20, 20 + F._WS_PER_KIND):
        F._workspace("mla", 64, cpu, stream=FakeStream(h))
    mla_streams = [k[2] for k in F._ws_cache if k[0] == "mla"]
    assert len(mla_streams) == F._WS_PER_KIND and 11 not in mla_streams and 12 not in mla_streams
    assert ("gqa", 0, 11) in F._ws_cache and ("calib", 0, 11) in F._ws_cache


def test_failed_calibration_drops_its_cached_workspace(monkeypatch):
    # After an error the key-count table may not be clear again: the binding must not
    # hand the cached buffer to the next calibration on that stream.
    import contextlib
    from collections import OrderedDict
    import torch
    from int8_head_kv_gb300 import fa3 as F

    class FakeStream:
        cuda_stream = 11

    class FakeLib:
        def fa3_calibrate_workspace_size(self, H):
            return 64

        def fa3_calibrate_perhead(self, *a):
            return 3                                    # FA3_ECUDA

        def fa3_status_string(self, s):
            return b"FA3_ECUDA"

    monkeypatch.setattr(F, "_ws_cache", OrderedDict())
    monkeypatch.setattr(F, "lib", lambda: FakeLib())
    monkeypatch.setattr(F, "_need", lambda *a: None)
    monkeypatch.setattr(F, "_need_contig", lambda *a: None)
    monkeypatch.setattr(F, "_stream", lambda s=None: None)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda dev=None: FakeStream())
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    x = torch.zeros(2, 8, dtype=torch.bfloat16)
    mn, mx = torch.zeros(2), torch.zeros(2)
    with pytest.raises(F.FA3Error):
        F.calibrate_perhead(x, 0.9, mn, mx)
    assert ("calib", 0, 11) not in F._ws_cache
