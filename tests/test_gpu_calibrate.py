"""GPU parity of the per-head Recall-Window calibration: bit-exact min/max against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from helpers import bf16_dev, fa3
from oracle import fa3_oracle as O

pytestmark = pytest.mark.gpu


def _gpu_calibrate(F, batches, ratio, H):
    mn = torch.full((H,), float("inf"), device="cuda")
    mx = torch.full((H,), float("-inf"), device="cuda")
    for x in batches:
        F.calibrate_perhead(bf16_dev(x), ratio, mn, mx)
    torch.cuda.synchronize()
    return mn.cpu().numpy(), mx.cpu().numpy()


def _bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def test_tiny_mla_calibration_bit_exact():
    F = fa3()
    w = W.mla_tiny()
    inp = W.mla_inputs(w)
    for batches in (inp.calib_q, inp.calib_kv):
        H = batches[0].shape[1]
        gmn, gmx = _gpu_calibrate(F, batches, w.ratio, H)
        omn, omx = O.calibrate(batches, w.ratio)
        assert np.array_equal(_bits(gmn), _bits(omn)) and np.array_equal(_bits(gmx), _bits(omx))
        sc = F.qparams(torch.from_numpy(gmn).cuda(), torch.from_numpy(gmx).cuda()).cpu().numpy()
        assert np.array_equal(_bits(sc), _bits(O.qparams(omn, omx)))


@pytest.mark.parametrize("ratio", [1.0, 0.9999, 0.99, 0.5, 0.1, 1e-9])
def test_ratios_and_ragged_chunks(ratio):
    # N = 3 * 40000 = 120000 spans two 65528-value chunks with a ragged tail.
    F = fa3()
    rng = np.random.default_rng(7)
    x = W.bf16_round((rng.standard_t(3, (3, 5, 200, 200)) * rng.uniform(0.05, 20, (1, 5, 1, 1))).astype(np.float32))
    gmn, gmx = _gpu_calibrate(F, [x], ratio, 5)
    omn, omx = O.calibrate([x], ratio)
    assert np.array_equal(_bits(gmn), _bits(omn)) and np.array_equal(_bits(gmx), _bits(omx))


def test_degenerate_heads():
    F = fa3()
    rng = np.random.default_rng(8)
    H = 6
    x = np.zeros((2, H, 16, 24), np.float32)
    x[:, 0] = 0.75                                            # all equal
    x[:, 1] = rng.integers(-2, 3, (2, 16, 24))                # heavy duplicates
    x[:, 2] = -np.abs(rng.standard_normal((2, 16, 24)))       # negative only
    x[:, 3] = np.where(rng.random((2, 16, 24)) < 0.5, 0.0, -0.0)  # signed zeros
    x[:, 4] = rng.standard_normal((2, 16, 24)) * 1e-30        # tiny magnitudes
    x[:, 5] = rng.standard_normal((2, 16, 24)) * 3e30         # huge magnitudes
    x = W.bf16_round(x)
    for ratio in (1.0, 0.9, 0.5):
        gmn, gmx = _gpu_calibrate(F, [x], ratio, H)
        omn, omx = O.calibrate([x], ratio)
        assert np.array_equal(_bits(gmn), _bits(omn)), (ratio, gmn, omn)
        assert np.array_equal(_bits(gmx), _bits(omx)), (ratio, gmx, omx)


def test_strided_layout_scalar_path_and_workspace_reuse():
    F = fa3()
    rng = np.random.default_rng(9)
    # L = 7 * 5 = 35 is not a multiple of 8: scalar loads.
    x = W.bf16_round(rng.standard_normal((3, 4, 7, 5)).astype(np.float32) * 2)
    big = torch.zeros(3, 6, 7, 5, dtype=torch.bfloat16, device="cuda")
    big[:, 1:5] = bf16_dev(x)
    view = big[:, 1:5]                                        # strided in H and B
    omn, omx = O.calibrate([x], 0.9)
    for _ in range(2):                                        # the workspace comes back clean
        mn = torch.full((4,), float("inf"), device="cuda")
        mx = torch.full((4,), float("-inf"), device="cuda")
        F.calibrate_perhead(view, 0.9, mn, mx)
        assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn))
        assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx))


def test_resume_from_saved_range():
    F = fa3()
    w = W.mla_tiny()
    b = W.mla_inputs(w).calib_q
    omn, omx = O.calibrate(b, w.ratio)
    mn0, mx0 = O.calibrate(b[:1], w.ratio)
    mn = torch.from_numpy(mn0.copy()).cuda()
    mx = torch.from_numpy(mx0.copy()).cuda()
    for x in b[1:]:
        F.calibrate_perhead(bf16_dev(x), w.ratio, mn, mx)
    assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn)) and np.array_equal(_bits(mx.cpu().numpy()), _bits(omx))


@pytest.mark.slow
def test_full_size_calibration_sampled_heads():
    # One (4, 128, 2048, 192) batch on the GPU; eight heads recomputed by the oracle.
    F = fa3()
    w = W.calib_scale()
    x = torch.empty(w.B, w.H, w.S, w.D, dtype=torch.bfloat16, device="cuda")
    for h in range(w.H):
        x[:, h] = bf16_dev(W.calib_head(w, 0, h))
    mn = torch.full((w.H,), float("inf"), device="cuda")
    mx = torch.full((w.H,), float("-inf"), device="cuda")
    F.calibrate_perhead(x, w.ratio, mn, mx)
    gmn, gmx = mn.cpu().numpy(), mx.cpu().numpy()
    for h in (0, 1, 17, 42, 63, 64, 100, 127):
        lo, hi = O.recall_window(W.calib_head(w, 0, h), w.ratio)
        assert (gmn[h], gmx[h]) == (np.float32(lo), np.float32(hi)), h


def _sampled_units(units, n_samples=512):
    # the strided sample the tail thresholds are drawn from (16-byte groups or values)
    return sorted({g * units // n_samples for g in range(n_samples)})


@pytest.mark.parametrize("vec", [True, False])
def test_thin_tails_fall_back_to_full_count(vec):
    # Plant one extreme value into sampled units of head 0 (25 groups of 8 values, or
    # 40 single values, more than the sample's tail rank of 16 or 5): the sample's
    # tail order statistic then falls on that value, whose count (200 or 40) is below
    # the 1574 smallest values a window can start from, so the tail-only count must
    # be rejected and the head counted again in full.  Head 1 is left as is.
    F = fa3()
    rng = np.random.default_rng(11)
    H, N = 2, 4 * 2048 * 192
    ratio = 0.999                                  # N - target_num + 1 = 1574 window starts
    x = W.bf16_round(rng.standard_normal((H, N)).astype(np.float32))
    per, n_plant = (8, 25) if vec else (1, 40)
    for u in _sampled_units(N // per)[:n_plant]:
        x[0, u * per:u * per + per] = -600.0
    if vec:
        xd = bf16_dev(x)
    else:
        pad = np.zeros((H, N + 1), np.float32)     # odd row stride: the scalar path
        pad[:, :N] = x
        xd = bf16_dev(pad)[:, :N]
    omn, omx = O.calibrate([x.reshape(1, H, 1, N)], ratio)
    for _ in range(2):                             # the workspace is left clean for the next call
        mn = torch.full((H,), float("inf"), device="cuda")
        mx = torch.full((H,), float("-inf"), device="cuda")
        F.calibrate_perhead(xd, ratio, mn, mx)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn))
        assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx))
