"""GPU parity of the per-head Recall-Window calibration: bit-exact min/max against the oracle."""
import os

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


def _exact_width_heads(N, t):
    """Two heads whose first two windows have lengths 1 + 2^-120 and 1 (equal in
    float64): the exact reading must pick the second, (0, 1).  Head 0 holds
    t - 3 copies of 0.5 between the ends and 2^100 after them; head 1
    repeats the hand-worked golden example's values to fill N."""
    a = np.empty(N, np.float32)
    a[0], a[1], a[2:t - 1], a[t - 1:t + 1], a[t + 1:] = -2.0 ** -120, 0.0, 0.5, 1.0, 2.0 ** 100
    b = np.tile(np.array([1.0, -2.0 ** -120, 1.0, 0.0], np.float32), N // 4)
    return np.stack([a, b])


@pytest.mark.parametrize("ratio", ["tail", "full"])
def test_exact_window_widths_mixed_magnitudes(ratio):
    # Window lengths that tie after rounding to float64 but not exactly, on the
    # tail path (few windows) and on the full-histogram path (many windows), plus
    # random heads spanning ~130 binades.
    F = fa3()
    N = 98304
    r = (N - 0.5) / N if ratio == "tail" else 0.5
    t = O.target_num(r, N)
    rng = np.random.default_rng(21)
    x = np.concatenate([_exact_width_heads(N, t)[:1] if ratio == "tail" else _exact_width_heads(N, t),
                        np.stack([W.mixed_magnitude_head(rng, N) for _ in range(3)])])
    H = x.shape[0]
    gmn, gmx = _gpu_calibrate(F, [x.reshape(1, H, 1, N)], r, H)
    omn, omx = O.calibrate([x.reshape(1, H, 1, N)], r)
    assert (float(omn[0]), float(omx[0])) == (0.0, 1.0)
    assert np.array_equal(_bits(gmn), _bits(omn)), (gmn, omn)
    assert np.array_equal(_bits(gmx), _bits(omx)), (gmx, omx)


@pytest.mark.slow
def test_full_size_calibration_all_heads_four_batches():
    # The (4, 128, 2048, 192) workload: four batches with the running min/max, every
    # head compared bit for bit after every batch (the oracle runs one thread per head).
    from concurrent.futures import ThreadPoolExecutor
    F = fa3()
    w = W.calib_scale()
    x = torch.empty(w.B, w.H, w.S, w.D, dtype=torch.bfloat16, device="cuda")
    mn = torch.full((w.H,), float("inf"), device="cuda")
    mx = torch.full((w.H,), float("-inf"), device="cuda")
    omn, omx = O.init_range(w.H)

    def head(kh):
        v = W.calib_head(w, *kh)
        return v, O.recall_window(v, w.ratio)

    with ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1))) as ex:
        for k in range(w.batches):
            lo, hi = np.empty(w.H, np.float32), np.empty(w.H, np.float32)
            for h, (v, (a, b)) in enumerate(ex.map(head, [(k, h) for h in range(w.H)])):
                x[:, h] = bf16_dev(v)
                lo[h], hi[h] = a, b
            F.calibrate_perhead(x, w.ratio, mn, mx)
            O.accumulate(omn, omx, lo, hi)
            torch.cuda.synchronize()
            assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn)), k
            assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx)), k
    sc = F.qparams(mn, mx).cpu().numpy()
    assert np.array_equal(_bits(sc), _bits(O.qparams(omn, omx)))


def _sample_runs(units, runs=16, run_len=128):
    # the tail thresholds' sample: 16 runs of 128 consecutive 16-byte groups, run r
    # from group r * units // 16; sampling thread 16 r + (w % 16) holds group w of run r
    return [[(r * units // runs + w) % units for w in range(run_len)] for r in range(runs)]


@pytest.mark.parametrize("vec", [True, False])
def test_thin_tails_fall_back_to_full_count(vec):
    # Plant one extreme value into the first sixteen sampled groups of runs 0..3 of
    # head 0 (512 values, one group in each of 64 sampling threads, more than the
    # sample rank of 53): the low threshold then falls on that value, whose count
    # (512) is below the 1574 smallest values a window can start from, so the tail
    # lists must be rejected and the head counted again in full.  Head 1 is left
    # as is.  With an odd row stride (vec False) the input takes the histogram path
    # instead; the result is the same either way.
    F = fa3()
    rng = np.random.default_rng(11)
    H, N = 2, 4 * 2048 * 192
    ratio = 0.999                                  # N - target_num + 1 = 1574 window starts
    x = W.bf16_round(rng.standard_normal((H, N)).astype(np.float32))
    for run in _sample_runs(N // 8)[:4]:
        for u in run[:16]:
            x[0, u * 8:u * 8 + 8] = -600.0
    if vec:
        xd = bf16_dev(x)
    else:
        pad = np.zeros((H, N + 1), np.float32)     # odd row stride: the histogram path
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


def test_tail_list_path_every_branch():
    # One (H, N) batch at ratio 0.9999 (158 window starts, sample rank 8), one head
    # per branch of the tail-list path (the low threshold sits near -26 for the
    # Student-t heads, so every planted -50 lands in the low list):
    #   0  ordinary Student-t head: decided from its lists;
    #   1  3000 copies of -50 inside one 64 KB piece of the row: one CTA stages most
    #      of a list, still decided from the lists;
    #   2  20000 copies of -50 spread over the row: no CTA stages too many, but the
    #      head's low list overflows its capacity, so the head is counted in full;
    #   3  a constant head: the sample's thresholds meet (degenerate), full count;
    #   4  negative values only, with a high tail of one repeated value;
    #   5  12000 copies of -50 inside one piece: one CTA meets more keys than it can
    #      stage, so the head is counted in full.
    F = fa3()
    rng = np.random.default_rng(12)
    H, N = 6, 4 * 2048 * 192
    ratio = 0.9999
    x = (rng.standard_t(3, (H, N)) * 2.0).astype(np.float32)
    x[1, 3 * 32768 + 100:3 * 32768 + 3100] = -50.0
    x[2, np.linspace(0, N - 1, 20000).astype(np.int64)] = -50.0
    x[3] = 1.5
    x[4] = -np.abs(x[4]) - 1.0
    x[4, rng.choice(N, 3000, replace=False)] = -0.5
    x[5, 5 * 32768 + 100:5 * 32768 + 12100] = -50.0
    x = W.bf16_round(x)
    omn, omx = O.calibrate([x.reshape(1, H, 1, N)], ratio)
    xd = bf16_dev(x)
    for _ in range(2):
        mn = torch.full((H,), float("inf"), device="cuda")
        mx = torch.full((H,), float("-inf"), device="cuda")
        F.calibrate_perhead(xd, ratio, mn, mx)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn)), (mn.cpu().numpy(), omn)
        assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx)), (mx.cpu().numpy(), omx)


def test_workspace_reused_across_head_counts():
    # One caller-owned workspace, sized for the largest H, serves calls with other
    # head counts and both paths (tail lists at ratio 0.9999, the full histogram at
    # 0.5); the per-H layout moves, so every call must leave it all zero.
    F = fa3()
    rng = np.random.default_rng(13)
    ws = torch.zeros(F.calibrate_workspace_size(8), dtype=torch.uint8, device="cuda")
    for H, ratio in ((8, 0.9999), (3, 0.9999), (5, 0.5), (6, 0.9999), (2, 0.5)):
        x = W.bf16_round((rng.standard_t(3, (2, H, 256, 128)) * rng.uniform(0.1, 10, (1, H, 1, 1)))
                         .astype(np.float32))
        mn = torch.full((H,), float("inf"), device="cuda")
        mx = torch.full((H,), float("-inf"), device="cuda")
        F.calibrate_perhead(bf16_dev(x), ratio, mn, mx, workspace=ws)
        omn, omx = O.calibrate([x], ratio)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn)), (H, ratio)
        assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx)), (H, ratio)
        assert int(torch.count_nonzero(ws)) == 0, (H, ratio)


def test_range_merge_matches_step_3_in_any_split():
    # R ranges folded into the running range in one call: the same bits as step 3
    # applied batch by batch (signed zeros ordered, infinities kept).
    F = fa3()
    rng = np.random.default_rng(31)
    R, H = 5, 300
    mins = rng.standard_normal((R, H)).astype(np.float32)
    maxs = rng.standard_normal((R, H)).astype(np.float32)
    mins[:, :8] = np.array([0.0, -0.0, 0.0, -0.0, np.inf, -np.inf, 1.0, -1.0], np.float32)
    maxs[:, :8] = np.array([-0.0, 0.0, -0.0, 0.0, -np.inf, np.inf, -1.0, 1.0], np.float32)
    mins[1, :4] = np.array([-0.0, 0.0, 0.0, -0.0], np.float32)
    mn0, mx0 = O.init_range(H)
    mn0[10:20] = -0.5
    mx0[10:20] = 0.5
    omn, omx = mn0.copy(), mx0.copy()
    for r in range(R):
        O.accumulate(omn, omx, mins[r], maxs[r])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    mn, mx = t(mn0), t(mx0)
    F.range_merge(t(mins), t(maxs), mn, mx)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn))
    assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx))


def test_batches_split_over_shards_then_merged_equal_one_pass():
    # What calibrate_perhead_sharded does on each rank, with the ranks' shares
    # calibrated one after another on this GPU: local ranges, then one merge.
    F = fa3()
    w = W.mla_tiny()
    batches = W.mla_inputs(w).calib_q
    omn, omx = O.calibrate(batches, w.ratio)
    shards = [batches[0::2], batches[1::2]]
    locs = [_gpu_calibrate(F, sh, w.ratio, w.H) for sh in shards]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    mn = torch.full((w.H,), float("inf"), device="cuda")
    mx = torch.full((w.H,), float("-inf"), device="cuda")
    F.range_merge(t(np.stack([l[0] for l in locs])), t(np.stack([l[1] for l in locs])), mn, mx)
    assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn))
    assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx))


# ------------------------------------------------------------------ float32 input
def _f32_heads(rng, H, N):
    x = np.empty((H, N), np.float32)
    x[0] = rng.standard_normal(N) * 3
    x[1] = rng.standard_t(3, N) * 0.01
    x[2] = rng.integers(-3, 4, N)                                  # heavy duplicates
    x[3] = 0.625                                                   # constant
    x[4] = np.where(rng.random(N) < 0.5, 0.0, -0.0)                # signed zeros
    x[5] = np.ldexp(rng.standard_normal(N), rng.integers(-120, 100, N)).astype(np.float32)   # ~220 binades
    x[6] = rng.standard_normal(N).astype(np.float32) * 1e-30 + 1.0  # fp32 detail below bf16's
    return x


@pytest.mark.parametrize("ratio", [1.0, 0.9999, 0.999, 0.99])
def test_float32_calibration_bit_exact(ratio):
    # (B, H, L) = (3, 7, 40000) per batch: N = 120000 values per head; 1 .. 1201 window starts
    F = fa3()
    rng = np.random.default_rng(51)
    B, H, L = 3, 7, 40000
    batches = [np.stack([_f32_heads(rng, H, L) for _ in range(B)]) for _ in range(2)]   # (B, H, L)
    omn, omx = O.init_range(H)
    for x in batches:
        for h in range(H):
            lo, hi = O.recall_window(x[:, h].reshape(-1), ratio)
            O.accumulate(omn[h:h + 1], omx[h:h + 1], np.float32([lo]), np.float32([hi]))
    mn = torch.full((H,), float("inf"), device="cuda")
    mx = torch.full((H,), float("-inf"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k, x in enumerate(batches):
        if k == 0:                                     # a strided view: (B, H) rows inside a larger array
            big = torch.zeros(B, H + 2, 1, L, dtype=torch.float32, device="cuda")
            big[:, 1:H + 1, 0] = torch.from_numpy(x).cuda()
            xd = big[:, 1:H + 1]
        else:
            xd = torch.from_numpy(x).cuda().reshape(B, H, 1, L)
        F.calibrate_perhead_f32(xd, ratio, mn, mx, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_bits(mn.cpu().numpy()), _bits(omn)), (mn.cpu().numpy(), omn)
    assert np.array_equal(_bits(mx.cpu().numpy()), _bits(omx)), (mx.cpu().numpy(), omx)


def test_float32_input_of_bf16_values_matches_the_bf16_path():
    F = fa3()
    w = W.mla_tiny()
    batches = W.mla_inputs(w).calib_q
    g16 = _gpu_calibrate(F, batches, w.ratio, w.H)
    mn = torch.full((w.H,), float("inf"), device="cuda")
    mx = torch.full((w.H,), float("-inf"), device="cuda")
    for x in batches:
        F.calibrate_perhead_f32(torch.from_numpy(np.ascontiguousarray(x)).cuda(), w.ratio, mn, mx)
    assert np.array_equal(_bits(mn.cpu().numpy()), _bits(g16[0]))
    assert np.array_equal(_bits(mx.cpu().numpy()), _bits(g16[1]))
