"""Pins for the FP8 (E4M3) state quantize-dequantize oracle (CPU only): the format's value
set against its definition's landmarks and torch's float8_e4m3fn, round-to-nearest-even at
every midpoint, saturation, the per-tile scale (amax maps to +-448 exactly), the zero tile,
partial value tiles, and idempotence."""
import numpy as np
import pytest
import torch

from oracle import fp8_qdq as Q


def test_value_set_landmarks():
    v = Q.e4m3_values()
    pos = v[v > 0]
    assert len(v) == 253            # 256 codes - 2 NaNs - one duplicate zero
    assert pos.max() == 448.0 and pos.min() == 2.0 ** -9
    assert 2.0 ** -6 in pos and 1.0 in pos and 1.125 in pos and 240.0 in pos
    assert 480.0 not in pos         # S.1111.111 is NaN, not 480


def test_value_set_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tv = np.unique(tv[np.isfinite(tv)])
    np.testing.assert_array_equal(tv, Q.e4m3_values())


def test_midpoints_round_to_even():
    pos = Q.e4m3_values()
    pos = pos[pos >= 0]
    mids = (pos[:-1] + pos[1:]) / 2.0
    got = Q.round_e4m3(mids)
    # the neighbour whose mantissa field is even: one of each adjacent pair
    for m, g, lo, hi in zip(mids, got, pos[:-1], pos[1:]):
        assert g in (lo, hi)
    # torch's cast rounds to nearest even as well
    ref = torch.from_numpy(mids).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(Q.round_e4m3(-mids), -ref)


def test_random_values_match_torch_and_saturate():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x.astype(np.float64)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(Q.round_e4m3(x), ref)
    assert Q.round_e4m3(np.array([1000.0, -1e9, 460.0]))[0] == 448.0
    np.testing.assert_array_equal(Q.round_e4m3(np.array([1000.0, -1e9, 460.0])), [448.0, -448.0, 448.0])


def test_tiles_scale_zero_tile_and_partial_tile():
    rng = np.random.default_rng(1)
    st = rng.standard_normal((2, 3, 8, 10)).astype(np.float32)    # [N, H, Dk, Dv]
    st[1, 2, :, :4] = 0.0                                          # an all-zero tile
    out = Q.state_fp8_qdq(st, block_v=4)                           # tiles [0,4) [4,8) [8,10)
    assert out.dtype == np.float32
    np.testing.assert_array_equal(out[1, 2, :, :4], 0.0)
    for v0 in (0, 4, 8):
        t, o = st[..., v0:v0 + 4], out[..., v0:v0 + 4]
        amax = np.max(np.abs(t), axis=(-2, -1))
        for n in range(2):
            for h in range(3):
                if amax[n, h] == 0:
                    continue
                scale = np.float32(amax[n, h]) / np.float32(448.0)
                # the tile's largest element maps to code 448 (or just under it), so it comes back
                # to within one rounding of amax, and nothing exceeds it by more than that
                assert np.max(np.abs(o[n, h])) <= amax[n, h] * (1 + 2 ** -20)
                # every element is an E4M3 value times the tile's scale (to float32 rounding)
                codes = (o[n, h] / scale).astype(np.float64).ravel()
                grid = Q.e4m3_values()
                near = grid[np.abs(codes[:, None] - grid[None, :]).argmin(axis=1)]
                np.testing.assert_allclose(codes, near, rtol=1e-6, atol=0)
    # a partial tile uses its own amax: scaling one column of the last tile changes only it
    st2 = st.copy()
    st2[..., 9] *= 100.0
    out2 = Q.state_fp8_qdq(st2, block_v=4)
    np.testing.assert_array_equal(out2[..., :8], out[..., :8])


def test_idempotent():
    rng = np.random.default_rng(2)
    st = rng.standard_normal((3, 16, 20)).astype(np.float32) * 3.0
    once = Q.state_fp8_qdq(st, block_v=8)
    np.testing.assert_array_equal(Q.state_fp8_qdq(once, block_v=8), once)
