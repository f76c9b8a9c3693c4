"""The seeded input generator against its own published definition (CPU only)."""
import math

import numpy as np
import pytest

import synth

M64 = (1 << 64) - 1


def _mix(z):
    z ^= z >> 30; z = (z * 0xBF58476D1CE4E5B9) & M64
    z ^= z >> 27; z = (z * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_stream_words_follow_splitmix64():
    seed, tid = 1234, 5
    key = _mix(seed ^ _mix((tid + 0x632BE59BD9B4E019) & M64))
    want = [_mix((key + (i + 1) * 0x9E3779B97F4A7C15) & M64) for i in range(64)]
    assert synth.raw_bits(seed, tid, 64).tolist() == want
    # counter based: any slice equals the same slice of the whole stream
    assert synth.raw_bits(seed, tid, 10, offset=50).tolist() == want[50:60]


def test_box_muller_values_and_moments():
    seed, tid = 99, 3
    bits = synth.raw_bits(seed, tid, 8)
    u = ((bits >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53
    z = synth.normal_f64(seed, tid, 1.0, (8,))
    for j in range(4):
        r = math.sqrt(-2.0 * math.log(u[2 * j]))
        assert math.isclose(z[2 * j], r * math.cos(2 * math.pi * u[2 * j + 1]), rel_tol=1e-14, abs_tol=1e-15)
        assert math.isclose(z[2 * j + 1], r * math.sin(2 * math.pi * u[2 * j + 1]), rel_tol=1e-14, abs_tol=1e-15)
    big = synth.normal_f64(seed, tid, 1.0, (400000,))
    assert abs(big.mean()) < 0.01 and abs(big.std() - 1.0) < 0.01


def test_bf16_and_int8_rounding_of_draws():
    import torch
    z = synth.normal_f64(7, 1, 0.02, (50000,))
    b = synth.normal_bf16(7, 1, 0.02, (50000,))
    got = synth.bf16_bits_to_f32(b).astype(np.float64)
    # nearest bf16 value: no bf16 neighbour is closer (ties are measure-zero here)
    up = synth.bf16_bits_to_f32((b.astype(np.int32) + 1).astype(np.uint16)).astype(np.float64)
    dn = synth.bf16_bits_to_f32((b.astype(np.int32) - 1).astype(np.uint16)).astype(np.float64)
    err = np.abs(got - z)
    assert np.all(err <= np.abs(up - z)) and np.all(err <= np.abs(dn - z))
    # agrees with torch wherever the float32 rounding cannot matter
    ref = torch.from_numpy(z.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.mean(ref == got) > 0.999
    q = synth.int8_codes(7, 2, 40.0, (50000,))
    zq = synth.normal_f64(7, 2, 40.0, (50000,))
    assert np.array_equal(q.astype(np.float64), np.clip(np.rint(zq), -127, 127))
    s = synth.uniform_f32(7, 3, 0.5e-3, 1e-3, (10000,))
    assert s.min() >= 0.5e-3 and s.max() <= 1e-3


def test_workload_shapes():
    w = synth.WORKLOADS
    assert (w["mixtral_prefill"].T, w["mixtral_prefill"].d, w["mixtral_prefill"].f) == (4096, 4096, 14336)
    assert (w["skewed"].E, w["skewed"].k, w["skewed"].bias) == (128, 4, True)
    assert (w["int8"].wdtype, w["int8"].k, w["int8"].E) == ("int8", 6, 64)
    b = synth.skew_bias(128)
    assert b[0] == 0.0 and math.isclose(b[127], 2 * math.log(1 / 128), rel_tol=1e-7)
    L = synth.make_layer(w["tiny"])
    assert L.x.shape == (64, 256) and L.wg.shape == (8, 512, 256) and L.wd.shape == (8, 256, 512)


def test_int4_weights_ranges_and_packing():
    """int4 layers: codes 0..15 packed two to a byte (element 2m low nibble), zero
    points 6..9, q - z within +-6, scales in [0.006, 0.010)."""
    shape = synth.custom_shape("i4", T=4, d=64, f=32, E=3, k=2, wdtype="int4", seed=5)
    L = synth.make_layer(shape)
    assert L.wg.shape == (3, 32, 32) and L.wd.shape == (3, 64, 16) and L.wg.dtype == np.uint8
    for w, z in ((L.wg, L.zg), (L.wu, L.zu), (L.wd, L.zd)):
        q = synth.unpack_int4(w).astype(int)
        assert q.min() >= 0 and q.max() <= 15
        assert z.min() >= 6 and z.max() <= 9
        c = q - z.astype(int)[..., None]
        assert np.abs(c).max() <= 6 and 2.0 < c.std() < 3.0
        assert np.array_equal(synth.pack_int4(q), w)
    for s in (L.sg, L.su, L.sd):
        assert s.dtype == np.float32 and s.min() >= 0.006 and s.max() < 0.010


def test_fp8_weights_are_rounded_e4m3_codes():
    """fp8 layers: e4m3 bytes (never the NaN codes) of 32 N(0,1) rounded to nearest with
    ties to the even code, the same as PyTorch's float8_e4m3fn conversion of the draws;
    scales in [0.5e-3, 1e-3)."""
    torch = pytest.importorskip("torch")
    shape = synth.custom_shape("f8", T=4, d=64, f=32, E=3, k=2, wdtype="fp8", seed=5)
    L = synth.make_layer(shape)
    assert L.wg.shape == (3, 32, 64) and L.wd.shape == (3, 64, 32) and L.wg.dtype == np.uint8
    for w in (L.wg, L.wu, L.wd):
        assert not np.any((w & 0x7F) == 0x7F)
    draws = synth.normal_f64(shape.seed, synth.TID_WG, synth.FP8_SCALE, (3, 32, 64))
    ref = torch.from_numpy(draws).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref, L.wg)
    # a tie between two e4m3 values goes to the even code: 1 + 1/16 lies between
    # 0x38 (1.0) and 0x39 (1.125), 1 + 3/16 between 0x39 and 0x3A, 2^-10 between
    # 0x00 and 0x01 (2^-9); past 448 saturates
    g = synth._e4m3_grid()
    assert g[0x38] == 1.0 and g[0x39] == 1.125 and g[0x7E] == 448.0
    got = synth.encode_e4m3([1 + 1 / 16, 1 + 3 / 16, -(1 + 1 / 16), 2.0 ** -10, 500.0, -1.0])
    assert got.tolist() == [0x38, 0x3A, 0xB8, 0x00, 0x7E, 0xB8]
    for s in (L.sg, L.su, L.sd):
        assert s.dtype == np.float32 and s.min() >= 0.5e-3 and s.max() < 1e-3
