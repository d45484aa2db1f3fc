"""The seeded input generator: C stream == numpy restatement, recipe properties."""
import numpy as np

import ring_inputs as ri


def test_c_stream_matches_numpy_restatement():
    for seed, first, count, mult in ((1, 0, 5000, 1.0), (628, 123457, 4099, 2.0), (3, 2**33 + 1, 777, 8.0)):
        a = ri.normal_bf16(seed, first, count, mult)
        b = ri.normal_bf16_numpy(seed, first, count, mult)
        assert np.array_equal(a, b)


def test_splitmix64_known_values():
    # SplitMix64 seeded with 0: the first outputs of the published reference generator
    assert ri.splitmix64(0, 0) == 0xE220A8397B1DCDAF
    assert ri.splitmix64(0, 1) == 0x6E789E6AA1B965F4
    assert ri.splitmix64(0, 2) == 0x06C45D188009454F


def test_normal_moments_and_rounding():
    x = ri.bf16_bits_to_f64(ri.normal_bf16(42, 0, 1 << 20))
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    # values are bf16: the low 16 bits of the fp32 pattern are zero by construction
    b = ri.normal_bf16(42, 0, 1000)
    assert np.array_equal(ri.f32_to_bf16_bits(ri.bf16_bits_to_f32(b)), b)


def test_multiplier_is_exact_power_of_two():
    a = ri.bf16_bits_to_f64(ri.normal_bf16(9, 10, 4096, 1.0))
    b = ri.bf16_bits_to_f64(ri.normal_bf16(9, 10, 4096, 2.0))
    assert np.array_equal(a * 2.0, b)


def test_stream_order_q_then_k_then_v():
    w = ri.WORKLOADS["small"]
    q, k, v = ri.generate(w)
    flat = ri.normal_bf16(w.seed, 0, w.n_q + 2 * w.n_kv)
    assert np.array_equal(q.reshape(-1), flat[: w.n_q])
    assert np.array_equal(k.reshape(-1), flat[w.n_q: w.n_q + w.n_kv])
    assert np.array_equal(v.reshape(-1), flat[w.n_q + w.n_kv:])


def test_outlier_rows_scaled_by_eight():
    w = ri.WORKLOADS["long_s128k_c"].with_(S=4096, P=4, Hq=2, Hkv=2)
    q, k, v = ri.generate(w)
    mask = ri.outlier_rows(w)
    assert 0.005 < mask.mean() < 0.015
    plain = ri.normal_bf16(w.seed, w.n_q, w.n_kv).reshape(k.shape)
    kf, pf = ri.bf16_bits_to_f64(k), ri.bf16_bits_to_f64(plain)
    assert np.array_equal(kf[mask], pf[mask] * 8.0)
    assert np.array_equal(kf[~mask], pf[~mask])


def test_generate_into_buffers_matches_arrays():
    w = ri.WORKLOADS["small"].with_(Hq=4, Hkv=2)
    q, k, v = ri.generate(w)
    bufs = [np.empty(n, dtype=np.uint16) for n in (w.n_q, w.n_kv, w.n_kv)]
    ri.generate(w, *(b.ctypes.data for b in bufs))
    assert np.array_equal(bufs[0], q.reshape(-1))
    assert np.array_equal(bufs[1], k.reshape(-1))
    assert np.array_equal(bufs[2], v.reshape(-1))


def test_row_sample_contents():
    w = ri.WORKLOADS["h32_s32k_c"]
    rows = ri.sample_rows(w)
    assert len(rows) >= 4096 and np.all(np.diff(rows) > 0)
    s = set(rows.tolist())
    for bh in range(w.B * w.Hq):
        for i in (0, 1, 127, 128, w.S - 1, w.L, w.L - 1, 3 * w.L, 5 * w.L - 1):
            assert bh * w.S + i in s


def test_workload_flops_and_bytes():
    w = ri.WORKLOADS["h32_s32k_nc"]
    assert w.flops() == 4 * 128 * 32768**2 * 32
    assert w.staging_bytes() == 240 * 32 * (1 << 20)
    assert ri.WORKLOADS["h32_s32k_c"].staging_bytes() == 120 * 32 * (1 << 20)
