"""Seeded input generators: determinism and the shape of each workload (no GPU)."""
import numpy as np

import synth

MASK = (1 << 64) - 1


def splitmix64_ref(seed, n):
    """SplitMix64 (Steele, Lea & Flood 2014) written out in Python integers."""
    out, s = [], seed
    for _ in range(n):
        s = (s + 0x9E3779B97F4A7C15) & MASK
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_vector():
    # first outputs for seed 1234567 as given with the generator's reference code
    assert synth.splitmix64(5, 1234567).tolist() == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]
    assert synth.splitmix64(100, 0x5EED0004).tolist() == splitmix64_ref(0x5EED0004, 100)


def test_deterministic_and_prefix_stable():
    a = synth.u32_uniform(10000, 42)
    b = synth.u32_uniform(20000, 42)
    assert np.array_equal(a, b[:10000])
    assert not np.array_equal(a, synth.u32_uniform(10000, 43))


def test_and4_bit_density():
    k = synth.u32_and4(1 << 16, 7)
    bits = np.unpackbits(k.view(np.uint8)).mean()
    assert abs(bits - 1 / 16) < 0.005


def test_morton_codes_are_30_bit_and_decode():
    k = synth.u32_morton30(4096, 0x1_5EED0004)
    assert int(k.max()) < (1 << 30)
    # x occupies bits 3b+2: de-interleave and check the coordinate range is used
    x = np.zeros_like(k)
    for b in range(10):
        x |= ((k >> (3 * b + 2)) & 1) << b
    assert x.max() > 1000 and x.min() < 24


def test_f32_specials_injected():
    n = 1 << 16
    k = synth.f32_normal_specials(n, 0x5EED0002)
    m = int(0.001 * n)
    assert int(np.sum(k == 0x80000000)) >= m
    assert int(np.sum(k == 0x00000000)) >= m
    assert int(np.sum(k == 0x7F800000)) == m
    assert int(np.sum(k == 0xFF800000)) == m
    assert int(np.sum(k == 0x7FC00000)) == m
    f = k.view(np.float32)
    finite = f[np.isfinite(f)]
    assert abs(float(finite.std()) - 1.0) < 0.05 and abs(float(finite.mean())) < 0.05


def test_workload_table():
    w = synth.WORKLOADS
    assert w["u32_uniform_2p28"].n == 1 << 28 and not w["u32_uniform_2p28"].with_values
    assert w["morton30_index_2p28"].end_bit == 30 and w["morton30_index_2p28"].with_values
    assert w["u64_uniform_index_2p28"].key_type == "u64"
    small = w["i32_uniform_index_2p26"].keys(n=1000)
    assert small.dtype == np.uint32 and small.size == 1000
    assert synth.sweep_workload(20).n == 1 << 20


def test_16bit_generators_are_seeded_and_prefix_stable():
    for gen in (synth.u16_uniform, synth.f16_edge, synth.f16_normal_specials):
        a = gen(1000, 5)
        assert a.dtype == np.uint16 and a.size == 1000
        assert np.array_equal(a, gen(1000, 5))
        assert not np.array_equal(a, gen(1000, 6))
    # the half-precision normals keep the float32 generator's injected specials
    f = synth.f16_normal_specials(100_000, 9)
    exp = (f >> 10) & 0x1F
    assert np.any(f == 0x8000) and np.any(f == 0) and np.any(f == 0x7C00) and np.any(f == 0xFC00)
    assert np.any((exp == 0x1F) & ((f & 0x3FF) != 0))
