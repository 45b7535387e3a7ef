"""Seeded mixed cases, bit-exact against the CPU oracle (needs a GPU).

Each case draws, from one fixed seed, a key type, a payload (none, 32-bit
index, 64-bit random), a ragged size, a digit range, an order, a schedule,
a digit width, in place or not, a pointer offset and a key distribution
(uniform, few distinct values, AND-of-4 skew, one repeated key), so that
combinations no hand-written test names still meet the oracle.  Expected
32-bit payloads are the oracle's own; 64-bit payloads are gathered by the
oracle's permutation.
"""
import numpy as np
import pytest

import lsd_radix_sort_key_gb300 as rs
import oracle
import synth
from gpu_util import NP_KEY, gpu_sort

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    rs.build()
    rs.lib()


KEY_TYPES = ["u32", "i32", "f32", "u64", "u16", "i16", "f16"]
DISTS = ["uniform", "few", "and4", "constant"]


def draw_keys(kt, n, dist, seed):
    bits = rs.KEY_BITS[kt]
    if bits == 64:
        raw = synth.u64_uniform(n, seed)
        if dist == "few":
            raw = raw & np.uint64(0x7)
        elif dist == "and4":
            raw = raw & synth.u64_uniform(n, seed + 1) & synth.u64_uniform(n, seed + 2) \
                & synth.u64_uniform(n, seed + 3)
        elif dist == "constant":
            raw = np.full(n, np.uint64(0x8000000000000001))
        return raw.astype(np.uint64)
    raw = synth.u32_uniform(n, seed)
    if dist == "few":
        raw = synth.u32_bits(n, seed, 3)
    elif dist == "and4":
        raw = synth.u32_and4(n, seed)
    elif dist == "constant":
        raw = np.full(n, np.uint32(0x80000001))
    if bits == 16:
        return (raw >> np.uint32(16)).astype(np.uint16) if dist != "few" else raw.astype(np.uint16)
    return raw.astype(np.uint32)


def draw_case(k):
    rng = np.random.default_rng(0x5EED0400 + k)
    kt = KEY_TYPES[rng.integers(len(KEY_TYPES))]
    vb = int(rng.choice([0, 4, 8]))
    n = int(rng.choice([1, 2, 33, 4097, 30_001, 65_536, 131_077, 262_147, 500_009]))
    bits = rs.KEY_BITS[kt]
    if rng.random() < 0.5:
        b, e = 0, bits
    else:
        b = int(rng.integers(0, bits))
        e = int(rng.integers(b, bits + 1))
    algo = str(rng.choice(["auto", "onesweep", "reduce_scan", "cluster"]))
    if algo == "cluster" and n > rs.rs_cluster_max_n(kt, vb if vb else False):
        algo = "auto"
    radix_bits = int(rng.choice([0, 8, 4]))
    descending = bool(rng.random() < 0.4)
    in_place = bool(rng.random() < 0.3)
    offset = int(rng.choice([0, 0, 1, 3]))
    dist = DISTS[rng.integers(len(DISTS))]
    return dict(kt=kt, vb=vb, n=n, b=b, e=e, algo=algo, radix_bits=radix_bits,
                descending=descending, in_place=in_place, offset=offset, dist=dist, seed=0x600 + 7 * k)


@pytest.mark.parametrize("k", range(48))
def test_mixed_case(k):
    c = draw_case(k)
    n, kt = c["n"], c["kt"]
    keys = draw_keys(kt, n, c["dist"], c["seed"])
    assert keys.dtype == NP_KEY[kt]
    idx = synth.iota_u32(n)
    if c["vb"] == 8:
        vals = synth.u64_uniform(n, c["seed"] + 11)
    elif c["vb"] == 4:
        vals = idx
    else:
        vals = None
    got_k, got_v = gpu_sort(kt, keys, vals, c["b"], c["e"], algo=c["algo"], radix_bits=c["radix_bits"],
                            offset=c["offset"], in_place=c["in_place"], descending=c["descending"])
    ref_k, perm = oracle.sort(kt, keys, idx, c["b"], c["e"], radix_bits=c["radix_bits"] or 8,
                              descending=c["descending"])
    assert np.array_equal(got_k, ref_k), f"keys differ: {c}"
    if c["vb"] == 8:
        assert np.array_equal(got_v, vals[perm]), f"64-bit values differ: {c}"
    elif c["vb"] == 4:
        assert np.array_equal(got_v, perm), f"values differ: {c}"
