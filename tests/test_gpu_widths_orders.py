"""16-bit keys, descending order and 64-bit payloads, bit-exact against the
CPU oracle (needs a GPU).

uint16, int16 and binary16 keys under every schedule and both digit widths,
with and without values, full and partial bit ranges, in place, unaligned
and through the typed entry points; descending order for every key type,
including the inputs that skip passes (already in ascending order: nothing
skipped; already in descending order: every pass skipped), whose skip record
is checked against its definition; uint64 payloads for 32-, 64- and 16-bit
keys (expected payloads gathered by the oracle's permutation); AUTO's
schedule for each key/value shape just above 2^22 keys.
"""
import numpy as np
import pytest

import lsd_radix_sort_key_gb300 as rs
import oracle
import synth
from gpu_util import gpu_sort, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    rs.build()
    rs.lib()


ALGOS = ["onesweep", "reduce_scan", "cluster"]


def gen_keys(kt, n, seed):
    if kt == "u64":
        return synth.u64_uniform(n, seed)
    if kt == "f32":
        return synth.f32_edge(n, seed)
    if kt == "f16":
        return synth.f16_edge(n, seed)
    if kt in ("u16", "i16"):
        return synth.u16_uniform(n, seed)
    return synth.u32_uniform(n, seed)


def check(kt, keys, vals, b, e, descending=False, **kw):
    got_k, got_v = gpu_sort(kt, keys, vals, b, e, descending=descending, **kw)
    ref_k, ref_v = oracle.sort(kt, keys, vals, b, e, descending=descending)
    assert np.array_equal(got_k, ref_k), f"keys differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"
    if vals is not None:
        assert np.array_equal(got_v, ref_v), f"values differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"


def sizes(algo, kt, with_vals):
    if algo == "cluster":
        cap = rs.rs_cluster_max_n(kt, with_vals)
        return [1, 31, 3841, cap // 2 + 1, cap]
    return [1, 31, 3841, 50_000, 300_001]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("kt", ["u16", "i16", "f16"])
@pytest.mark.parametrize("with_vals", [False, True])
@pytest.mark.parametrize("radix_bits", [8, 4])
def test_16bit_keys(algo, kt, with_vals, radix_bits):
    for i, n in enumerate(sizes(algo, kt, with_vals)):
        keys = gen_keys(kt, n, 900 + i)
        vals = synth.iota_u32(n) if with_vals else None
        check(kt, keys, vals, 0, 16, algo=algo, radix_bits=radix_bits)


@pytest.mark.parametrize("algo", ALGOS)
def test_16bit_ranges_in_place_unaligned(algo):
    n = sizes(algo, "u16", True)[-1]
    keys = synth.u16_uniform(n, 950)
    for b, e in [(0, 5), (3, 14), (8, 16), (4, 12)]:
        check("u16", keys, synth.iota_u32(n), b, e, algo=algo)
    check("f16", synth.f16_normal_specials(n, 951), synth.iota_u32(n), 0, 16, algo=algo, in_place=True)
    check("i16", keys, None, 0, 16, algo=algo, offset=1)
    check("u16", keys & np.uint16(0xFF), synth.iota_u32(n), 0, 16, algo=algo)     # high pass skipped


def test_16bit_typed_entry_points():
    n = 70_001
    keys = synth.f16_normal_specials(n, 960)
    kin = to_dev(keys, "cuda:0")
    kout = torch.empty_like(kin)
    vin = to_dev(synth.iota_u32(n), "cuda:0")
    vout = torch.empty_like(vin)
    tb = rs.rs_temp_bytes("f16", True, n, 0, 16)
    temp = torch.empty(tb, dtype=torch.uint8, device="cuda:0")
    assert rs.rs_sort_pairs_f16(kin, kout, vin, vout, n, 0, 16, temp, tb, None) == 0
    torch.cuda.synchronize()
    ref_k, ref_v = oracle.sort("f16", keys, synth.iota_u32(n), 0, 16)
    assert np.array_equal(kout.cpu().numpy().view(np.uint16), ref_k)
    assert np.array_equal(vout.cpu().numpy().view(np.uint32), ref_v)
    assert rs.rs_sort_keys_u16(kin, kout, n, 0, 16, temp, tb, None) == 0
    torch.cuda.synchronize()
    assert np.array_equal(kout.cpu().numpy().view(np.uint16), oracle.sort("u16", keys)[0])


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("kt", ["u32", "i32", "f32", "u64", "u16", "f16"])
@pytest.mark.parametrize("with_vals", [False, True])
def test_descending(algo, kt, with_vals):
    for i, n in enumerate(sizes(algo, kt, with_vals)):
        keys = gen_keys(kt, n, 1000 + i)
        vals = synth.iota_u32(n) if with_vals else None
        check(kt, keys, vals, 0, rs.KEY_BITS[kt], descending=True, algo=algo)


@pytest.mark.parametrize("algo", ALGOS)
def test_descending_partial_ranges_ties_and_skips(algo):
    n = sizes(algo, "u32", True)[-1]
    keys = synth.u32_uniform(n, 1100)
    vals = synth.iota_u32(n)
    check("u32", keys, vals, 5, 27, descending=True, algo=algo, radix_bits=4)
    check("u32", synth.u32_bits(n, 1101, 3), vals, 0, 32, descending=True, algo=algo)     # ties
    check("u32", keys, vals, 0, 32, descending=True, algo=algo, in_place=True)
    up = oracle.sort("u32", keys, None, 0, 32)[0]
    down = oracle.sort("u32", keys, None, 0, 32, descending=True)[0]
    for inp, unordered in ((up, 1), (down, 0)):
        got, _, rec = gpu_sort("u32", inp, None, 0, 32, algo=algo, descending=True, want_record=True)
        assert np.array_equal(got, down)
        assert rec[1] == unordered


def check64(kt, keys, b, e, descending=False, **kw):
    """64-bit payloads: the oracle gives the permutation (values = index) and
    the expected payloads are the random 64-bit values gathered by it."""
    n = len(keys)
    vals64 = synth.u64_uniform(n, 4242 + n)
    got_k, got_v = gpu_sort(kt, keys, vals64, b, e, descending=descending, **kw)
    ref_k, perm = oracle.sort(kt, keys, synth.iota_u32(n), b, e, descending=descending)
    assert np.array_equal(got_k, ref_k), f"keys differ ({kt}, n={n}, {kw})"
    assert got_v.dtype == np.uint64 and np.array_equal(got_v, vals64[perm]), f"values differ ({kt}, n={n}, {kw})"


def sizes64(algo, kt):
    if algo == "cluster":
        cap = rs.rs_cluster_max_n(kt, 8)
        return [1, 31, cap // 3, cap]
    return [1, 3841, 300_001]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("kt", ["u32", "f32", "u64", "u16"])
def test_64bit_values(algo, kt):
    for i, n in enumerate(sizes64(algo, kt)):
        check64(kt, gen_keys(kt, n, 1200 + i), 0, rs.KEY_BITS[kt], algo=algo)
    n = sizes64(algo, kt)[-1]
    keys = gen_keys(kt, n, 1210)
    check64(kt, keys, 0, rs.KEY_BITS[kt], algo=algo, radix_bits=4)
    check64(kt, keys, 0, rs.KEY_BITS[kt], algo=algo, descending=True)
    check64(kt, keys, 0, rs.KEY_BITS[kt], algo=algo, in_place=True)
    if kt in ("u32", "u64", "u16"):
        check64(kt, keys, 3, rs.KEY_BITS[kt] - 2, algo=algo)


def test_64bit_values_unaligned_keys_and_sort_wrapper():
    n = 100_003
    keys = synth.u32_uniform(n, 1220)
    check64("u32", keys, 0, 32, offset=1)   # keys 4-byte aligned only; values still 8-byte aligned
    kin = to_dev(keys, "cuda:0")
    vin = to_dev(synth.u64_uniform(n, 1221), "cuda:0")
    ko, vo = rs.sort(kin, vin, key_type="u32", descending=True)
    torch.cuda.synchronize()
    ref_k, perm = oracle.sort("u32", keys, synth.iota_u32(n), 0, 32, descending=True)
    assert np.array_equal(ko.cpu().numpy().view(np.uint32), ref_k)
    assert np.array_equal(vo.cpu().numpy().view(np.uint64), synth.u64_uniform(n, 1221)[perm])


# AUTO picks the schedule by size and shape: 64-bit keys alone and 32-bit
# keys with values take the chained scan up to 2^23 keys, 64-bit keys with
# 64-bit values take it at every size it supports.  Each case sorts through
# AUTO just above 2^22 keys (a ragged last tile) and checks the schedule by
# its kernel count as well as the result.
@pytest.mark.parametrize("kt,vb,chained", [("u64", 0, True), ("u32", 4, True), ("u32", 8, True),
                                           ("u64", 8, True), ("u64", 4, False), ("u32", 0, False)])
def test_auto_schedule_by_shape(kt, vb, chained):
    n = (1 << 22) + 5
    keys = gen_keys(kt, n, 1300 + vb)
    bits = rs.KEY_BITS[kt]
    passes = bits // 8
    vin, vout = ((0x3 << 40), (0x4 << 40)) if vb else (None, None)  # addresses for the count query only
    d = rs.make_desc(kt, None, None, vin, vout, n, 0, bits, None, 0, 0, "auto", 0, value_bytes=vb)
    assert rs.rs_sort_kernel_count(d) == (1 + passes if chained else 3 * passes)
    if vb == 8:
        check64(kt, keys, 0, bits)
    else:
        check(kt, keys, synth.iota_u32(n) if vb else None, 0, bits)
