"""The one-kernel cluster schedule, bit-exact against the CPU oracle (needs a GPU).

Every key type, with and without values, both digit widths, at sizes from
one key to the schedule's capacity (one CTA, a partial last CTA, exactly
full CTAs, 8 CTAs and one more, all sixteen), partial bit ranges, in place, unaligned pointers,
tie-heavy keys, and the inputs that skip passes (sorted, constant digits),
whose skip record is checked against its definition.
"""
import numpy as np
import pytest

import lsd_radix_sort_key_gb300 as rs
import oracle
import synth
from gpu_util import gpu_sort

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    rs.build()
    rs.lib()


def gen_keys(kt, n, seed):
    if kt == "u64":
        return synth.u64_uniform(n, seed)
    if kt == "f32":
        return synth.f32_edge(n, seed)
    return synth.u32_uniform(n, seed)


def check(kt, keys, vals, b, e, **kw):
    got_k, got_v = gpu_sort(kt, keys, vals, b, e, algo="cluster", **kw)
    ref_k, ref_v = oracle.sort(kt, keys, vals, b, e)
    assert np.array_equal(got_k, ref_k), f"keys differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"
    if vals is not None:
        assert np.array_equal(got_v, ref_v), f"values differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"


def sizes(kt, with_vals):
    cap = rs.rs_cluster_max_n(kt, with_vals)
    tile = cap // 16  # one CTA's share
    return [1, 2, 31, 1000, tile - 1, tile, tile + 1, 3 * tile + 17, 8 * tile, 8 * tile + 1, cap - 1, cap]


@pytest.mark.parametrize("radix_bits", [8, 4])
@pytest.mark.parametrize("kt", ["u32", "i32", "f32", "u64"])
@pytest.mark.parametrize("with_vals", [False, True])
def test_full_range(radix_bits, kt, with_vals):
    for i, n in enumerate(sizes(kt, with_vals)):
        keys = gen_keys(kt, n, 500 + i)
        vals = synth.iota_u32(n) if with_vals else None
        check(kt, keys, vals, 0, rs.KEY_BITS[kt], radix_bits=radix_bits)


@pytest.mark.parametrize("kt", ["u32", "i32", "f32", "u64"])
def test_partial_ranges_in_place_unaligned(kt):
    n = rs.rs_cluster_max_n(kt, True) - 5
    keys = gen_keys(kt, n, 77)
    bits = rs.KEY_BITS[kt]
    for b, e in [(0, 7), (3, 19), (bits - 9, bits), (5, 5 + 8 * 3)]:
        check(kt, keys, synth.iota_u32(n), b, e)
    check(kt, keys, synth.iota_u32(n), 0, bits, in_place=True)
    check(kt, keys, None, 0, bits - 8, in_place=True)  # an odd pass count for 32-bit keys
    check(kt, keys, synth.iota_u32(n), 0, bits, offset=1)


def test_ties_low_entropy_and_skipped_passes():
    cap = rs.rs_cluster_max_n("u32", True)
    keys = synth.u32_and4(cap, 78)
    check("u32", keys, synth.iota_u32(cap), 0, 32)
    check("u32", keys & np.uint32(0x3), synth.iota_u32(cap), 0, 32)        # 3 of 4 passes skipped
    check("u32", np.full(cap, 9, np.uint32), synth.iota_u32(cap), 0, 32)   # no pass runs
    srt = oracle.sort("u32", synth.u32_uniform(cap, 79), None, 0, 32)[0]
    got, _, rec = gpu_sort("u32", srt, None, 0, 32, algo="cluster", want_record=True)
    assert np.array_equal(got, srt) and rec[1] == 0
    srt[100], srt[101] = srt[101], srt[100]
    check("u32", srt, None, 0, 32)
    k = synth.u32_uniform(cap, 80) & np.uint32(0xFF00FF)
    got, _, rec = gpu_sort("u32", k, None, 0, 32, algo="cluster", want_record=True)
    assert np.array_equal(got, oracle.sort("u32", k, None, 0, 32)[0])
    o = k.astype(np.uint64)
    assert rec == (int(np.bitwise_or.reduce(o ^ o[0])), 1)


def test_auto_takes_the_cluster_below_its_capacity():
    for kt, v in [("u32", False), ("u32", True), ("u64", False), ("u64", True)]:
        cap = rs.rs_cluster_max_n(kt, v)
        vin = 3 << 40 if v else None
        vout = 4 << 40 if v else None
        one = rs.make_desc(kt, None, None, vin, vout, cap, 0, rs.KEY_BITS[kt], None, 0, 0, "auto")
        assert rs.rs_sort_kernel_count(one) == 1
        more = rs.make_desc(kt, None, None, vin, vout, cap + 1, 0, rs.KEY_BITS[kt], None, 0, 0, "auto")
        assert rs.rs_sort_kernel_count(more) > 1
