"""Pass skipping on the device, bit-exact against the CPU oracle (needs a GPU).

Inputs whose digit is constant in some passes (the first, a middle one, the
last ones, all but one, all), inputs already in order, and near-sorted inputs
whose single out-of-order pair sits on each boundary the order check crosses:
inside a 16-byte vector, between the vectors of one warp, between warps,
between rounds of the vector loop, between the CTAs' chunks, in the scalar
tail, at the very end.  Both schedules and digit widths, every key type,
with and without values, in place and out of place, aligned and unaligned,
and a CUDA graph replayed over inputs that skip different passes.  The skip
record the sort leaves in temp is compared with its definition computed on
the CPU, so a check that silently stopped firing would fail here.
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


def expected_record(kt, keys, b, e):
    """(differing_bits, unordered) from their definitions, on the oracle's
    ordered keys."""
    o = oracle.ordered_keys(kt, keys).astype(np.uint64)
    diff = int(np.bitwise_or.reduce(o ^ o[0])) if len(o) else 0
    width = e - b
    mask = np.uint64((1 << width) - 1) if width < 64 else np.uint64(0xFFFFFFFFFFFFFFFF)
    d = (o >> np.uint64(b)) & mask
    unordered = int(bool(np.any(d[:-1] > d[1:])))
    return diff, unordered


def passes_run(kt, diff, unordered, b, e, rb):
    if not unordered:
        return 0
    return sum(1 for s in range(b, e, rb) if (diff >> s) & ((1 << min(rb, e - s)) - 1))


def check(kt, keys, vals, b, e, expect_runs=None, **kw):
    got_k, got_v, rec = gpu_sort(kt, keys, vals, b, e, want_record=True, **kw)
    ref_k, ref_v = oracle.sort(kt, keys, vals, b, e)
    assert np.array_equal(got_k, ref_k), f"keys differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"
    if vals is not None:
        assert np.array_equal(got_v, ref_v), f"values differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"
    want = expected_record(kt, keys, b, e)
    assert rec == want, f"skip record {rec} != {want}"
    if expect_runs is not None:
        rb = kw.get("radix_bits") or 8
        assert passes_run(kt, rec[0], rec[1], b, e, rb) == expect_runs


N = 300_001  # several tiles and CTAs, a ragged tail


def u32(seed, n=N):
    return synth.u32_uniform(n, seed)


# (name, key transform, passes that run at r = 8 over [0, 32))
CONSTANT_DIGITS = [
    ("low_half_only", lambda k: k & np.uint32(0xFFFF), 2),
    ("low_byte_constant", lambda k: (k & np.uint32(0xFFFFFF00)) | np.uint32(0x5A), 3),
    ("second_byte_constant", lambda k: (k & np.uint32(0xFFFF00FF)) | np.uint32(0x3C00), 3),
    ("third_byte_only", lambda k: k & np.uint32(0x00FF0000), 1),
    ("all_equal", lambda k: np.full_like(k, 0xDEADBEEF), 0),
]


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
@pytest.mark.parametrize("name,fn,runs", CONSTANT_DIGITS, ids=[c[0] for c in CONSTANT_DIGITS])
@pytest.mark.parametrize("with_vals", [False, True])
@pytest.mark.parametrize("in_place", [False, True])
def test_constant_digits(algo, name, fn, runs, with_vals, in_place):
    keys = fn(u32(11))
    vals = synth.iota_u32(N) if with_vals else None
    check("u32", keys, vals, 0, 32, expect_runs=runs, algo=algo, in_place=in_place)


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
def test_constant_digits_radix4_and_partial_range(algo):
    keys = u32(12) & np.uint32(0x0F0FF0F0)
    check("u32", keys, None, 0, 32, expect_runs=4, algo=algo, radix_bits=4)
    check("u32", keys, synth.iota_u32(N), 4, 28, algo=algo, radix_bits=4, in_place=True)
    check("u32", keys, None, 8, 20, algo=algo)


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
def test_other_key_types(algo):
    # i32 in [0, 2^16): the ordered keys share their top 16 bits.
    k = (u32(13) & np.uint32(0xFFFF))
    check("i32", k, synth.iota_u32(N), 0, 32, expect_runs=2, algo=algo)
    # f32 in [1, 2): sign and exponent shared.
    f = (np.uint32(0x3F800000) | (u32(14) & np.uint32(0x007FFFFF)))
    check("f32", f, None, 0, 32, expect_runs=3, algo=algo)
    # u64 below 2^32: the upper four passes are skipped.
    k64 = synth.u64_uniform(N, 15) & np.uint64(0xFFFFFFFF)
    check("u64", k64, synth.iota_u32(N), 0, 64, expect_runs=4, algo=algo)
    check("u64", k64, None, 0, 64, expect_runs=4, algo=algo, in_place=True)


def sorted_input(kt, n, seed):
    keys = synth.u64_uniform(n, seed) if kt == "u64" else u32(seed, n)
    if kt == "f32":
        keys = synth.f32_edge(n, seed)
    return oracle.sort(kt, keys, None, 0, rs.KEY_BITS[kt])[0]


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
@pytest.mark.parametrize("kt", ["u32", "i32", "f32", "u64"])
def test_already_sorted(algo, kt):
    keys = sorted_input(kt, N, 21)
    check(kt, keys, synth.iota_u32(N), 0, rs.KEY_BITS[kt], expect_runs=0, algo=algo)
    check(kt, keys, None, 0, rs.KEY_BITS[kt], expect_runs=0, algo=algo, in_place=True)
    check(kt, keys, None, 0, rs.KEY_BITS[kt], expect_runs=0, algo=algo, offset=1)
    # Ties only: all keys equal is sorted too.
    check(kt, np.full_like(keys, keys[N // 2]), None, 0, rs.KEY_BITS[kt], expect_runs=0, algo=algo)


def test_sorted_within_range_only():
    # Bits [8, 16) ascending, the rest random: in order for that range.
    k = u32(22)
    k = (k & np.uint32(0xFFFF00FF)) | (np.sort(k & np.uint32(0xFF00)))
    for algo in ("onesweep", "reduce_scan"):
        check("u32", k, synth.iota_u32(N), 8, 16, expect_runs=0, algo=algo)
        check("u32", k, None, 0, 32, algo=algo)


# Large enough that every CTA of the first read owns whole rounds of the
# vector loop (reduce-then-scan: 2 rounds of 2048 vectors per chunk; chained
# scan: 3 rounds over the grid), so both the shuffled and the loaded
# neighbour paths of the order check run.
N_BIG = (1 << 23) + 3
SWAPS = [1, 3, 127, 4095, 8191, 16383, 16384 * 37 - 1, 622_592 * 4 - 1, (1 << 23) - 1, N_BIG - 2]


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
def test_one_pair_out_of_order(algo):
    base = np.arange(N_BIG, dtype=np.uint32) * np.uint32(3)
    for i in SWAPS:
        keys = base.copy()
        keys[i], keys[i + 1] = keys[i + 1], keys[i]
        check("u32", keys, None, 0, 32, algo=algo)
    check("u32", base, None, 0, 32, expect_runs=0, algo=algo)
    # Unaligned: the whole first read takes the scalar path.
    keys = base.copy()
    keys[4095], keys[4096] = keys[4096], keys[4095]
    check("u32", keys, None, 0, 32, algo=algo, offset=1)


def test_graph_replays_follow_the_data():
    n = N
    kin = torch.empty(n, dtype=torch.int32, device="cuda:0")
    kout = torch.empty_like(kin)
    tb = rs.rs_temp_bytes("u32", False, n, 0, 32)
    temp = torch.empty(tb, dtype=torch.uint8, device="cuda:0")
    stream = torch.cuda.Stream()
    d = rs.make_desc("u32", kin, kout, None, None, n, 0, 32, temp, tb, stream)
    g = rs.Graph(d)
    try:
        for keys in (u32(31), sorted_input("u32", n, 32), u32(33) & np.uint32(0xFF00FF),
                     np.full(n, 7, np.uint32), u32(34)):
            kin.copy_(to_dev(keys, "cuda:0"))
            torch.cuda.synchronize()
            g.launch(stream)
            stream.synchronize()
            got = kout.cpu().numpy().view(np.uint32)
            assert np.array_equal(got, oracle.sort("u32", keys, None, 0, 32)[0])
            assert rs.rs_skip_record(temp, stream)[1:] == expected_record("u32", keys, 0, 32)
    finally:
        g.close()


# Large enough that every reduce-then-scan CTA walks several tiles (more
# tiles than CTAs), so the running passes take their buffers from the plan
# through several tile iterations: keys only (staged tiles) and with values,
# in place and out of place, ascending and descending.
N_MULTI = (1 << 22) + 5


@pytest.mark.parametrize("with_vals", [False, True])
@pytest.mark.parametrize("in_place", [False, True])
def test_skipped_passes_over_many_tiles(with_vals, in_place):
    keys = u32(41, N_MULTI) & np.uint32(0x00FF00FF)    # passes 1 and 3 skipped
    vals = synth.iota_u32(N_MULTI) if with_vals else None
    check("u32", keys, vals, 0, 32, expect_runs=2, algo="reduce_scan", in_place=in_place)
    got, gv, rec = gpu_sort("u32", keys, vals, 0, 32, algo="reduce_scan", in_place=in_place,
                            descending=True, want_record=True)
    ref_k, ref_v = oracle.sort("u32", keys, vals, 0, 32, descending=True)
    assert np.array_equal(got, ref_k)
    if with_vals:
        assert np.array_equal(gv, ref_v)
