"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each ``pin_*`` function checks the oracle (or a planted-mistake copy of it,
passed as ``lib``) against something other than itself:

* the base-10 worked example printed pass by pass in "Radix sort paralelo
  sobre el scan", section "La idea y el requisito de estabilidad";
* the one-bit split of "Radix sort を実装 & 測定してみた", section
  "アルゴリズムの詳細", against a plain stable partition;
* the global-position formula P_d[n] + m of "高性能计算：GPU上的基数排序",
  section "GPU上的基数排序", on a hand-built case with the page's numbers, and
  the digit-major block-count scan of "Radix sort paralelo sobre el scan",
  section "Las tres fases de una pasada", on random cases;
* the Blelloch up-sweep / down-sweep of "高性能计算：GPU上的基数排序", section
  "GPU上的扫描", against the oracle's exclusive scan;
* the ordering invariants of the float32 map ("Radix sort を実装 & 測定してみた",
  section "符号付型、浮動小数点型に対する radix sort": negatives before
  positives, NaN/Inf last) and of the int32 map ("Radix sort paralelo sobre el
  scan", section "Claves con signo y en coma flotante"), checked against IEEE
  and two's-complement order with Python's own comparisons;
* brute force: Python's stable ``sorted`` on tiny and small inputs, exhaustive
  over 3-value alphabets;
* 16-bit keys (uint16, int16 and IEEE binary16, sorted "by the same
  procedure" as "Radix sort を実装 & 測定してみた" says of other widths): the
  maps' ordering invariants against Python's half-precision unpacking and
  two's-complement values, and brute force;
* descending order against Python's stable ``sorted(..., reverse=True)``,
  which keeps ties in input order.

``test_planted_mistakes_are_caught`` compiles copies of oracle.c with one
plausible mistake each and checks that some pin fails for every copy.
"""
import itertools
import os
import struct
import subprocess

import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden

# ------------------------------------------------------------ independent orders


def f32_order_key(bits: int):
    """Total order the float32 sort must produce, from IEEE semantics alone.

    Finite values by numeric value, -0.0 just before +0.0, and every NaN and
    both infinities tied after everything else.
    """
    if (bits >> 23) & 0xFF == 0xFF:
        return (2, 0.0, 0)
    v = struct.unpack("<f", struct.pack("<I", bits))[0]
    if v == 0.0:
        return (1, 0.0, -1 if bits & 0x80000000 else 0)
    return (1, v, 0)


def f16_order_key(bits: int):
    """The same total order for IEEE binary16 (Python unpacks half precision)."""
    if (bits >> 10) & 0x1F == 0x1F:
        return (2, 0.0, 0)
    v = struct.unpack("<e", struct.pack("<H", bits))[0]
    if v == 0.0:
        return (1, 0.0, -1 if bits & 0x8000 else 0)
    return (1, v, 0)


def i32_value(bits: int) -> int:
    return bits - (1 << 32) if bits & 0x80000000 else bits


def i16_value(bits: int) -> int:
    return bits - (1 << 16) if bits & 0x8000 else bits


def brute_force_perm(key_type, keys, begin_bit, end_bit, descending=False):
    """Stable order of indices by the definition of the sort (Python's sort is
    stable, also with reverse=True)."""
    n = len(keys)
    full = begin_bit == 0 and end_bit == oracle.KEY_BITS[key_type]
    by = {"f32": f32_order_key, "f16": f16_order_key, "i32": i32_value, "i16": i16_value}
    if key_type in by and full:
        f = by[key_type]
        return sorted(range(n), key=lambda i: f(int(keys[i])), reverse=descending)
    if key_type in ("u32", "u64", "u16"):
        mask = (1 << (end_bit - begin_bit)) - 1
        return sorted(range(n), key=lambda i: (int(keys[i]) >> begin_bit) & mask, reverse=descending)
    raise ValueError("no independent order for a partial bit range of a signed/float key")


BOUNDARY_F32 = [
    0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007FFFFF, 0x807FFFFF, 0x00800000,
    0x80800000, 0x3F800000, 0xBF800000, 0x3F800001, 0xBF800001, 0x7F7FFFFF, 0xFF7FFFFF,
    0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7FFFFFFF,
    0xFFFFFFFF, 0x7FA00000, 0x40490FDB, 0xC0490FDB,
]
BOUNDARY_I32 = [0x80000000, 0x80000001, 0xFFFFFFFE, 0xFFFFFFFF, 0, 1, 2, 0x7FFFFFFE, 0x7FFFFFFF,
                0x00010000, 0xFFFF0000, 0x40000000, 0xC0000000]

# ------------------------------------------------------------------------ pins


def pin_decimal_example(lib=None):
    rows = dict(read_golden("decimal_lsd_example.txt"))
    keys = [int(t) for t in rows["input"]]
    trace = oracle.decimal_lsd_trace(keys, 3, lib=lib)
    for p, label in enumerate(["units", "tens", "hundreds"]):
        assert trace[p].tolist() == [int(t) for t in rows[label]], label


def pin_one_bit_split(lib=None):
    rng = np.random.default_rng(11)
    for trial in range(6):
        n = [1, 2, 7, 64, 257, 1000][trial]
        keys = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
        vals = np.arange(n, dtype=np.uint32)
        for bit in (0, 5, 31):
            zeros = [i for i in range(n) if not (int(keys[i]) >> bit) & 1]
            ones = [i for i in range(n) if (int(keys[i]) >> bit) & 1]
            want = zeros + ones
            k1, v1 = oracle.one_bit_split_sort("u32", keys, vals, bit, bit + 1, lib=lib)
            assert v1.tolist() == want
            assert k1.tolist() == [int(keys[i]) for i in want]
            k2, v2 = oracle.sort("u32", keys, vals, bit, bit + 1, radix_bits=1, lib=lib)
            assert v2.tolist() == want


def pin_global_position(lib=None):
    rows = dict(read_golden("global_position_example.txt"))
    digits = np.array([int(t) for t in rows["digits"]], dtype=np.uint32)
    bs = int(rows["block_size"][0])
    e = int(rows["element_index"][0])
    d = int(digits[e])
    blk = e // bs
    m = int(np.sum(digits[blk * bs:e] == d))                       # local prefix
    nb = len(digits) // bs
    counts = np.array([[np.sum(digits[b * bs:(b + 1) * bs] == dd) for b in range(nb)]
                       for dd in range(4)])                        # counts[digit][block]
    P = oracle.exclusive_scan(counts.reshape(-1), lib=lib).reshape(4, nb)  # digit-major
    assert d == int(rows["page_digit"][0])
    assert blk + 1 == int(rows["page_block"][0])
    assert m == int(rows["page_local_prefix"][0])
    assert int(P[d, blk]) == int(rows["page_block_prefix"][0])
    assert int(P[d, blk]) + m == int(rows["page_position"][0])
    _, perm = oracle.sort("u32", digits, np.arange(len(digits), dtype=np.uint32), 0, 2, lib=lib)
    assert int(np.nonzero(perm == e)[0][0]) == int(rows["page_position"][0])


def pin_digit_major_scan(lib=None):
    rng = np.random.default_rng(5)
    for r, nb, bs in [(2, 7, 33), (4, 13, 256), (8, 5, 1000)]:
        bins = 1 << r
        n = nb * bs - 17
        digits = rng.integers(0, bins, size=n).astype(np.uint32)
        counts = np.zeros((bins, nb), dtype=np.uint64)
        for b in range(nb):
            counts[:, b] = np.bincount(digits[b * bs:(b + 1) * bs], minlength=bins)
        base = oracle.exclusive_scan(counts.reshape(-1), lib=lib).reshape(bins, nb)
        pos = np.empty(n, dtype=np.int64)
        seen = {}
        for i in range(n):
            b, d = i // bs, int(digits[i])
            m = seen.get((b, d), 0)
            seen[(b, d)] = m + 1
            pos[i] = int(base[d, b]) + m
        _, perm = oracle.sort("u32", digits, np.arange(n, dtype=np.uint32), 0, r, radix_bits=r,
                              lib=lib)
        inv = np.empty(n, dtype=np.int64)
        inv[perm.astype(np.int64)] = np.arange(n)
        assert np.array_equal(inv, pos)


def blelloch_exclusive_scan(data):
    """Work-efficient up-sweep / down-sweep on a power-of-two array."""
    a = list(data)
    size = len(a)
    stride = 1
    while stride < size:
        for t in range(size):
            idx = (t + 1) * stride * 2 - 1
            if idx < size:
                a[idx] += a[idx - stride]
        stride <<= 1
    a[size - 1] = 0
    stride = size // 2
    while stride > 0:
        for t in range(size):
            idx = (t + 1) * stride * 2 - 1
            if idx < size:
                a[idx - stride], a[idx] = a[idx], a[idx] + a[idx - stride]
        stride >>= 1
    return a


def pin_blelloch_scan(lib=None):
    rng = np.random.default_rng(3)
    for size in (8, 16, 256):
        x = rng.integers(0, 1000, size=size).astype(np.uint64)
        assert oracle.exclusive_scan(x, lib=lib).tolist() == blelloch_exclusive_scan(x.tolist())


def pin_f32_invariants(lib=None):
    rng = np.random.default_rng(9)
    table = BOUNDARY_F32 + [int(v) for v in synth.f32_edge(200, 77)]
    keys = np.array(table, dtype=np.uint32)
    ordk = oracle.ordered_keys("f32", keys, lib=lib).tolist()
    ref = [f32_order_key(int(b)) for b in keys]
    for i in range(len(table)):
        for j in range(len(table)):
            assert (ordk[i] < ordk[j]) == (ref[i] < ref[j]), (hex(table[i]), hex(table[j]))
            assert (ordk[i] == ordk[j]) == (ref[i] == ref[j]), (hex(table[i]), hex(table[j]))
    # every NaN and both infinities take the single maximum code; nothing finite does
    for b in table:
        special = ((b >> 23) & 0xFF) == 0xFF
        o = int(oracle.ordered_keys("f32", np.array([b], dtype=np.uint32), lib=lib)[0])
        assert (o == 0xFFFFFFFF) == special, hex(b)
    del rng


def pin_i32_invariants(lib=None):
    rng = np.random.default_rng(21)
    table = BOUNDARY_I32 + rng.integers(0, 2**32, size=100, dtype=np.uint64).tolist()
    keys = np.array(table, dtype=np.uint32)
    ordk = oracle.ordered_keys("i32", keys, lib=lib).tolist()
    vals = [i32_value(int(b)) for b in keys]
    for i in range(len(table)):
        for j in range(len(table)):
            assert (ordk[i] < ordk[j]) == (vals[i] < vals[j]), (hex(table[i]), hex(table[j]))


def _check_against_brute(key_type, keys, begin_bit, end_bit, lib=None, radix_bits=8, descending=False):
    n = len(keys)
    vals = np.arange(n, dtype=np.uint32)
    want = brute_force_perm(key_type, keys, begin_bit, end_bit, descending)
    ko, vo = oracle.sort(key_type, keys, vals, begin_bit, end_bit, radix_bits=radix_bits, lib=lib,
                         descending=descending)
    assert vo.tolist() == want
    assert ko.tolist() == [int(keys[i]) for i in want]
    ko2, _ = oracle.sort(key_type, keys, None, begin_bit, end_bit, radix_bits=radix_bits, lib=lib,
                         descending=descending)
    assert np.array_equal(ko, ko2)


def pin_brute_force(lib=None):
    rng = np.random.default_rng(1234)
    for n in (0, 1, 2, 3, 31, 300, 4096):
        u32 = synth.u32_uniform(n, 100 + n)
        _check_against_brute("u32", u32, 0, 32, lib)
        ties = synth.u32_bits(n, 200 + n, 5)                      # many equal keys
        _check_against_brute("u32", ties, 0, 32, lib)
        for _ in range(3):
            b = int(rng.integers(0, 32))
            e = int(rng.integers(b, 33))
            _check_against_brute("u32", u32, b, e, lib)
        _check_against_brute("i32", u32, 0, 32, lib)
        f = synth.f32_edge(n, 300 + n)
        _check_against_brute("f32", f, 0, 32, lib)
        u64 = synth.u64_uniform(n, 400 + n)
        _check_against_brute("u64", u64, 0, 64, lib)
        b = int(rng.integers(0, 64))
        e = int(rng.integers(b, 65))
        _check_against_brute("u64", u64, b, e, lib)


def pin_exhaustive_tiny(lib=None):
    alph = {
        "u32": [0, 0x80000001, 0xFFFFFFFF],
        "i32": [0xFFFFFFFF, 0, 0x80000000],
        "f32": [0x80000000, 0x00000000, 0x7FC00000],
        "u64": [0, 1 << 40, (1 << 64) - 1],
    }
    for kt, letters in alph.items():
        dt = oracle.KEY_DTYPE[kt]
        for n in range(0, 6):
            for combo in itertools.product(letters, repeat=n):
                _check_against_brute(kt, np.array(combo, dtype=dt), 0, oracle.KEY_BITS[kt], lib)


BOUNDARY_I16 = [0x8000, 0x8001, 0xFFFE, 0xFFFF, 0, 1, 2, 0x7FFE, 0x7FFF, 0x0100, 0xFF00, 0x4000, 0xC000]


def pin_f16_invariants(lib=None):
    table = [int(v) for v in synth.F16_BOUNDARY] + [int(v) for v in synth.f16_edge(150, 78)]
    keys = np.array(table, dtype=np.uint16)
    ordk = oracle.ordered_keys("f16", keys, lib=lib).tolist()
    ref = [f16_order_key(b) for b in table]
    for i in range(len(table)):
        for j in range(len(table)):
            assert (ordk[i] < ordk[j]) == (ref[i] < ref[j]), (hex(table[i]), hex(table[j]))
            assert (ordk[i] == ordk[j]) == (ref[i] == ref[j]), (hex(table[i]), hex(table[j]))
    for b in table:
        special = ((b >> 10) & 0x1F) == 0x1F
        assert (int(oracle.ordered_keys("f16", np.array([b], np.uint16), lib=lib)[0]) == 0xFFFF) == special


def pin_i16_invariants(lib=None):
    table = BOUNDARY_I16 + [int(v) for v in synth.u16_uniform(100, 22)]
    ordk = oracle.ordered_keys("i16", np.array(table, dtype=np.uint16), lib=lib).tolist()
    vals = [i16_value(b) for b in table]
    for i in range(len(table)):
        for j in range(len(table)):
            assert (ordk[i] < ordk[j]) == (vals[i] < vals[j]), (hex(table[i]), hex(table[j]))


def pin_brute_force_16bit(lib=None):
    rng = np.random.default_rng(99)
    for n in (0, 1, 2, 31, 300, 2000):
        u16 = synth.u16_uniform(n, 500 + n)
        _check_against_brute("u16", u16, 0, 16, lib)
        _check_against_brute("u16", u16 & np.uint16(0x0F0F), 0, 16, lib)     # many ties
        b = int(rng.integers(0, 16))
        e = int(rng.integers(b, 17))
        _check_against_brute("u16", u16, b, e, lib)
        _check_against_brute("i16", u16, 0, 16, lib)
        _check_against_brute("f16", synth.f16_edge(n, 600 + n), 0, 16, lib)
        _check_against_brute("f16", synth.f16_normal_specials(n, 700 + n), 0, 16, lib, radix_bits=4)


def pin_descending(lib=None):
    rng = np.random.default_rng(7)
    for n in (0, 1, 2, 3, 64, 777):
        u32 = synth.u32_uniform(n, 800 + n)
        _check_against_brute("u32", u32, 0, 32, lib, descending=True)
        _check_against_brute("u32", synth.u32_bits(n, 801 + n, 4), 0, 32, lib, descending=True)  # ties
        b = int(rng.integers(0, 32))
        e = int(rng.integers(b, 33))
        _check_against_brute("u32", u32, b, e, lib, descending=True, radix_bits=5)
        _check_against_brute("i32", u32, 0, 32, lib, descending=True)
        _check_against_brute("f32", synth.f32_edge(n, 802 + n), 0, 32, lib, descending=True)
        _check_against_brute("u64", synth.u64_uniform(n, 803 + n), 0, 64, lib, descending=True)
        _check_against_brute("u16", synth.u16_uniform(n, 804 + n), 3, 13, lib, descending=True)
        _check_against_brute("i16", synth.u16_uniform(n, 805 + n), 0, 16, lib, descending=True)
        _check_against_brute("f16", synth.f16_edge(n, 806 + n), 0, 16, lib, descending=True)
    for kt, letters in {"u32": [0, 7, 0xFFFFFFFF], "f16": [0x8000, 0x0000, 0x7E00]}.items():
        dt = oracle.KEY_DTYPE[kt]
        for n in range(0, 6):
            for combo in itertools.product(letters, repeat=n):
                _check_against_brute(kt, np.array(combo, dtype=dt), 0, oracle.KEY_BITS[kt], lib,
                                     descending=True)


def pin_f32_specials_keep_order(lib=None):
    # -Inf, +Inf and NaNs of any payload all tie at the top and keep input order
    keys = np.array([0x7FC00000, 0x3F800000, 0xFF800000, 0x7F800000, 0xBF800000, 0xFFC00001,
                     0x80000000, 0x00000000], dtype=np.uint32)
    ko, vo = oracle.sort("f32", keys, np.arange(8, dtype=np.uint32), lib=lib)
    assert vo.tolist() == [4, 6, 7, 1, 0, 2, 3, 5]


ALL_PINS = [pin_decimal_example, pin_one_bit_split, pin_global_position, pin_digit_major_scan,
            pin_blelloch_scan, pin_f32_invariants, pin_i32_invariants, pin_brute_force,
            pin_exhaustive_tiny, pin_f32_specials_keep_order, pin_f16_invariants,
            pin_i16_invariants, pin_brute_force_16bit, pin_descending]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_one_bit_path_agrees_with_counting_path():
    for kt, keys in [("f32", synth.f32_edge(3000, 8)), ("i32", synth.u32_uniform(3000, 9)),
                     ("u64", synth.u64_uniform(1000, 10))]:
        vals = np.arange(len(keys), dtype=np.uint32)
        a = oracle.sort(kt, keys, vals)
        b = oracle.one_bit_split_sort(kt, keys, vals)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_std_stable_sort_agrees_with_the_oracle():
    # One std::stable_sort of (ordered key bits, index) records solves the same
    # problem by comparison; it must give the oracle's keys and payload order
    # for every key type, random bit ranges and both orders (ties in input
    # order, "Radix sort paralelo sobre el scan", La idea y el requisito de
    # estabilidad).  Small alphabets force many ties.
    rng = np.random.default_rng(2024)
    for kt, bits in [("u32", 32), ("i32", 32), ("f32", 32), ("u64", 64), ("u16", 16), ("i16", 16),
                     ("f16", 16)]:
        for trial in range(4):
            n = int(rng.integers(1, 3000))
            if kt == "f32":
                keys = synth.f32_edge(n, 100 + trial)
            elif bits == 64:
                keys = synth.u64_uniform(n, 200 + trial)
            else:
                raw = synth.u32_uniform(n, 300 + trial)
                if trial % 2:
                    raw = raw & np.uint32(0x0F0F000F)  # few distinct values: ties
                keys = raw.astype(np.uint16) if bits == 16 else raw
            b = int(rng.integers(0, bits + 1))
            e = int(rng.integers(b, bits + 1))
            vals = np.arange(n, dtype=np.uint32)
            for desc in (False, True):
                want = oracle.sort(kt, keys, vals, b, e, descending=desc)
                got = oracle.stable_sort_baseline(kt, keys, vals, b, e, descending=desc)
                assert np.array_equal(want[0], got[0]) and np.array_equal(want[1], got[1]), (kt, b, e, desc)


def test_parallel_baseline_agrees_with_the_oracle():
    # The multi-threaded CPU baseline (one block per thread, digit-major scan
    # of the blocks' counts) must give the oracle's keys and payload order on
    # any number of threads, including more threads than keys.
    rng = np.random.default_rng(77)
    for kt, bits in [("u32", 32), ("i32", 32), ("f32", 32), ("u64", 64), ("u16", 16), ("f16", 16)]:
        n = int(rng.integers(1, 5000))
        if kt == "f32":
            keys = synth.f32_edge(n, 400)
        elif bits == 64:
            keys = synth.u64_uniform(n, 401)
        else:
            raw = synth.u32_uniform(n, 402) & np.uint32(0x0F0F0F0F)
            keys = raw.astype(np.uint16) if bits == 16 else raw
        b = int(rng.integers(0, bits))
        e = int(rng.integers(b, bits + 1))
        vals = np.arange(n, dtype=np.uint32)
        want = oracle.sort(kt, keys, vals, b, e)
        for threads in (1, 2, 7, 64):
            got = oracle.parallel_lsd_sort(kt, keys, vals, b, e, threads=threads)
            assert np.array_equal(want[0], got[0]) and np.array_equal(want[1], got[1]), (kt, b, e, threads)


def test_digit_width_does_not_change_result():
    keys = synth.u32_uniform(5000, 12)
    ref = oracle.sort("u32", keys, np.arange(5000, dtype=np.uint32), 3, 29, radix_bits=8)
    for r in (1, 3, 4, 5, 11, 16):
        got = oracle.sort("u32", keys, np.arange(5000, dtype=np.uint32), 3, 29, radix_bits=r)
        assert np.array_equal(ref[1], got[1]), r


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.sort("u32", np.zeros(4, np.uint32), None, 5, 3)
    with pytest.raises(ValueError):
        oracle.sort("u32", np.zeros(4, np.uint32), None, 0, 33)
    with pytest.raises(ValueError):
        oracle.sort("u64", np.zeros(4, np.uint64), None, 0, 65)


# ------------------------------------------------------- planted mistakes

MUTANTS = {
    # walks each bucket back to front: still a permutation, but not stable
    "unstable_placement": ("uint64_t j = start[digit[i]]++;",
                           "uint64_t j = start[digit[i]] + count[digit[i]] - 1; count[digit[i]]--;"),
    # drops the NaN/Inf rule of the float map
    "no_special_values": ("    if ((bits & 0x7F800000u) == 0x7F800000u)\n        return 0xFFFFFFFFu;\n", ""),
    # flips all bits of negative ints (reverses the order of negatives)
    "int_flip_all": ("uint32_t oracle_ordered_i32(uint32_t bits)\n{\n    return bits ^ 0x80000000u;",
                     "uint32_t oracle_ordered_i32(uint32_t bits)\n{\n"
                     "    return (bits & 0x80000000u) ? ~bits : (bits ^ 0x80000000u);"),
    # forgets the sign bit of positive floats
    "float_positive_unshifted": ("        return ~bits;\n    return bits ^ 0x80000000u;",
                                 "        return ~bits;\n    return bits;"),
    # does not cut the last digit at end_bit
    "last_digit_uncut": ("int width = end_bit - lo < radix_bits ? end_bit - lo : radix_bits;",
                         "int width = radix_bits;"),
    # drops the NaN/Inf rule of the binary16 map
    "no_special_values_f16": ("    if ((bits & 0x7C00u) == 0x7C00u)\n        return 0xFFFFu;\n", ""),
    # flips all bits of negative int16 keys
    "int16_flip_all": ("    return (bits ^ 0x8000u) & 0xFFFFu;",
                       "    return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits ^ 0x8000u);"),
    # sorts ascending whatever was asked
    "descending_ignored": ("const uint64_t flip = descending ? mask : 0;", "const uint64_t flip = 0;"),
    # reverses only the lowest digit (a per-pass mistake the full-key checks see)
    "descending_first_pass_only": ("const uint64_t flip = descending ? mask : 0;",
                                   "const uint64_t flip = (descending && lo == begin_bit) ? mask : 0;"),
    # one-bit split fills the ones from the back (a permutation, but not stable)
    "one_bit_ones_reversed": ("uint64_t dst = one ? F + (uint64_t)i - s[i] : s[i];",
                              "uint64_t dst = one ? (uint64_t)n - 1 - ((uint64_t)i - s[i]) : s[i];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"liboracle_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(path)])
    lib = oracle.load_variant(str(so))
    failures = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failures.append(pin.__name__)
    assert failures, f"no pin caught the planted mistake {name}"
