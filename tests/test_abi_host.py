"""The C-ABI library on the CPU: it loads, exports every declared symbol, and
rejects bad arguments before touching the GPU (no CUDA call is reached)."""
import ctypes
import os
import re

import pytest

import lsd_radix_sort_key_gb300 as rs
from lsd_radix_sort_key_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return rs.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(rs_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "rs_sort_keys_u32" in names and "rs_temp_bytes" in names
    for name in names:
        assert hasattr(lib, name), name
        assert name in rs.SIGNATURES, f"binding lacks a signature for {name}"


def test_temp_bytes_layout(lib):
    n = 1 << 20
    t = rs.rs_temp_bytes("u32", False, n, 0, 32)
    assert t >= 4 * n  # at least the ping-pong buffer
    assert rs.rs_temp_bytes("u32", True, n, 0, 32) >= t + 4 * n
    assert rs.rs_temp_bytes("u64", True, n, 0, 64) > rs.rs_temp_bytes("u32", True, n, 0, 32)
    assert rs.rs_temp_bytes("u32", False, 0, 0, 32) == 0
    bad = ctypes.c_size_t(-1).value
    assert rs.rs_temp_bytes("u32", False, 10, 0, 33) == bad
    assert rs.rs_temp_bytes("u32", False, 10, 5, 4) == bad
    assert rs.rs_temp_bytes("u64", False, 10, 0, 65) == bad
    assert rs.rs_temp_bytes("u32", False, 1 << 33, 0, 32) == bad


def test_kernel_counts(lib):
    def count(kt, n, b, e, algo, rb=0, vals=False, vbytes=0):
        v = 0x3 << 40 if vals else None
        vo = 0x4 << 40 if vals else None
        return rs.rs_sort_kernel_count(rs.make_desc(kt, None, None, v, vo, n, b, e, None, 0, 0,
                                                    algo, rb, value_bytes=vbytes))
    assert count("u32", 1 << 20, 0, 32, "onesweep") == 1 + 4
    assert count("u32", 1 << 20, 0, 30, "onesweep") == 1 + 4
    assert count("u32", 1 << 20, 0, 32, "onesweep", 4) == 1 + 8
    assert count("u64", 1 << 20, 0, 64, "onesweep", vals=True) == 1 + 8
    assert count("u32", 1 << 20, 0, 32, "reduce_scan") == 3 * 4
    assert count("u32", 1 << 20, 7, 7, "onesweep") == 0
    assert count("u32", 0, 0, 32, "onesweep") == 0
    # AUTO: chained scan below 2^22 keys (2^23 for 32-bit keys with values
    # and for 64-bit keys alone), reduce-then-scan from there on; 64-bit keys
    # with 64-bit values always take the chained scan (below its 2^30 limit)
    assert count("u32", 1 << 20, 0, 32, "auto") == 5
    assert count("u32", (1 << 22) - 1, 0, 32, "auto") == 5
    assert count("u32", 1 << 22, 0, 32, "auto") == 12
    assert count("u64", (1 << 22) - 1, 0, 64, "auto", vals=True) == 9
    assert count("u64", 1 << 22, 0, 64, "auto", vals=True) == 24
    assert count("u64", 1 << 22, 0, 64, "auto") == 9
    assert count("u64", (1 << 23) - 1, 0, 64, "auto") == 9
    assert count("u64", 1 << 23, 0, 64, "auto") == 24
    assert count("u32", 1 << 22, 0, 32, "auto", vals=True) == 5
    assert count("u32", 1 << 23, 0, 32, "auto", vals=True) == 12
    assert count("u32", 1 << 22, 0, 32, "auto", vals=True, vbytes=8) == 5
    assert count("u32", 1 << 23, 0, 32, "auto", vals=True, vbytes=8) == 12
    assert count("u64", 1 << 28, 0, 64, "auto", vals=True, vbytes=8) == 9
    assert count("u16", 1 << 22, 0, 16, "auto", vals=True) == 6
    assert count("u32", 1 << 26, 0, 32, "auto") == 12
    assert count("u32", 1 << 26, 0, 32, "auto", vals=True) == 12
    assert count("u64", 1 << 26, 0, 64, "auto") == 24
    assert count("u32", 1 << 30, 0, 32, "auto") == 12
    # The cluster schedule: one kernel up to its capacity, refused above it.
    assert count("u32", 1 << 16, 0, 32, "auto") == 1
    assert count("u32", 1000, 0, 32, "cluster") == 1
    assert count("u32", (1 << 16) + 1, 0, 32, "cluster") == -1
    assert count("u32", (1 << 16) + 1, 0, 32, "auto") == 1 + 4
    # In place: one more kernel, the copy back from temp after an odd number
    # of running passes (it returns at once otherwise).
    fake = 1 << 40
    inplace = rs.make_desc("u32", fake, fake, None, None, 1 << 20, 0, 32, None, 0, 0, "onesweep")
    assert rs.rs_sort_kernel_count(inplace) == 1 + 4 + 1
    inplace = rs.make_desc("u32", fake, fake, None, None, 1 << 26, 0, 24, None, 0, 0, "reduce_scan")
    assert rs.rs_sort_kernel_count(inplace) == 3 * 3 + 1


FAKE = 1 << 40  # 256-byte aligned addresses that are never dereferenced


def desc(**kw):
    n = kw.pop("n", 1000)
    base = dict(key_type="u32", keys_in=FAKE, keys_out=2 * FAKE, vals_in=None, vals_out=None,
                n=n, begin_bit=0, end_bit=32, temp=3 * FAKE,
                temp_bytes=rs.rs_temp_bytes("u32", True, n, 0, 32), stream=0)
    base.update(kw)
    return rs.make_desc(base["key_type"], base["keys_in"], base["keys_out"], base["vals_in"],
                        base["vals_out"], base["n"], base["begin_bit"], base["end_bit"],
                        base["temp"], base["temp_bytes"], base["stream"],
                        kw.get("algo", "auto"), kw.get("radix_bits", 0), 0, kw.get("stall_tile", 0))


@pytest.mark.parametrize("kw,code", [
    (dict(keys_in=None), 1),
    (dict(keys_out=None), 1),
    (dict(temp=None), 1),
    (dict(begin_bit=-1), 1),
    (dict(end_bit=33), 1),
    (dict(begin_bit=9, end_bit=8), 1),
    (dict(key_type="u64", end_bit=65), 1),
    (dict(radix_bits=5), 1),
    (dict(vals_in=4 * FAKE), 1),                      # values in without values out
    (dict(keys_in=FAKE + 2), 1),                      # misaligned for 4-byte keys
    (dict(temp=3 * FAKE + 16), 1),                    # temp not 256-byte aligned
    (dict(temp_bytes=100), 2),
    (dict(keys_out=FAKE + 4 * 500), 3),               # partial overlap
    (dict(temp=FAKE + 256), 3),                       # temp overlaps the input
    (dict(n=1 << 31, algo="onesweep"), 7),            # chained scan limited to n < 2^30
    (dict(n=(1 << 16) + 1, algo="cluster"), 7),       # cluster sort limited to its capacity
])
def test_argument_errors(lib, kw, code):
    d = desc(**kw)
    assert rs.rs_sort(d) == code


def test_n_zero_is_a_no_op(lib):
    # n == 0 needs no buffers and launches nothing
    assert rs.rs_sort(desc(n=0, keys_in=None, keys_out=None, temp=None, temp_bytes=0)) == 0
    assert rs.rs_sort_keys_u32(None, None, 0, 0, 32, None, 0, 0) == 0


def test_typed_entry_points_validate(lib):
    assert rs.rs_sort_keys_u32(FAKE, 2 * FAKE, 100, 0, 40, 3 * FAKE, 1 << 30, 0) == 1
    assert rs.rs_sort_pairs_f32(FAKE, 2 * FAKE, None, 4 * FAKE, 100, 0, 32, 3 * FAKE, 1 << 30, 0) == 1
    assert rs.rs_sort_keys_u64(FAKE, 2 * FAKE, 100, 0, 64, 3 * FAKE, 10, 0) == 2


def test_cluster_capacity(lib):
    # 16 CTAs x one 512-thread tile: 8 uint32 keys per thread, 6 with values
    # or for uint64 keys, 4 for uint64 keys with values.
    assert rs.rs_cluster_max_n("u32", False) == 16 * 512 * 8
    assert rs.rs_cluster_max_n("f32", True) == 16 * 512 * 6
    assert rs.rs_cluster_max_n("u64", False) == 16 * 512 * 6
    assert rs.rs_cluster_max_n("u64", True) == 16 * 512 * 4


def test_64bit_values_shape_and_checks(lib):
    n = 1 << 20
    assert rs.rs_temp_bytes("u32", 8, n, 0, 32) >= rs.rs_temp_bytes("u32", True, n, 0, 32) + 4 * n
    assert rs.rs_cluster_max_n("u32", 8) == 16 * 512 * 4
    assert rs.rs_cluster_max_n("u64", 8) == 16 * 512 * 3
    tb = rs.rs_temp_bytes("u32", 8, 1000, 0, 32)

    def d(**kw):
        base = dict(vals_in=4 * FAKE, vals_out=5 * FAKE, value_bytes=8)
        base.update(kw)
        return rs.make_desc("u32", FAKE, 2 * FAKE, base["vals_in"], base["vals_out"], 1000, 0, 32,
                            3 * FAKE, tb, 0, "onesweep", 0, value_bytes=base["value_bytes"])
    assert rs.rs_sort_kernel_count(d()) == 1 + 4
    assert rs.rs_sort(d(value_bytes=3)) == 1                     # not 0, 4 or 8
    assert rs.rs_sort(d(vals_in=4 * FAKE + 4)) == 1              # 4-byte aligned, needs 8
    # the same buffer holds 1000 uint64 values only if temp was sized for them
    assert rs.rs_sort(rs.make_desc("u32", FAKE, 2 * FAKE, 4 * FAKE, 5 * FAKE, 1000, 0, 32, 3 * FAKE,
                                   rs.rs_temp_bytes("u32", True, 1000, 0, 32), 0, "onesweep", 0,
                                   value_bytes=8)) == 2


def test_host_batches_shape_and_checks(lib):
    n = 1000
    assert rs.rs_host_batches_work_bytes("u32", False, n, 0, 32) >= 2 * rs.rs_host_work_bytes("u32", False, n, 0, 32)
    assert rs.rs_host_batches_work_bytes("u32", False, n, 0, 40) == 2**64 - 1   # bad bit range
    assert rs.rs_host_batches_work_bytes("u32", False, 0, 0, 32) == 0
    wb = rs.rs_host_batches_work_bytes("u32", True, n, 0, 32)
    ins, outs = [FAKE, 2 * FAKE], [3 * FAKE, 4 * FAKE]
    vin, vout = [5 * FAKE, 6 * FAKE], [7 * FAKE, 8 * FAKE]

    def call(k_in=ins, k_out=outs, v_in=vin, v_out=vout, n=n, work=9 * FAKE, wbytes=wb, e=32):
        return rs.rs_sort_host_batches("u32", k_in, k_out, v_in, v_out, n, 0, e, work, wbytes, 0)
    assert call(e=33) == 1                                   # bad bit range
    assert call(k_out=[3 * FAKE, None]) == 1                 # a NULL output
    assert call(v_in=[5 * FAKE, None]) == 1                  # a NULL value input
    assert call(v_out=None) == 1                             # values in but not out
    assert call(work=None) == 1                              # no work buffer
    assert call(k_in=[], k_out=[], v_in=[], v_out=[]) == 0   # no batches: nothing to do
    assert call(n=0) == 0                                    # empty batches: nothing to do
    assert lib.rs_sort_host_batches(0, -1, None, None, None, None, n, 0, 32, FAKE, wb, None) == 1
    with pytest.raises(ValueError):
        call(k_out=[3 * FAKE])


def test_status_strings(lib):
    for code in range(8):
        assert rs.rs_status_string(code)
    assert rs.rs_status_string(99) == "unknown status"


def test_product_path_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(rs, "_lib", None)
    monkeypatch.setattr(rs, "LIB_PATH", "/nonexistent/librs.so")
    with pytest.raises(RuntimeError, match="missing"):
        rs.lib()


def test_package_does_not_import_oracle():
    import subprocess
    import sys
    code = ("import sys; import lsd_radix_sort_key_gb300 as rs; "
            "assert 'oracle' not in sys.modules, 'product imported the oracle'")
    subprocess.check_call([sys.executable, "-c", code], cwd=ROOT)


def test_noalloc_limit_matches_the_header():
    # The binding's NOALLOC_MAX_N is a copy of RS_NOALLOC_MAX_N; the rejection
    # test on the GPU relies on the two agreeing.
    text = open(os.path.join(ROOT, "include", "rs.h")).read()
    m = re.search(r"#define\s+RS_NOALLOC_MAX_N\s+(\d+)", text)
    assert m and int(m.group(1)) == rs.NOALLOC_MAX_N
