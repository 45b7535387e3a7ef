"""Bit-exact parity of the CUDA sort with the CPU oracle (needs a GPU).

Sizes span one tile, several tiles and a ragged tail for every key type, with
and without values, under both schedules and both digit widths; the edge
cases cover n = 0..2, empty and partial bit ranges, in-place sorts, unaligned
pointers, tie-heavy and low-entropy keys, float specials, the CUDA-graph, the
profiled and the host-buffer entry points, and the look-back timeout path.
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


def gen_keys(kt, n, seed):
    if kt == "u64":
        return synth.u64_uniform(n, seed)
    if kt == "f32":
        return synth.f32_edge(n, seed)
    return synth.u32_uniform(n, seed)


def check(kt, keys, vals, b, e, **kw):
    got_k, got_v = gpu_sort(kt, keys, vals, b, e, **kw)
    ref_k, ref_v = oracle.sort(kt, keys, vals, b, e)
    assert np.array_equal(got_k, ref_k), f"keys differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"
    if vals is not None:
        assert np.array_equal(got_v, ref_v), f"values differ ({kt}, n={len(keys)}, [{b},{e}), {kw})"


SIZES = [1, 2, 31, 3839, 3840, 3841, 50_000, (1 << 17) + 123]


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
@pytest.mark.parametrize("radix_bits", [8, 4])
@pytest.mark.parametrize("kt", ["u32", "i32", "f32", "u64"])
@pytest.mark.parametrize("with_vals", [False, True])
def test_full_range(algo, radix_bits, kt, with_vals):
    for i, n in enumerate(SIZES):
        keys = gen_keys(kt, n, 1000 + i)
        vals = synth.iota_u32(n) if with_vals else None
        check(kt, keys, vals, 0, rs.KEY_BITS[kt], algo=algo, radix_bits=radix_bits)


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
@pytest.mark.parametrize("kt", ["u32", "i32", "f32", "u64"])
def test_partial_bit_ranges(algo, kt):
    rng = np.random.default_rng(77)
    bits = rs.KEY_BITS[kt]
    n = 70_001
    keys = gen_keys(kt, n, 5)
    vals = synth.iota_u32(n)
    ranges = [(0, 1), (bits - 1, bits), (3, 3 + 8), (5, 5 + 13), (0, bits - 2)]
    ranges += [tuple(sorted(int(x) for x in rng.integers(0, bits + 1, size=2))) for _ in range(4)]
    for b, e in ranges:
        check(kt, keys, vals, b, e, algo=algo)


@pytest.mark.parametrize("kt", ["u32", "u64"])
def test_empty_bit_range_is_a_copy(kt):
    keys = gen_keys(kt, 10_000, 8)
    vals = synth.iota_u32(10_000)
    got_k, got_v = gpu_sort(kt, keys, vals, 7, 7)
    assert np.array_equal(got_k, keys) and np.array_equal(got_v, vals)


def test_tiny_and_empty():
    for n in (0, 1, 2):
        keys = synth.u32_uniform(n, 3)
        check("u32", keys, synth.iota_u32(n), 0, 32)


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
@pytest.mark.parametrize("end_bit", [32, 24])  # even and odd pass counts
def test_in_place(algo, end_bit):
    n = 100_003
    keys = synth.u32_uniform(n, 9)
    vals = synth.iota_u32(n)
    got_k, got_v = gpu_sort("u32", keys, vals, 0, end_bit, algo=algo, in_place=True)
    ref_k, ref_v = oracle.sort("u32", keys, vals, 0, end_bit)
    assert np.array_equal(got_k, ref_k) and np.array_equal(got_v, ref_v)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_pointers(offset):
    n = 40_000
    for kt in ("u32", "f32"):
        keys = gen_keys(kt, n, 10 + offset)
        got_k, _ = gpu_sort(kt, keys, None, 0, 32, offset=offset)
        assert np.array_equal(got_k, oracle.sort(kt, keys)[0])
    keys = synth.u64_uniform(n, 20 + offset)
    got_k, got_v = gpu_sort("u64", keys, synth.iota_u32(n), 0, 64, offset=offset)
    ref = oracle.sort("u64", keys, synth.iota_u32(n))
    assert np.array_equal(got_k, ref[0]) and np.array_equal(got_v, ref[1])


@pytest.mark.parametrize("algo", ["onesweep", "reduce_scan"])
def test_ties_and_low_entropy(algo):
    n = 200_000
    cases = [synth.u32_bits(n, 1, 3),         # 8 distinct keys: stability everywhere
             synth.u32_and4(n, 2),            # digit 0 holds ~60% of keys in every pass
             np.full(n, 0xDEADBEEF, np.uint32),
             np.zeros(n, np.uint32),
             np.arange(n, dtype=np.uint32)[::-1].copy(),
             np.arange(n, dtype=np.uint32)]
    for keys in cases:
        check("u32", keys, synth.iota_u32(n), 0, 32, algo=algo)


def test_float_specials_and_signed_zero():
    n = 300_000
    keys = synth.f32_normal_specials(n, 0x5EED0002)
    vals = synth.iota_u32(n)
    check("f32", keys, vals, 0, 32)
    got_k, got_v = gpu_sort("f32", keys, vals)
    f = got_k.view(np.float32)
    specials = ~np.isfinite(f)
    k = int(specials.sum())
    assert specials[n - k:].all()                      # NaN / +-Inf last ...
    assert np.all(np.diff(got_v[n - k:].astype(np.int64)) > 0)  # ... in input order
    zeros = np.nonzero(f == 0)[0]
    neg = got_k[zeros] == 0x80000000
    assert neg[: int(neg.sum())].all()                 # -0.0 before +0.0


@pytest.mark.parametrize("kt", ["u32", "i32", "f32", "u16"])
@pytest.mark.parametrize("descending", [False, True])
def test_keys_only_mixed_entropy_chunks(kt, descending):
    # Keys-only reduce-then-scan over chunks of different digit skew (uniform,
    # AND of 4, 8 distinct values, one repeated key, uniform), so the CTAs of
    # one pass see very different digit mixes.
    m = 300_001
    raw = np.concatenate([synth.u32_uniform(m, 41), synth.u32_and4(m, 42), synth.u32_bits(m, 1, 3),
                          np.full(m, 0x80000001, np.uint32), synth.u32_uniform(m + 777, 43)])
    keys = (raw >> np.uint32(16)).astype(np.uint16) if kt == "u16" else raw
    bits = 16 if kt == "u16" else 32
    got_k, _ = gpu_sort(kt, keys, None, 0, bits, algo="reduce_scan", descending=descending)
    assert np.array_equal(got_k, oracle.sort(kt, keys, None, 0, bits, descending=descending)[0])


@pytest.mark.parametrize("dist", ["uniform", "and4", "eight_values", "low_byte_only"])
@pytest.mark.parametrize("kt", ["u32", "f32", "u16"])
def test_keys_only_digit_skews(dist, kt):
    # Keys-only reduce-then-scan (the staged tiles) over uniform digits, AND-of-4
    # skew, eight distinct keys and keys whose upper bytes are all zero, both
    # orders.
    n = (1 << 20) + 77
    raw = {"uniform": synth.u32_uniform(n, 70), "and4": synth.u32_and4(n, 71),
           "eight_values": synth.u32_bits(n, 72, 3), "low_byte_only": synth.u32_uniform(n, 73) & np.uint32(0xFF)}[dist]
    keys = (raw >> np.uint32(16)).astype(np.uint16) if kt == "u16" and dist in ("uniform", "and4") \
        else raw.astype(np.uint16) if kt == "u16" else raw
    bits = rs.KEY_BITS[kt]
    for descending in (False, True):
        got_k, _ = gpu_sort(kt, keys, None, 0, bits, algo="reduce_scan", descending=descending)
        assert np.array_equal(got_k, oracle.sort(kt, keys, None, 0, bits, descending=descending)[0])


@pytest.mark.parametrize("kt,vals,bytes_per_key", [("u32", False, 4), ("u32", True, 8), ("u64", False, 8),
                                                   ("u64", True, 12), ("u16", False, 4)])
def test_chained_scan_tile_width_boundary(kt, vals, bytes_per_key):
    # The chained scan runs 256-thread tiles below 4 MiB of keys and values
    # (16-bit keys counted as 4 bytes) and 512-thread tiles from there: sort
    # just below and at the boundary.
    edge = (4 << 20) // bytes_per_key
    for i, n in enumerate((edge - 1, edge, edge + 1)):
        keys = synth.u16_uniform(n, 60 + i) if kt == "u16" else gen_keys(kt, n, 60 + i)
        check(kt, keys, synth.iota_u32(n) if vals else None, 0, rs.KEY_BITS[kt], algo="onesweep")


def test_many_tiles_onesweep_lookback():
    # > 256 tiles per pass, uneven tail: exercises long look-back chains
    n = (1 << 22) + 12345
    keys = synth.u32_uniform(n, 31)
    check("u32", keys, None, 0, 32, algo="onesweep")
    check("u32", keys, synth.iota_u32(n), 0, 32, algo="reduce_scan")


def test_typed_c_entry_points():
    dev = "cuda:0"
    n = 123_457
    for kt in ("u32", "i32", "f32", "u64"):
        keys = gen_keys(kt, n, 40)
        vals = synth.iota_u32(n)
        kin, vin = to_dev(keys, dev), to_dev(vals, dev)
        kout, vout = torch.empty_like(kin), torch.empty_like(vin)
        tb = rs.rs_temp_bytes(kt, True, n, 0, rs.KEY_BITS[kt])
        temp = torch.empty(tb, dtype=torch.uint8, device=dev)
        fn = getattr(rs, f"rs_sort_pairs_{kt}")
        assert fn(kin, kout, vin, vout, n, 0, rs.KEY_BITS[kt], temp, tb) == 0
        kout2 = torch.empty_like(kin)
        fk = getattr(rs, f"rs_sort_keys_{kt}")
        assert fk(kin, kout2, n, 0, rs.KEY_BITS[kt], temp, tb) == 0
        torch.cuda.synchronize()
        ref_k, ref_v = oracle.sort(kt, keys, vals)
        assert np.array_equal(kout.cpu().numpy().view(ref_k.dtype), ref_k)
        assert np.array_equal(vout.cpu().numpy().view(np.uint32), ref_v)
        assert np.array_equal(kout2.cpu().numpy().view(ref_k.dtype), ref_k)


def test_graph_replay():
    dev = "cuda:0"
    n = 1 << 16
    keys = synth.u32_uniform(n, 0x5EED0001)
    kin = to_dev(keys, dev)
    kout = torch.empty_like(kin)
    tb = rs.rs_temp_bytes("u32", False, n, 0, 32)
    temp = torch.empty(tb, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    d = rs.make_desc("u32", kin, kout, None, None, n, 0, 32, temp, tb, s)
    g = rs.Graph(d)
    ref = oracle.sort("u32", keys)[0]
    for _ in range(3):
        kout.zero_()
        torch.cuda.synchronize()
        g.launch(s)
        s.synchronize()
        assert np.array_equal(kout.cpu().numpy().view(np.uint32), ref)
    assert rs.rs_device_status(temp, s) == 0
    g.close()


def test_profiled_entry_point():
    dev = "cuda:0"
    n = 1 << 20
    keys = synth.u32_uniform(n, 50)
    kin = to_dev(keys, dev)
    kout = torch.empty_like(kin)
    tb = rs.rs_temp_bytes("u32", False, n, 0, 32)
    temp = torch.empty(tb, dtype=torch.uint8, device=dev)
    d = rs.make_desc("u32", kin, kout, None, None, n, 0, 32, temp, tb, None, "onesweep")
    events = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    st, kinds = rs.rs_sort_profiled(d, events)
    assert st == 0
    assert [rs.KERNEL_KINDS[k] for k in kinds] == ["histogram"] + ["onesweep_pass"] * 4
    torch.cuda.synchronize()
    times = [events[i].elapsed_time(events[i + 1]) for i in range(len(kinds))]
    assert all(t > 0 for t in times)
    assert np.array_equal(kout.cpu().numpy().view(np.uint32), oracle.sort("u32", keys)[0])


def test_profiled_sorts_captured_in_a_graph():
    # Under stream capture the events become graph nodes: every replay records
    # them, and the sorts inside the graph are still correct.
    dev = "cuda:0"
    n = 1 << 20
    keys = synth.u32_uniform(n, 51)
    kin = to_dev(keys, dev)
    kout = torch.empty_like(kin)
    tb = rs.rs_temp_bytes("u32", False, n, 0, 32)
    temp = torch.empty(tb, dtype=torch.uint8, device=dev)
    cap = torch.cuda.Stream()
    d = rs.make_desc("u32", kin, kout, None, None, n, 0, 32, temp, tb, cap, "reduce_scan")
    steps = [[torch.cuda.Event(enable_timing=True) for _ in range(14)] for _ in range(3)]
    for ev in steps:  # a plain run first: library caches filled outside the capture
        assert rs.rs_sort_profiled(d, ev)[0] == 0
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
        for ev in steps:
            st, kinds = rs.rs_sort_profiled(d, ev)
            assert st == 0
    kout.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert [rs.KERNEL_KINDS[k] for k in kinds] == ["upsweep", "spine_scan", "downsweep"] * 4
    for ev in steps:
        times = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(kinds))]
        assert all(t > 0 for t in times)
    assert np.array_equal(kout.cpu().numpy().view(np.uint32), oracle.sort("u32", keys)[0])
    assert rs.rs_device_status(temp) == 0


def test_host_buffer_entry_point():
    n = 200_001
    keys = synth.u64_uniform(n, 60)
    vals = synth.iota_u32(n)
    hk = torch.from_numpy(keys.view(np.int64)).pin_memory()
    hv = torch.from_numpy(vals.view(np.int32)).pin_memory()
    hko = torch.empty_like(hk).pin_memory()
    hvo = torch.empty_like(hv).pin_memory()
    wb = rs.rs_host_work_bytes("u64", True, n, 0, 64)
    work = torch.empty(wb, dtype=torch.uint8, device="cuda:0")
    assert rs.rs_sort_host("u64", hk, hko, hv, hvo, n, 0, 64, work, wb) == 0
    torch.cuda.synchronize()
    ref_k, ref_v = oracle.sort("u64", keys, vals)
    assert np.array_equal(hko.numpy().view(np.uint64), ref_k)
    assert np.array_equal(hvo.numpy().view(np.uint32), ref_v)


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # the refused capture records nothing
@pytest.mark.parametrize("kt,with_vals,batches", [("u32", False, 5), ("f32", True, 4), ("u64", True, 1),
                                                  ("i32", False, 2)])
def test_host_batches_entry_point(kt, with_vals, batches):
    """Pipelined host batches: every batch (distinct keys, both slots reused,
    an odd count ending in slot 0) equals the oracle's sort of it."""
    n = 150_001
    gen = {"u32": synth.u32_uniform, "i32": synth.u32_uniform, "f32": synth.f32_edge,
           "u64": synth.u64_uniform}[kt]
    keys = [gen(n, 80 + i) for i in range(batches)]
    vals = [synth.u32_uniform(n, 90 + i) for i in range(batches)] if with_vals else None
    pin = lambda a: torch.from_numpy(a.view(np.int64 if a.dtype == np.uint64 else np.int32)).pin_memory()
    hk = [pin(k) for k in keys]
    hko = [torch.empty_like(h).pin_memory() for h in hk]
    hv = [pin(v) for v in vals] if with_vals else None
    hvo = [torch.empty_like(h).pin_memory() for h in hv] if with_vals else None
    bits = rs.KEY_BITS[kt]
    wb = rs.rs_host_batches_work_bytes(kt, with_vals, n, 0, bits)
    work = torch.empty(wb, dtype=torch.uint8, device="cuda:0")
    stream = torch.cuda.Stream()
    assert rs.rs_sort_host_batches(kt, hk, hko, hv, hvo, n, 0, bits, work, wb, stream) == 0
    stream.synchronize()
    udt = np.uint64 if kt == "u64" else np.uint32
    for i in range(batches):
        ref_k, ref_v = oracle.sort(kt, keys[i], vals[i] if with_vals else None, 0, bits)
        assert np.array_equal(hko[i].numpy().view(udt), ref_k), f"batch {i} keys"
        if with_vals:
            assert np.array_equal(hvo[i].numpy().view(np.uint32), ref_v), f"batch {i} values"
    # too small a work buffer, and a capturing stream, are refused before any work
    assert rs.rs_sort_host_batches(kt, hk, hko, hv, hvo, n, 0, bits, work, wb - 1, stream) == 2
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        code = rs.rs_sort_host_batches(kt, hk, hko, hv, hvo, n, 0, bits, work, wb, stream)
    assert code == 7  # RS_ERR_UNSUPPORTED


def test_lookback_timeout_is_reported_and_recoverable():
    """Tile 3 never publishes: the waits behind it run out after a short bound,
    the sort reports RS_ERR_DEVICE_TIMEOUT, and the next sort is correct."""
    dev = "cuda:0"
    n = 64 * 3840
    keys = synth.u32_uniform(n, 70)
    kin = to_dev(keys, dev)
    kout = torch.empty_like(kin)
    tb = rs.rs_temp_bytes("u32", False, n, 0, 32)
    temp = torch.empty(tb, dtype=torch.uint8, device=dev)
    d = rs.make_desc("u32", kin, kout, None, None, n, 0, 32, temp, tb, None, "onesweep",
                     0, 2000, 4)
    assert rs.rs_sort(d) == 0
    assert rs.rs_device_status(temp) == 5  # RS_ERR_DEVICE_TIMEOUT
    d2 = rs.make_desc("u32", kin, kout, None, None, n, 0, 32, temp, tb, None, "onesweep")
    assert rs.rs_sort(d2) == 0
    assert rs.rs_device_status(temp) == 0
    assert np.array_equal(kout.cpu().numpy().view(np.uint32), oracle.sort("u32", keys)[0])
