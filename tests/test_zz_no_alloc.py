"""The allocation-free entry point (rs_sort_keys_u32_noalloc), for callers
that cannot allocate device memory where they sort.

Its output is checked bit for bit, on two calls in a row, against the CPU
oracle and against the ordinary entry point (rs_sort_keys_u32, with a
caller-provided temp) -- the tolerance every other sort test uses.  This file
is collected last on purpose.
"""
import numpy as np
import pytest

import lsd_radix_sort_key_gb300 as rs
import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def reference_sort(kin, n, begin_bit, end_bit):
    out = torch.empty_like(kin)
    tb = rs.rs_temp_bytes("u32", False, n, begin_bit, end_bit)
    temp = torch.empty(tb, dtype=torch.uint8, device=kin.device)
    assert rs.rs_sort_keys_u32(kin, out, n, begin_bit, end_bit, temp, tb) == 0
    return out


def test_noalloc_matches_the_temp_buffer_entry_point():
    rs.build()
    dev = "cuda:0"
    cases = [(rs.NOALLOC_MAX_N, 0, 32, 1), (1_000_003, 5, 29, 2)]  # two calls in a row
    outs = []
    for n, b, e, seed in cases:
        keys = synth.u32_uniform(n, 0xA110C + seed)
        kin = torch.from_numpy(keys.view(np.int32)).to(dev)
        kout = torch.full_like(kin, -1)
        assert rs.rs_sort_keys_u32_noalloc(kin, kout, n, b, e) == 0
        outs.append((kin, kout, n, b, e))
    torch.cuda.synchronize()
    for kin, kout, n, b, e in outs:
        want, _ = oracle.sort("u32", kin.cpu().numpy().view(np.uint32), None, b, e)
        assert np.array_equal(kout.cpu().numpy().view(np.uint32), want)
        ref = reference_sort(kin, n, b, e)
        torch.cuda.synchronize()
        assert torch.equal(kout, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    rs.build()
    dev = "cuda:0"
    kin = torch.zeros(16, dtype=torch.int32, device=dev)
    assert rs.rs_sort_keys_u32_noalloc(kin, kin, rs.NOALLOC_MAX_N + 1, 0, 32) == 1
    assert rs.rs_sort_keys_u32_noalloc(None, None, 0, 0, 32) == 0
