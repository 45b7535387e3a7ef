"""The largest n the library accepts, RS_MAX_N = 2^32 - 2^16 uint32 keys
(16 GiB per buffer), sorted on the GPU (needs a GPU and ~50 GB of device
and host memory; a minute or so).

At this size the oracle would take minutes per run, so the result is checked
by properties that hold at any size: the output is in order, and it is a
permutation of the input (equal sums of the keys and of their squares, mod
2^64, and equal counts of every value of the top byte).  Smaller sizes are
compared with the oracle element by element elsewhere.
"""
import numpy as np
import pytest

import lsd_radix_sort_key_gb300 as rs
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _fingerprint(a):
    """(sum, sum of squares) mod 2^64 and the top-byte histogram, in chunks."""
    s1 = s2 = np.uint64(0)
    top = np.zeros(256, dtype=np.int64)
    step = 1 << 28
    with np.errstate(over="ignore"):
        for i in range(0, a.size, step):
            c32 = a[i:i + step]
            c = c32.astype(np.uint64)
            s1 += np.sum(c, dtype=np.uint64)
            s2 += np.sum(c * c, dtype=np.uint64)
            top += np.bincount(c32 >> np.uint32(24), minlength=256)
    return int(s1), int(s2), top


def _in_order(a):
    step = 1 << 28
    for i in range(0, a.size - 1, step):
        c = a[i:i + step + 1]
        if not np.all(c[1:] >= c[:-1]):
            return False
    return True


def test_largest_n():
    n = rs.MAX_N
    free, _ = torch.cuda.mem_get_info()
    need = 3 * 4 * n + (1 << 28)
    if free < need:
        pytest.skip(f"needs {need >> 30} GiB of device memory, {free >> 30} free")
    keys = synth.u32_uniform(n, 0x5EED00FF)
    kin = torch.from_numpy(keys.view(np.int32)).to("cuda:0")
    ko, _ = rs.sort(kin, key_type="u32")
    assert rs.rs_sort_kernel_count(rs.make_desc("u32", None, None, None, None, n, 0, 32, None, 0, 0)) == 12
    torch.cuda.synchronize()
    out = ko.cpu().numpy().view(np.uint32)
    del kin, ko
    assert _in_order(out)
    f_in, f_out = _fingerprint(keys), _fingerprint(out)
    assert f_in[0] == f_out[0] and f_in[1] == f_out[1]
    assert np.array_equal(f_in[2], f_out[2])
