"""Stream order around a sort (needs a GPU).

Inside a sort, every kernel after the first is launched as a programmatic
dependent of the kernel before it; the first one is launched plainly.  These
tests put device work right before and right after each sort on the same
stream, with no host synchronisation in between: a copy writes the keys just
before the sort, a clone reads the result just after it, and a fill then
overwrites the input.  The sort must have seen the keys written before it,
and the work after it must see the whole sorted result, for every schedule,
keys only and with values, in place and out of place, several sorts back to
back on reused buffers.
"""
import numpy as np
import pytest

import lsd_radix_sort_key_gb300 as rs
import oracle
import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    rs.build()
    rs.lib()


CASES = [("cluster", 60_000), ("onesweep", 300_001), ("reduce_scan", 300_001), ("reduce_scan", (1 << 22) + 5),
         ("auto", (1 << 22) + 5)]


@pytest.mark.parametrize("algo,n", CASES)
@pytest.mark.parametrize("with_vals", [False, True])
@pytest.mark.parametrize("in_place", [False, True])
def test_work_before_and_after_each_sort(algo, n, with_vals, in_place):
    if algo == "cluster":
        n = min(n, rs.rs_cluster_max_n("u32", with_vals))
    dev = "cuda:0"
    seeds = [1300, 1301, 1302]
    keys = [synth.u32_uniform(n, sd) for sd in seeds]
    keys[1] = keys[1] & np.uint32(0x00FF00FF)  # two passes skipped in the middle sort
    vals = synth.u32_uniform(n, 1310) if with_vals else None
    srcs = [to_dev(k, dev) for k in keys]
    vsrc = to_dev(vals, dev) if with_vals else None
    kin = torch.empty_like(srcs[0])
    kout = kin if in_place else torch.empty_like(kin)
    vin = torch.empty_like(vsrc) if with_vals else None
    vout = (vin if in_place else torch.empty_like(vin)) if with_vals else None
    tb = rs.rs_temp_bytes("u32", with_vals, n, 0, 32)
    temp = torch.empty(tb, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    d = rs.make_desc("u32", kin, kout, vin, vout, n, 0, 32, temp, tb, s, algo)
    torch.cuda.synchronize()
    results = []
    with torch.cuda.stream(s):
        for src in srcs:
            kin.copy_(src)                      # written right before the sort
            if with_vals:
                vin.copy_(vsrc)
            assert rs.rs_sort(d) == 0
            results.append((kout.clone(), vout.clone() if with_vals else None))  # read right after
            kin.fill_(0)                        # the next writer of the buffers
            if with_vals:
                vin.fill_(0)
    s.synchronize()
    assert rs.rs_device_status(temp, s) == 0
    for i, ((ko, vo), k) in enumerate(zip(results, keys)):
        ref_k, ref_v = oracle.sort("u32", k, vals, 0, 32)
        assert np.array_equal(ko.cpu().numpy().view(np.uint32), ref_k), f"sort {i}: keys"
        if with_vals:
            assert np.array_equal(vo.cpu().numpy().view(np.uint32), ref_v), f"sort {i}: values"
