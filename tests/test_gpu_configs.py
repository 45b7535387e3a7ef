"""Full-size workloads, bit-exact against the CPU oracle (needs a GPU).

Every workload runs at its full size in the launch configuration the bench
times (the default schedule and digit width), and the whole output is
compared with the oracle's, element by element.  The schedule the default
does not pick for 2^28 uint32 keys (the chained scan) is also checked at
that size, and the size sweep's largest point (2^29 uint32 keys) once.
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


def run_workload(w, algo="auto"):
    keys = w.keys()
    vals = w.values()
    got_k, got_v = gpu_sort(w.key_type, keys, vals, w.begin_bit, w.end_bit, algo=algo)
    ref_k, ref_v = oracle.sort(w.key_type, keys, vals, w.begin_bit, w.end_bit)
    bad = np.nonzero(got_k != ref_k)[0]
    assert bad.size == 0, f"{w.name}: {bad.size} keys differ, first at {bad[:5]}"
    if vals is not None:
        bad = np.nonzero(got_v != ref_v)[0]
        assert bad.size == 0, f"{w.name}: {bad.size} values differ, first at {bad[:5]}"


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_full_size(name):
    run_workload(synth.WORKLOADS[name])


def test_chained_scan_full_size():
    run_workload(synth.WORKLOADS["u32_uniform_2p28"], algo="onesweep")


def test_chained_scan_pairs_full_size():
    run_workload(synth.WORKLOADS["morton30_index_2p28"], algo="onesweep")


def test_sweep_largest_size():
    run_workload(synth.sweep_workload(29))
