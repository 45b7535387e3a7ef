"""The range-checked build (RS_CHECKED=1) on the GPU.

RS_CHECKED=1 makes every tile kernel also record, in the device error word,
any shuffle position that had to be clamped into its tile (the clamp itself
and the scatter's bounds check are always on).  This builds that variant of
the library into a scratch folder, sorts with every schedule (one cluster
kernel, chained scan, reduce-then-scan), keys only and with values, several
key types and both digit widths, and checks each result against the CPU
oracle bit for bit and the device error word for RS_OK.  The variant runs in
a child process so that this process keeps the ordinary library.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
import lsd_radix_sort_key_gb300 as rs
rs.LIB_PATH = LIB
import oracle, synth
dev = "cuda:0"
out = []
cases = [
    # key type, n, values, begin, end, schedule, digit bits
    ("u32", 40_000, False, 0, 32, "cluster", 8),
    ("f32", 40_000, True, 0, 32, "cluster", 4),
    ("u32", 300_001, False, 0, 32, "onesweep", 8),
    ("i32", 300_001, True, 0, 32, "onesweep", 8),
    ("u64", 200_003, True, 3, 61, "onesweep", 4),
    ("u32", 1_000_003, False, 0, 32, "reduce_scan", 8),
    ("f32", 1_000_003, True, 0, 32, "reduce_scan", 8),
    ("u64", 500_001, False, 0, 64, "reduce_scan", 8),
    ("u16", 700_001, True, 0, 16, "reduce_scan", 4),
]
for kt, n, with_vals, b, e, algo, rb in cases:
    if kt == "u64":
        keys = synth.u64_uniform(n, 41); tk = torch.from_numpy(keys.view(np.int64))
    elif kt == "u16":
        keys = (synth.u32_uniform(n, 42) & 0xFFFF).astype(np.uint16); tk = torch.from_numpy(keys.view(np.int16))
    elif kt == "f32":
        keys = synth.f32_normal_specials(n, 43, per_special=50); tk = torch.from_numpy(keys.view(np.int32))
    else:
        keys = synth.u32_uniform(n, 44); tk = torch.from_numpy(keys.view(np.int32))
    vals = synth.iota_u32(n) if with_vals else None
    kin = tk.to(dev)
    vin = torch.from_numpy(vals.view(np.int32)).to(dev) if with_vals else None
    tb = rs.rs_temp_bytes(kt, bool(with_vals), n, b, e)
    temp = torch.empty(tb, dtype=torch.uint8, device=dev)
    kout, vout = rs.sort(kin, vin, key_type=kt, begin_bit=b, end_bit=e, algo=algo, radix_bits=rb, temp=temp)
    status = rs.rs_device_status(temp)
    want_k, want_v = oracle.sort(kt, keys, vals, b, e)
    ok = np.array_equal(kout.cpu().numpy().view(want_k.dtype), want_k)
    if with_vals:
        ok = ok and np.array_equal(vout.cpu().numpy().view(np.uint32), want_v)
    out.append({"case": f"{kt}/{n}/{int(with_vals)}/{b}-{e}/{algo}/r{rb}", "ok": bool(ok), "status": status})
print("RESULT " + json.dumps(out))
"""


def test_checked_build_sorts_every_schedule_cleanly(tmp_path):
    from lsd_radix_sort_key_gb300 import _build
    lib = _build.build(force=True, extra_flags=["-DRS_CHECKED=1"], libdir=str(tmp_path / "checked"))
    code = f"ROOT={ROOT!r}\nLIB={lib!r}\n" + CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")]
    assert line, r.stdout[-2000:]
    results = json.loads(line[0][7:])
    assert len(results) == 9
    for res in results:
        assert res["ok"], res
        assert res["status"] == 0, res
