"""Helpers for the GPU tests: run the CUDA sort through the C ABI on numpy
inputs and return numpy outputs."""
import numpy as np

import lsd_radix_sort_key_gb300 as rs

NP_KEY = {"u32": np.uint32, "i32": np.uint32, "f32": np.uint32, "u64": np.uint64,
          "u16": np.uint16, "i16": np.uint16, "f16": np.uint16}
_VIEW = {8: np.int64, 4: np.int32, 2: np.int16}


def to_dev(a, dev):
    import torch
    if a is None:
        return None
    view = a.view(_VIEW[a.dtype.itemsize])
    return torch.from_numpy(np.ascontiguousarray(view)).to(dev)


def gpu_sort(kt, keys, vals=None, begin_bit=0, end_bit=None, algo="auto", radix_bits=0,
             dev="cuda:0", offset=0, in_place=False, check_status=True, want_record=False,
             descending=False):
    """Sort on the GPU via rs_sort; `offset` elements of padding before the
    input exercise unaligned pointers.  Returns (keys, vals) as numpy, plus
    the pass-skip record (differing_bits, unordered) if want_record."""
    import torch
    end_bit = rs.KEY_BITS[kt] if end_bit is None else end_bit
    n = len(keys)
    kb = rs.KEY_BYTES[kt]
    pad_k = np.zeros(offset, dtype=keys.dtype)
    kin_full = to_dev(np.concatenate([pad_k, keys]) if offset else keys, dev)
    kin = kin_full[offset:]
    vin = None
    if vals is not None:
        vin_full = to_dev(np.concatenate([np.zeros(offset, vals.dtype), vals]) if offset else vals, dev)
        vin = vin_full[offset:]
    if in_place:
        kout, vout = kin, vin
    else:
        kout = torch.empty_like(kin) if n else kin
        vout = None if vin is None else (torch.empty_like(vin) if n else vin)
    vb = 0 if vals is None else vals.dtype.itemsize
    tb = rs.rs_temp_bytes(kt, vb if vb else False, n, begin_bit, end_bit)
    temp = torch.empty(max(tb, 256), dtype=torch.uint8, device=dev)
    d = rs.make_desc(kt, kin if n else None, kout if n else None, vin if n else None,
                     vout if n else None, n, begin_bit, end_bit, temp, temp.numel(),
                     None, algo, radix_bits, descending=descending, value_bytes=vb)
    st = rs.rs_sort(d)
    assert st == 0, rs.STATUS.get(st, st)
    torch.cuda.synchronize()
    if check_status and n:
        assert rs.rs_device_status(temp) == 0
    ko = kout.cpu().numpy().view(NP_KEY[kt]) if n else np.empty(0, NP_KEY[kt])
    vdt = np.uint64 if vb == 8 else np.uint32
    vo = None if vals is None else (vout.cpu().numpy().view(vdt) if n else np.empty(0, vdt))
    assert kb == ko.dtype.itemsize
    if want_record:
        st, bits, unordered = rs.rs_skip_record(temp)
        assert st == 0
        return ko, vo, (bits, unordered)
    return ko, vo
