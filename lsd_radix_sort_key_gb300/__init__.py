"""Python binding of the GB300 LSD radix sort (C ABI in include/rs.h).

Argument marshalling only: every step of the sort runs in the CUDA library
``_lib/librs.so``.  PyTorch supplies device memory and streams.  If the
library has not been built this module raises on first use -- there is no
fallback.

Low-level functions carry the C names (``rs_sort_keys_u32``, ``rs_sort_pairs_f32``,
``rs_temp_bytes``, ``rs_sort``, ...) and accept torch tensors or raw integer
addresses for pointers.  ``sort()`` is the convenience wrapper that allocates
outputs and temp with torch.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

KEY_TYPES = {"u32": 0, "i32": 1, "f32": 2, "u64": 3, "u16": 4, "i16": 5, "f16": 6}
KEY_BYTES = {"u32": 4, "i32": 4, "f32": 4, "u64": 8, "u16": 2, "i16": 2, "f16": 2}
KEY_BITS = {k: 8 * b for k, b in KEY_BYTES.items()}
ALGOS = {"auto": 0, "onesweep": 1, "reduce_scan": 2, "cluster": 3}
STATUS = {0: "RS_OK", 1: "RS_ERR_INVALID_ARG", 2: "RS_ERR_TEMP_TOO_SMALL", 3: "RS_ERR_ALIAS",
          4: "RS_ERR_CUDA", 5: "RS_ERR_DEVICE_TIMEOUT", 6: "RS_ERR_CHECK_FAILED",
          7: "RS_ERR_UNSUPPORTED"}
KERNEL_KINDS = {1: "histogram", 2: "onesweep_pass", 3: "upsweep", 4: "spine_scan",
                5: "downsweep", 6: "copy", 7: "cluster_sort"}
LIB_PATH = _build.LIB


class RadixSortError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class SortDesc(ctypes.Structure):
    """Mirror of rs_sort_desc."""
    _fields_ = [("key_type", ctypes.c_int), ("keys_in", ctypes.c_void_p),
                ("keys_out", ctypes.c_void_p), ("vals_in", ctypes.c_void_p),
                ("vals_out", ctypes.c_void_p), ("n", ctypes.c_size_t),
                ("begin_bit", ctypes.c_int), ("end_bit", ctypes.c_int), ("algo", ctypes.c_int),
                ("radix_bits", ctypes.c_int), ("temp", ctypes.c_void_p),
                ("temp_bytes", ctypes.c_size_t), ("stream", ctypes.c_void_p),
                ("spin_limit", ctypes.c_uint32), ("stall_tile", ctypes.c_int32),
                ("descending", ctypes.c_int), ("value_bytes", ctypes.c_int)]


_lib = None

# C signatures of every exported symbol (name -> (restype, argtypes)).
_vp, _sz, _i, _u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
_KEYS_SIG = (_i, [_vp, _vp, _sz, _i, _i, _vp, _sz, _vp])
_PAIRS_SIG = (_i, [_vp, _vp, _vp, _vp, _sz, _i, _i, _vp, _sz, _vp])
SIGNATURES = {
    "rs_temp_bytes": (_sz, [_i, _i, _sz, _i, _i]),
    "rs_sort": (_i, [ctypes.POINTER(SortDesc)]),
    "rs_sort_profiled": (_i, [ctypes.POINTER(SortDesc), ctypes.POINTER(_vp), _i,
                              ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "rs_sort_kernel_count": (_i, [ctypes.POINTER(SortDesc)]),
    "rs_device_status": (_i, [_vp, _vp]),
    "rs_skip_record": (_i, [_vp, _vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(_i)]),
    "rs_cluster_max_n": (_sz, [_i, _i]),
    "rs_status_string": (ctypes.c_char_p, [_i]),
    "rs_graph_create": (_i, [ctypes.POINTER(SortDesc), ctypes.POINTER(_vp)]),
    "rs_graph_launch": (_i, [_vp, _vp]),
    "rs_graph_destroy": (None, [_vp]),
    "rs_host_work_bytes": (_sz, [_i, _i, _sz, _i, _i]),
    "rs_sort_host": (_i, [_i, _vp, _vp, _vp, _vp, _sz, _i, _i, _vp, _sz, _vp]),
    "rs_host_batches_work_bytes": (_sz, [_i, _i, _sz, _i, _i]),
    "rs_sort_host_batches": (_i, [_i, _i, _vp, _vp, _vp, _vp, _sz, _i, _i, _vp, _sz, _vp]),
}
SIGNATURES["rs_sort_keys_u32_noalloc"] = (_i, [_vp, _vp, _sz, _i, _i, _vp])
SIGNATURES["rs_lbvh_build"] = (_i, [_vp, _sz, _vp, _vp, _vp, _vp, _vp, _vp, _vp])
LBVH_LEAF = 0x80000000
NOALLOC_MAX_N = 1 << 22
MAX_N = (1 << 32) - (1 << 16)  # RS_MAX_N
for _t in ("u32", "i32", "f32", "u64", "u16", "i16", "f16"):
    SIGNATURES[f"rs_sort_keys_{_t}"] = _KEYS_SIG
    SIGNATURES[f"rs_sort_pairs_{_t}"] = _PAIRS_SIG


def build(force: bool = False) -> str:
    return _build.build(force=force)


def lib():
    """The loaded CUDA library; raises if it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} is missing: run __graft_entry__.build() "
                               "(or python -m lsd_radix_sort_key_gb300._build) first")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != 0:
        raise RadixSortError(code, where)


# ---------------------------------------------------------- C-named wrappers

def _with_values(v) -> int:
    """C with_values argument: False/0 none, 8 uint64 values, True/4 uint32 values."""
    return 8 if (v is not True and v == 8) else int(bool(v))


def rs_temp_bytes(key_type: str, with_values, n: int, begin_bit: int, end_bit: int) -> int:
    """with_values: False, True (uint32 values) or 8 (uint64 values)."""
    return lib().rs_temp_bytes(KEY_TYPES[key_type], _with_values(with_values), n, begin_bit, end_bit)


def rs_host_work_bytes(key_type: str, with_values: bool, n: int, begin_bit: int, end_bit: int) -> int:
    return lib().rs_host_work_bytes(KEY_TYPES[key_type], int(bool(with_values)), n, begin_bit, end_bit)


def rs_status_string(code: int) -> str:
    return lib().rs_status_string(code).decode()


def _typed(name):
    def keys_fn(keys_in, keys_out, n, begin_bit, end_bit, temp, temp_bytes, stream=None):
        return getattr(lib(), f"rs_sort_keys_{name}")(
            _addr(keys_in), _addr(keys_out), n, begin_bit, end_bit, _addr(temp), temp_bytes,
            _stream(stream))

    def pairs_fn(keys_in, keys_out, vals_in, vals_out, n, begin_bit, end_bit, temp, temp_bytes,
                 stream=None):
        return getattr(lib(), f"rs_sort_pairs_{name}")(
            _addr(keys_in), _addr(keys_out), _addr(vals_in), _addr(vals_out), n, begin_bit,
            end_bit, _addr(temp), temp_bytes, _stream(stream))

    keys_fn.__name__ = f"rs_sort_keys_{name}"
    pairs_fn.__name__ = f"rs_sort_pairs_{name}"
    return keys_fn, pairs_fn


rs_sort_keys_u32, rs_sort_pairs_u32 = _typed("u32")
rs_sort_keys_i32, rs_sort_pairs_i32 = _typed("i32")
rs_sort_keys_f32, rs_sort_pairs_f32 = _typed("f32")
rs_sort_keys_u64, rs_sort_pairs_u64 = _typed("u64")
rs_sort_keys_u16, rs_sort_pairs_u16 = _typed("u16")
rs_sort_keys_i16, rs_sort_pairs_i16 = _typed("i16")
rs_sort_keys_f16, rs_sort_pairs_f16 = _typed("f16")


def rs_sort_keys_u32_noalloc(keys_in, keys_out, n, begin_bit, end_bit, stream=None):
    """uint32 keys-only sort whose scratch is a fixed device array inside the
    library (no allocation anywhere; n <= NOALLOC_MAX_N)."""
    return lib().rs_sort_keys_u32_noalloc(_addr(keys_in), _addr(keys_out), n, begin_bit, end_bit,
                                          _stream(stream))


def rs_lbvh_build(sorted_codes, n, left, right, first, last, leaf_parent, node_parent, stream=None) -> int:
    """The binary radix tree over n sorted uint32 codes (see include/rs.h)."""
    return lib().rs_lbvh_build(_addr(sorted_codes), n, _addr(left), _addr(right), _addr(first), _addr(last),
                               _addr(leaf_parent), _addr(node_parent), _stream(stream))


def lbvh_build(sorted_codes, stream=None) -> dict:
    """rs_lbvh_build with its outputs allocated by torch on the codes' device:
    a dict of int32 tensors (uint32 bit patterns) left, right, first, last,
    node_parent (n-1 each) and leaf_parent (n).  Enqueued on `stream`, not
    synchronised."""
    import torch
    if sorted_codes.element_size() != 4 or not sorted_codes.is_contiguous() or not sorted_codes.is_cuda:
        raise ValueError("codes must be a contiguous CUDA tensor of 4-byte elements")
    n = sorted_codes.numel()
    m = max(n - 1, 0)
    dev = sorted_codes.device
    out = {k: torch.empty(m, dtype=torch.int32, device=dev)
           for k in ("left", "right", "first", "last", "node_parent")}
    out["leaf_parent"] = torch.empty(n, dtype=torch.int32, device=dev)
    _check(rs_lbvh_build(sorted_codes, n, out["left"], out["right"], out["first"], out["last"],
                         out["leaf_parent"], out["node_parent"], stream), "rs_lbvh_build")
    return out


def make_desc(key_type, keys_in, keys_out, vals_in, vals_out, n, begin_bit, end_bit, temp,
              temp_bytes, stream=None, algo="auto", radix_bits=0, spin_limit=0, stall_tile=0,
              descending=False, value_bytes=0):
    return SortDesc(KEY_TYPES[key_type], _addr(keys_in), _addr(keys_out), _addr(vals_in),
                    _addr(vals_out), n, begin_bit, end_bit, ALGOS[algo], radix_bits, _addr(temp),
                    temp_bytes, _stream(stream), spin_limit, stall_tile, int(bool(descending)),
                    value_bytes)


def rs_sort(desc: SortDesc) -> int:
    return lib().rs_sort(ctypes.byref(desc))


def rs_sort_kernel_count(desc: SortDesc) -> int:
    return lib().rs_sort_kernel_count(ctypes.byref(desc))


def rs_sort_profiled(desc: SortDesc, events):
    """events: list of torch.cuda.Event(enable_timing=True); returns (status, kinds)."""
    for e in events:
        if e.cuda_event == 0:
            # torch creates events lazily; record once on the stream to create them
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    nk = ctypes.c_int(0)
    kinds = (ctypes.c_int * len(events))()
    st = lib().rs_sort_profiled(ctypes.byref(desc), arr, len(events), ctypes.byref(nk), kinds)
    return st, [kinds[i] for i in range(nk.value)]


def rs_device_status(temp, stream=None) -> int:
    return lib().rs_device_status(_addr(temp), _stream(stream))


def rs_cluster_max_n(key_type: str, with_values) -> int:
    """Largest n the one-kernel cluster schedule sorts (with_values as for rs_temp_bytes)."""
    return lib().rs_cluster_max_n(KEY_TYPES[key_type], _with_values(with_values))


def rs_skip_record(temp, stream=None):
    """(status, differing_bits, unordered) of the last sort that used temp."""
    bits, unordered = ctypes.c_uint64(0), _i(0)
    st = lib().rs_skip_record(_addr(temp), _stream(stream), ctypes.byref(bits), ctypes.byref(unordered))
    return st, bits.value, unordered.value


def rs_sort_host(key_type, h_keys_in, h_keys_out, h_vals_in, h_vals_out, n, begin_bit, end_bit,
                 d_work, work_bytes, stream=None) -> int:
    return lib().rs_sort_host(KEY_TYPES[key_type], _addr(h_keys_in), _addr(h_keys_out),
                              _addr(h_vals_in), _addr(h_vals_out), n, begin_bit, end_bit,
                              _addr(d_work), work_bytes, _stream(stream))


def rs_host_batches_work_bytes(key_type: str, with_values: bool, n: int, begin_bit: int,
                               end_bit: int) -> int:
    return lib().rs_host_batches_work_bytes(KEY_TYPES[key_type], int(bool(with_values)), n,
                                            begin_bit, end_bit)


def _ptr_array(bufs):
    """A C array of the buffers' addresses (None stays None)."""
    if bufs is None:
        return None
    return (ctypes.c_void_p * len(bufs))(*[_addr(b) for b in bufs])


def rs_sort_host_batches(key_type, h_keys_in, h_keys_out, h_vals_in, h_vals_out, n, begin_bit,
                         end_bit, d_work, work_bytes, stream=None) -> int:
    """h_keys_in / h_keys_out (and h_vals_* or None): equal-length lists of
    host buffers, one per batch."""
    batches = len(h_keys_in)
    if len(h_keys_out) != batches or (h_vals_in is not None and len(h_vals_in) != batches) or \
            (h_vals_out is not None and len(h_vals_out) != batches):
        raise ValueError("every buffer list needs one entry per batch")
    arrays = [_ptr_array(x) for x in (h_keys_in, h_keys_out, h_vals_in, h_vals_out)]  # alive until return
    ptrs = [None if a is None else ctypes.addressof(a) for a in arrays]
    return lib().rs_sort_host_batches(KEY_TYPES[key_type], batches, *ptrs, n, begin_bit, end_bit,
                                      _addr(d_work), work_bytes, _stream(stream))


class Graph:
    """A captured, instantiated CUDA graph of one whole sort (rs_graph_*)."""

    def __init__(self, desc: SortDesc):
        h = ctypes.c_void_p()
        _check(lib().rs_graph_create(ctypes.byref(desc), ctypes.byref(h)), "rs_graph_create")
        self._h = h

    def launch(self, stream=None):
        _check(lib().rs_graph_launch(self._h, _stream(stream)), "rs_graph_launch")

    def close(self):
        if self._h:
            lib().rs_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------- convenience

def key_type_of(t) -> str:
    import torch
    m = {torch.int32: "i32", torch.float32: "f32", torch.int16: "i16", torch.float16: "f16"}
    for name in ("uint32", "uint64", "uint16"):
        dt = getattr(torch, name, None)
        if dt is not None:
            m[dt] = "u" + name[4:]
    if t.dtype not in m:
        raise TypeError(f"pass key_type= for keys of dtype {t.dtype}")
    return m[t.dtype]


def sort(keys, values=None, *, key_type=None, begin_bit=0, end_bit=None, algo="auto",
         radix_bits=0, keys_out=None, values_out=None, temp=None, stream=None, descending=False):
    """Stable radix sort of a CUDA tensor of keys (and 32- or 64-bit values),
    ascending or descending (ties keep their input order either way).

    Returns (keys_out, values_out or None).  Allocates the outputs and temp
    with torch when they are not given; enqueues on `stream` (default: the
    current stream) and does not synchronise.
    """
    import torch
    kt = key_type or key_type_of(keys)
    if keys.element_size() != KEY_BYTES[kt] or not keys.is_contiguous() or not keys.is_cuda:
        raise ValueError("keys must be a contiguous CUDA tensor with elements of the key size")
    n = keys.numel()
    end_bit = KEY_BITS[kt] if end_bit is None else end_bit
    if keys_out is None:
        keys_out = torch.empty_like(keys)
    if values is not None and values_out is None:
        values_out = torch.empty_like(values)
    vb = 0 if values is None else values.element_size()
    if vb not in (0, 4, 8):
        raise ValueError("values must have 4- or 8-byte elements")
    tb = rs_temp_bytes(kt, vb if vb else False, n, begin_bit, end_bit)
    if tb == ctypes.c_size_t(-1).value:
        raise RadixSortError(1, "rs_temp_bytes")
    if temp is None:
        temp = torch.empty(max(tb, 1), dtype=torch.uint8, device=keys.device)
    desc = make_desc(kt, keys, keys_out, values, values_out, n, begin_bit, end_bit, temp,
                     temp.numel(), stream, algo, radix_bits, descending=descending, value_bytes=vb)
    _check(rs_sort(desc), "rs_sort")
    return keys_out, values_out
