"""CPU oracle for the stable LSD radix sort -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's ``cpu_baseline`` /
``--impl reference`` legs may import this package.  The CUDA library never
does, and the two share no code.  The arithmetic lives in ``oracle.c`` (plain,
single-threaded C, compiled on first use with the host C compiler); this file
only marshals numpy arrays.

Functions:
  sort(key_type, keys, values=None, begin_bit=0, end_bit=None, radix_bits=8, descending=False)
      LSD radix sort by counting-sort passes (key types u32 i32 f32 u64 u16 i16 f16) ("Radix sort を実装 & 測定してみた",
      section アルゴリズムの詳細; "Radix sort paralelo sobre el scan", section
      Las tres fases de una pasada).
  one_bit_split_sort(...)
      the one-bit index-formula sort of "Radix sort を実装 & 測定してみた",
      section アルゴリズムの詳細, as an independent second path.
  decimal_lsd_trace(keys, passes)
      the base-10 worked example of "Radix sort paralelo sobre el scan",
      section La idea y el requisito de estabilidad.
  ordered_keys(key_type, keys)
      the order-preserving unsigned map ("Radix sort を実装 & 測定してみた",
      section 符号付型、浮動小数点型に対する radix sort, for float32; "Radix sort
      paralelo sobre el scan", section Claves con signo y en coma flotante, for
      int32).
  exclusive_scan(values)
      the exclusive prefix sum ("高性能计算：GPU上的基数排序", section CPU上的扫描).
  stable_sort_baseline(key_type, keys, values=None, begin_bit=0, end_bit=None, descending=False)
      the same problem as one std::stable_sort (stable_sort_baseline.cpp): a CPU
      baseline for the bench and a cross-check for the tests.
  hardware_concurrency()
      std::thread::hardware_concurrency() of this host.
  lbvh_build(sorted_codes)
      the binary radix tree (linear BVH hierarchy) over sorted codes, built
      top-down from its definition (lbvh.c).
  parallel_lsd_sort(key_type, keys, values=None, begin_bit=0, end_bit=None, threads=None)
      a multi-threaded CPU LSD radix sort (parallel_baseline.c, OpenMP when
      the compiler has it): the all-cores CPU baseline of the bench.
  parallel_threads()
      how many threads that sort uses by default.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SRC_CPP = os.path.join(_HERE, "stable_sort_baseline.cpp")
_SRC_LBVH = os.path.join(_HERE, "lbvh.c")
_SRC_PAR = os.path.join(_HERE, "parallel_baseline.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

KEY_TYPES = {"u32": 0, "i32": 1, "f32": 2, "u64": 3, "u16": 4, "i16": 5, "f16": 6}
KEY_DTYPE = {"u32": np.uint32, "i32": np.uint32, "f32": np.uint32, "u64": np.uint64,
             "u16": np.uint16, "i16": np.uint16, "f16": np.uint16}
KEY_BITS = {"u32": 32, "i32": 32, "f32": 32, "u64": 64, "u16": 16, "i16": 16, "f16": 16}


def build(force: bool = False) -> str:
    """Compile oracle.c (host C compiler) and stable_sort_baseline.cpp (host C++
    compiler) into one shared library, -O2, no vectorisation flags."""
    with _lock:
        newest = max(os.path.getmtime(x) for x in (_SRC, _SRC_CPP, _SRC_LBVH, _SRC_PAR))
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
            os.makedirs(_LIBDIR, exist_ok=True)
            tag = f".{os.getpid()}"
            obj_c = os.path.join(_LIBDIR, "oracle.o" + tag)
            obj_cpp = os.path.join(_LIBDIR, "stable_sort_baseline.o" + tag)
            obj_lbvh = os.path.join(_LIBDIR, "lbvh.o" + tag)
            obj_par = os.path.join(_LIBDIR, "parallel_baseline.o" + tag)
            tmp = _LIB + tag + ".tmp"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-c", "-o", obj_c, _SRC])
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-c", "-o", obj_lbvh, _SRC_LBVH])
            subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-c", "-o", obj_cpp, _SRC_CPP])
            # OpenMP for the multi-threaded baseline when the compiler has it; one thread otherwise
            omp = ["-fopenmp"]
            r = subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", *omp, "-c", "-o", obj_par, _SRC_PAR],
                               capture_output=True)
            if r.returncode != 0:
                omp = []
                subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-c", "-o", obj_par, _SRC_PAR])
            r = subprocess.run(["g++", "-shared", *omp, "-o", tmp, obj_c, obj_lbvh, obj_par, obj_cpp],
                               capture_output=True)
            if r.returncode != 0 and omp:  # no OpenMP runtime to link: build the one-thread form
                subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-c", "-o", obj_par, _SRC_PAR])
                subprocess.check_call(["g++", "-shared", "-o", tmp, obj_c, obj_lbvh, obj_par, obj_cpp])
            elif r.returncode != 0:
                raise RuntimeError(r.stderr.decode(errors="replace"))
            os.replace(tmp, _LIB)
            for o in (obj_c, obj_lbvh, obj_par, obj_cpp):
                os.remove(o)
    return _LIB


def _bind(lib):
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.oracle_lsd_sort.argtypes = [i32, vp, vp, vp, vp, sz, i32, i32, i32]
    lib.oracle_lsd_sort.restype = i32
    lib.oracle_lsd_sort_dir.argtypes = [i32, vp, vp, vp, vp, sz, i32, i32, i32, i32]
    lib.oracle_lsd_sort_dir.restype = i32
    lib.oracle_one_bit_split_sort.argtypes = [i32, vp, vp, vp, vp, sz, i32, i32]
    lib.oracle_one_bit_split_sort.restype = i32
    lib.oracle_decimal_lsd_trace.argtypes = [vp, sz, i32, vp]
    lib.oracle_decimal_lsd_trace.restype = i32
    lib.oracle_ordered_keys.argtypes = [i32, vp, sz, vp]
    lib.oracle_ordered_keys.restype = None
    lib.oracle_exclusive_scan.argtypes = [vp, vp, sz]
    lib.oracle_exclusive_scan.restype = None
    if hasattr(lib, "cpu_stable_sort"):  # absent from the planted-mistake copies of oracle.c
        lib.cpu_stable_sort.argtypes = [i32, vp, vp, vp, vp, sz, i32, i32, i32]
        lib.cpu_stable_sort.restype = i32
        lib.cpu_hardware_concurrency.argtypes = []
        lib.cpu_hardware_concurrency.restype = ctypes.c_uint
        lib.oracle_lbvh_build.argtypes = [vp, sz, vp, vp, vp, vp, vp, vp]
        lib.oracle_lbvh_build.restype = i32
        lib.cpu_parallel_lsd_sort.argtypes = [i32, vp, vp, vp, vp, sz, i32, i32, i32]
        lib.cpu_parallel_lsd_sort.restype = i32
        lib.cpu_parallel_threads.argtypes = []
        lib.cpu_parallel_threads.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _as_keys(key_type: str, keys) -> np.ndarray:
    dt = KEY_DTYPE[key_type]
    a = np.ascontiguousarray(keys)
    if a.dtype.itemsize != np.dtype(dt).itemsize:
        raise TypeError(f"{key_type} keys need {np.dtype(dt).itemsize}-byte elements, got {a.dtype}")
    return a.view(dt)


def _vp(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def sort(key_type: str, keys, values=None, begin_bit: int = 0, end_bit: int | None = None,
         radix_bits: int = 8, lib=None, descending: bool = False):
    """Stable LSD radix sort, ascending or descending (ties in input order);
    returns (keys_out, values_out or None) as new arrays."""
    k = _as_keys(key_type, keys)
    end_bit = KEY_BITS[key_type] if end_bit is None else end_bit
    n = k.size
    ko = np.empty_like(k)
    vi = None if values is None else np.ascontiguousarray(values, dtype=np.uint32)
    vo = None if vi is None else np.empty_like(vi)
    if vi is not None and vi.size != n:
        raise ValueError("values must match keys in length")
    rc = (lib or _load()).oracle_lsd_sort_dir(KEY_TYPES[key_type], _vp(k), _vp(ko), _vp(vi), _vp(vo), n,
                                              begin_bit, end_bit, radix_bits, int(bool(descending)))
    if rc != 0:
        raise ValueError(f"oracle_lsd_sort failed with code {rc}")
    return ko, vo


def one_bit_split_sort(key_type: str, keys, values=None, begin_bit: int = 0,
                       end_bit: int | None = None, lib=None):
    """The one-bit index-formula sort, one pass per bit of [begin_bit, end_bit)."""
    k = _as_keys(key_type, keys)
    end_bit = KEY_BITS[key_type] if end_bit is None else end_bit
    n = k.size
    ko = np.empty_like(k)
    vi = None if values is None else np.ascontiguousarray(values, dtype=np.uint32)
    vo = None if vi is None else np.empty_like(vi)
    rc = (lib or _load()).oracle_one_bit_split_sort(KEY_TYPES[key_type], _vp(k), _vp(ko), _vp(vi), _vp(vo),
                                           n, begin_bit, end_bit)
    if rc != 0:
        raise ValueError(f"oracle_one_bit_split_sort failed with code {rc}")
    return ko, vo


def decimal_lsd_trace(keys, passes: int, lib=None) -> np.ndarray:
    """Array after each base-10 LSD pass, shape (passes, n)."""
    k = np.ascontiguousarray(keys, dtype=np.uint64)
    out = np.empty((passes, k.size), dtype=np.uint64)
    rc = (lib or _load()).oracle_decimal_lsd_trace(_vp(k), k.size, passes, _vp(out))
    if rc != 0:
        raise ValueError(f"oracle_decimal_lsd_trace failed with code {rc}")
    return out


def ordered_keys(key_type: str, keys, lib=None) -> np.ndarray:
    """The order-preserving unsigned key of every element (uint64 array)."""
    k = _as_keys(key_type, keys)
    out = np.empty(k.size, dtype=np.uint64)
    (lib or _load()).oracle_ordered_keys(KEY_TYPES[key_type], _vp(k), k.size, _vp(out))
    return out


def exclusive_scan(values, lib=None) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.uint64)
    out = np.empty_like(v)
    (lib or _load()).oracle_exclusive_scan(_vp(v), _vp(out), v.size)
    return out


def stable_sort_baseline(key_type: str, keys, values=None, begin_bit: int = 0, end_bit: int | None = None,
                         descending: bool = False):
    """The same sort as one single-threaded std::stable_sort; returns (keys_out, values_out or None)."""
    k = _as_keys(key_type, keys)
    end_bit = KEY_BITS[key_type] if end_bit is None else end_bit
    n = k.size
    ko = np.empty_like(k)
    vi = None if values is None else np.ascontiguousarray(values, dtype=np.uint32)
    vo = None if vi is None else np.empty_like(vi)
    if vi is not None and vi.size != n:
        raise ValueError("values must match keys in length")
    rc = _load().cpu_stable_sort(KEY_TYPES[key_type], _vp(k), _vp(ko), _vp(vi), _vp(vo), n, begin_bit, end_bit,
                                 int(bool(descending)))
    if rc != 0:
        raise ValueError(f"cpu_stable_sort failed with code {rc}")
    return ko, vo


def parallel_threads() -> int:
    """Threads the multi-threaded baseline uses by default (1 without OpenMP)."""
    return int(_load().cpu_parallel_threads())


def parallel_lsd_sort(key_type: str, keys, values=None, begin_bit: int = 0, end_bit: int | None = None,
                      threads: int | None = None):
    """The same sort, ascending, on `threads` host threads (default: all);
    returns (keys_out, values_out or None)."""
    k = _as_keys(key_type, keys)
    end_bit = KEY_BITS[key_type] if end_bit is None else end_bit
    n = k.size
    ko = np.empty_like(k)
    vi = None if values is None else np.ascontiguousarray(values, dtype=np.uint32)
    vo = None if vi is None else np.empty_like(vi)
    if vi is not None and vi.size != n:
        raise ValueError("values must match keys in length")
    t = parallel_threads() if threads is None else threads
    rc = _load().cpu_parallel_lsd_sort(KEY_TYPES[key_type], _vp(k), _vp(ko), _vp(vi), _vp(vo), n, begin_bit,
                                       end_bit, t)
    if rc != 0:
        raise ValueError(f"cpu_parallel_lsd_sort failed with code {rc}")
    return ko, vo


def hardware_concurrency() -> int:
    """std::thread::hardware_concurrency() of this host."""
    return int(_load().cpu_hardware_concurrency())


LBVH_LEAF = 0x80000000
LBVH_NONE = 0xFFFFFFFF


def lbvh_build(sorted_codes) -> dict:
    """The binary radix tree over sorted uint32 codes: a dict of uint32 arrays
    left, right, first, last, node_parent (n-1 each) and leaf_parent (n);
    a child with bit 31 set (LBVH_LEAF) is a leaf."""
    c = np.ascontiguousarray(sorted_codes, dtype=np.uint32)
    n = c.size
    m = max(n - 1, 0)
    out = {k: np.empty(m, dtype=np.uint32) for k in ("left", "right", "first", "last", "node_parent")}
    out["leaf_parent"] = np.empty(n, dtype=np.uint32)
    rc = _load().oracle_lbvh_build(_vp(c), n, *(_vp(out[k]) for k in
                                                ("left", "right", "first", "last", "leaf_parent", "node_parent")))
    if rc != 0:
        raise ValueError(f"oracle_lbvh_build failed with code {rc}")
    return out


def load_variant(path: str):
    """Bind a separately compiled copy of oracle.c (the tests plant mistakes in copies)."""
    return _bind(ctypes.CDLL(path))
