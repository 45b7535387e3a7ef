"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no sorting arithmetic: it only draws keys and payloads
(SplitMix64, Steele, Lea & Flood 2014, used as a counter-based generator) so
that the CUDA library and the CPU oracle consume identical bytes.  The draws
run in ``synth.c``, compiled on first use with the host C compiler.

Workloads (``WORKLOADS``) mirror the sort's published use: uniform 32-bit keys,
N(0,1) floats with injected signed zeros / infinities / NaNs, uniform signed
ints with an index payload, 30-bit Morton codes of uniform 3-D points, a
low-entropy AND-of-four-words distribution and uniform 64-bit keys.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library (host C compiler, -O2)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            os.makedirs(_LIBDIR, exist_ok=True)
            tmp = _LIB + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, sz, u64, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64, ctypes.c_int
        for name in ("synth_u32_uniform", "synth_u64_uniform", "synth_u32_and4",
                     "synth_u32_morton30", "synth_splitmix64", "synth_f32_edge"):
            getattr(lib, name).argtypes = [vp, sz, u64]
            getattr(lib, name).restype = None
        lib.synth_u32_bits.argtypes = [vp, sz, u64, i32]
        lib.synth_u32_bits.restype = None
        lib.synth_iota_u32.argtypes = [vp, sz]
        lib.synth_iota_u32.restype = None
        lib.synth_f32_normal_specials.argtypes = [vp, sz, u64, sz, vp]
        lib.synth_f32_normal_specials.restype = i32
        _lib = lib
    return _lib


def _ptr(a) -> int:
    """Address of a C-contiguous numpy array or a CPU torch tensor."""
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    assert a.is_contiguous() and a.device.type == "cpu"
    return a.data_ptr()


def _out(out, n, dtype):
    if out is None:
        return np.empty(n, dtype=dtype)
    size = out.size if isinstance(out, np.ndarray) else out.numel()
    if size < n or out.dtype.itemsize != np.dtype(dtype).itemsize:
        raise ValueError("output buffer too small or of the wrong element size")
    return out


def splitmix64(n: int, seed: int, out=None):
    out = _out(out, n, np.uint64)
    _load().synth_splitmix64(_ptr(out), n, seed)
    return out


def u32_uniform(n: int, seed: int, out=None):
    out = _out(out, n, np.uint32)
    _load().synth_u32_uniform(_ptr(out), n, seed)
    return out


def u64_uniform(n: int, seed: int, out=None):
    out = _out(out, n, np.uint64)
    _load().synth_u64_uniform(_ptr(out), n, seed)
    return out


def u32_and4(n: int, seed: int, out=None):
    out = _out(out, n, np.uint32)
    _load().synth_u32_and4(_ptr(out), n, seed)
    return out


def u32_bits(n: int, seed: int, bits: int, out=None):
    out = _out(out, n, np.uint32)
    _load().synth_u32_bits(_ptr(out), n, seed, bits)
    return out


def u32_morton30(n: int, seed: int, out=None):
    out = _out(out, n, np.uint32)
    _load().synth_u32_morton30(_ptr(out), n, seed)
    return out


def iota_u32(n: int, out=None):
    out = _out(out, n, np.uint32)
    _load().synth_iota_u32(_ptr(out), n)
    return out


def f32_normal_specials(n: int, seed: int, per_special: int | None = None, out=None):
    """Bit patterns (uint32) of N(0,1) floats with signed zeros, infinities and NaN injected."""
    if per_special is None:
        per_special = int(0.001 * n)
    out = _out(out, n, np.uint32)
    scratch = np.empty(max(n, 1), dtype=np.uint32)
    rc = _load().synth_f32_normal_specials(_ptr(out), n, seed, per_special, scratch.ctypes.data)
    if rc != 0:
        raise ValueError("too many specials for n")
    return out


def f32_edge(n: int, seed: int, out=None):
    """Bit patterns (uint32) mixing boundary floats, NaN payloads and random bits."""
    out = _out(out, n, np.uint32)
    _load().synth_f32_edge(_ptr(out), n, seed)
    return out


def u16_uniform(n: int, seed: int, out=None):
    """16-bit keys: the low halves of the uint32 stream of the same seed."""
    out = _out(out, n, np.uint16)
    out[:n] = (u32_uniform(n, seed) & np.uint32(0xFFFF)).astype(np.uint16)
    return out


# binary16 boundary patterns: zeros, subnormals, the smallest normal, +-1,
# the largest finite, infinities and NaN payloads of both signs.
F16_BOUNDARY = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x83FF, 0x0400, 0x8400, 0x3C00,
                         0xBC00, 0x3C01, 0xBC01, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00, 0xFE00,
                         0x7C01, 0xFC01, 0x7FFF, 0xFFFF, 0x4248, 0xC248], dtype=np.uint16)


def f16_edge(n: int, seed: int, out=None):
    """binary16 bit patterns: every third key a boundary pattern, the rest
    random bits (any class: normal, subnormal, zero, Inf, NaN)."""
    out = _out(out, n, np.uint16)
    rnd = (u32_uniform(n, seed) & np.uint32(0xFFFF)).astype(np.uint16)
    pick = u32_uniform(n, seed ^ 0x16) % np.uint32(3 * len(F16_BOUNDARY))
    out[:n] = np.where(pick < len(F16_BOUNDARY), F16_BOUNDARY[np.minimum(pick, len(F16_BOUNDARY) - 1)], rnd)
    return out


def f16_normal_specials(n: int, seed: int, out=None):
    """binary16 bit patterns of N(0,1) values (the float32 generator's values
    rounded to half precision, its injected -0.0, +0.0, +-Inf and NaN kept)."""
    out = _out(out, n, np.uint16)
    f = f32_normal_specials(n, seed).view(np.float32)
    out[:n] = f.astype(np.float16).view(np.uint16)
    return out


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    name: str          # short id used by tests and the bench
    key_type: str      # "u32" | "i32" | "f32" | "u64"
    log2n: int
    with_values: bool  # payload = original index
    begin_bit: int
    end_bit: int
    seed: int
    generator: str     # "uniform32" | "normal_specials32" | "morton30" | "and4" | "uniform64"
    description: str

    @property
    def n(self) -> int:
        return 1 << self.log2n

    def keys(self, n: int | None = None, out=None):
        """Key bit patterns (uint32 or uint64 array); n overrides the size (prefix-stable)."""
        n = self.n if n is None else n
        gen = {"uniform32": lambda: u32_uniform(n, self.seed, out),
               "normal_specials32": lambda: f32_normal_specials(n, self.seed, out=out),
               "morton30": lambda: u32_morton30(n, self.seed, out),
               "and4": lambda: u32_and4(n, self.seed, out),
               "uniform64": lambda: u64_uniform(n, self.seed, out)}
        if self.generator not in gen:
            raise KeyError(self.generator)
        return gen[self.generator]()

    def values(self, n: int | None = None, out=None):
        n = self.n if n is None else n
        return iota_u32(n, out) if self.with_values else None


WORKLOADS = {
    w.name: w
    for w in [
        Workload("u32_uniform_2p16", "u32", 16, False, 0, 32, 0x5EED0001, "uniform32",
                 "2^16 uint32 keys uniform over 32 bits, keys-only, bits [0,32)"),
        Workload("f32_normal_specials_2p24", "f32", 24, False, 0, 32, 0x5EED0002, "normal_specials32",
                 "2^24 float32 N(0,1) keys with 0.1% each of -0.0, +0.0, +Inf, -Inf, qNaN; keys-only"),
        Workload("i32_uniform_index_2p26", "i32", 26, True, 0, 32, 0x5EED0003, "uniform32",
                 "2^26 int32 keys uniform over the signed range, payload = index"),
        Workload("u32_uniform_2p28", "u32", 28, False, 0, 32, 0x5EED0004, "uniform32",
                 "2^28 uint32 keys uniform over 32 bits, keys-only"),
        Workload("morton30_index_2p28", "u32", 28, True, 0, 30, 0x1_5EED0004, "morton30",
                 "2^28 30-bit Morton codes of uniform 3-D points, payload = index, bits [0,30)"),
        Workload("u32_and4_2p28", "u32", 28, False, 0, 32, 0x2_5EED0004, "and4",
                 "2^28 uint32 keys, each the AND of 4 uniform words (P(bit)=1/16), keys-only"),
        Workload("u64_uniform_index_2p28", "u64", 28, True, 0, 64, 0x5EED0005, "uniform64",
                 "2^28 uint64 keys uniform over 64 bits, payload = index, bits [0,64)"),
    ]
}


def sweep_workload(log2n: int) -> Workload:
    """Uniform uint32 keys-only at 2^log2n (the roofline-knee size sweep, 2^16..2^29)."""
    return Workload(f"sweep_u32_2p{log2n}", "u32", log2n, False, 0, 32,
                    0x5EED0005 + (log2n << 32), "uniform32", f"2^{log2n} uint32 keys uniform, keys-only")
