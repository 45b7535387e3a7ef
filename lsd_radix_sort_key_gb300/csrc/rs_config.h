// rs_config.h -- compile-time shapes shared by the host planner and the kernels.
//
// Everything here is plain constexpr arithmetic so that rs_temp_bytes() can
// size the scratch buffer on a machine without a GPU, and the kernels agree
// with it by construction.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace rs {

// Largest number of digit passes any request can need (64-bit keys, 4-bit digits).
constexpr int kMaxPasses = 16;

// The "meta" block at the start of temp: the device error word; the pass-skip
// record written by the first read of the keys (words kSkipBase..+3: the OR
// over all keys of ordered(key) ^ ordered(keys[0]) as two 32-bit halves, a
// flag set when some adjacent pair is out of order, and a count of the CTAs
// that have added their share); one tile ticket per pass (chained scan); the
// pass plan the last of those CTAs derives from the record (one word per
// pass: runs | index among running passes << 8 | running passes << 16); and
// one 256-bin global histogram per pass.
constexpr int kErrWord = 0;
constexpr int kSkipBase = 4;
constexpr int kTicketBase = 16;
constexpr int kPlanBase = 32;
constexpr int kGhistBase = 64;
constexpr int kMetaWords = kGhistBase + kMaxPasses * 256;

// Reduce-then-scan: at most this many CTAs, each owning a contiguous chunk.
constexpr int kRtsMaxCtas = 4096;

// Tile shapes.  A tile is THREADS x ITEMS keys; ITEMS is chosen per (key
// bytes, has values) so that keys, packed ranks and values stay in registers
// at 1024 resident threads per SM (64 registers each).  The chained-scan pass
// uses larger tiles than the reduce-then-scan downsweep: fewer tiles mean a
// shorter look-back and less status traffic; the downsweep uses 512 threads
// when values ride along or keys are 64-bit (longer digit runs per tile).
// (All measured on 2^28 keys.)
#ifndef RS_RTS_THREADS
#define RS_RTS_THREADS 256
#endif
#ifndef RS_RTS_THREADS_PAIRS
#define RS_RTS_THREADS_PAIRS 512
#endif
#ifndef RS_RTS_THREADS_U64
#define RS_RTS_THREADS_U64 512
#endif
#ifndef RS_OS_THREADS
#define RS_OS_THREADS 512
#endif
// Small chained-scan sorts (8-bit digits, under kOsSmallTileMaxBytes of keys
// and values) run 256-thread tiles instead: twice as many tiles keep more SMs
// busy.  Graph replays on GB300, ms per sort, 256 vs 512 threads: uint32 keys
// 2^17 / 2^18 / 2^19 0.0350 / 0.0370 / 0.0411 vs 0.0411 / 0.0430 / 0.0452,
// 2^20 0.0491 either way; uint32 pairs 2^18 0.0391 vs 0.0451, 2^19 0.0470 vs
// 0.0472; uint64 keys 2^18 0.0677 vs 0.0779; uint16 keys 2^18 0.0226 vs
// 0.0248; uint64 keys + uint32 values 2^19 0.0902 vs 0.0863.
#ifndef RS_OS_THREADS_SMALL
#define RS_OS_THREADS_SMALL 256
#endif
#ifndef RS_ITEMS_U32_KEYS
#define RS_ITEMS_U32_KEYS 16
#endif
enum : int { kAlgoOnesweep = 1, kAlgoReduceScan = 2 };
// vb = bytes of the value that rides along each key: 0 (keys only), 4 or 8.
constexpr int tile_threads(int algo, int key_bytes, int vb)
{
    return algo == kAlgoOnesweep ? RS_OS_THREADS
           : key_bytes == 8      ? RS_RTS_THREADS_U64
           : vb != 0             ? RS_RTS_THREADS_PAIRS
                                 : RS_RTS_THREADS;
}
#ifndef RS_ITEMS_U32_PAIRS
#define RS_ITEMS_U32_PAIRS 12
#endif
constexpr int tile_items(int key_bytes, int vb)
{
    // 16-bit keys live in 32-bit registers: the 32-bit shapes.  64-bit values
    // take two registers each, so fewer keys per thread.
    return key_bytes <= 4 ? (vb == 0 ? RS_ITEMS_U32_KEYS : vb == 4 ? RS_ITEMS_U32_PAIRS : 8)
                          : (vb == 0 ? 12 : vb == 4 ? 9 : 6);
}
constexpr int tile_keys(int algo, int key_bytes, int vb)
{
    return tile_threads(algo, key_bytes, vb) * tile_items(key_bytes, vb);
}
constexpr size_t kOsSmallTileMaxBytes = (size_t)4 << 20;  // exclusive
// The chained scan's threads per tile for n keys of key_bytes with vb-byte
// values (16-bit keys count as 32-bit: they occupy a 32-bit register each).
constexpr int onesweep_threads(size_t n, int key_bytes, int vb, int radix_bits)
{
    const size_t bytes = n * (size_t)((key_bytes < 4 ? 4 : key_bytes) + vb);
    return (radix_bits == 8 && bytes < kOsSmallTileMaxBytes) ? RS_OS_THREADS_SMALL : RS_OS_THREADS;
}

// Small sorts: one kernel on a cluster of at most kClusterMaxCtas CTAs, each
// holding one tile of kClusterThreads x cluster_items keys in shared memory.
// 16 CTAs of 512 x 8 measured fastest on GB300 for 2^12..2^16 uint32 keys
// (8 CTAs of 512 x 16: 1.3x slower; 16 of 1024 x 4 or 256 x 16: 1.07x).
// 16 is above the portable cluster size: the launch opts in, and a device
// that cannot schedule it falls back to the chained scan (AUTO).
#ifndef RS_CL_MAX_CTAS
#define RS_CL_MAX_CTAS 16
#endif
#ifndef RS_CL_THREADS
#define RS_CL_THREADS 512
#endif
#ifndef RS_CL_ITEMS
#define RS_CL_ITEMS 8
#endif
constexpr int kClusterMaxCtas = RS_CL_MAX_CTAS;
constexpr int kClusterThreads = RS_CL_THREADS;
constexpr int cluster_items(int key_bytes, int vb)
{
    // uint32 keys RS_CL_ITEMS per thread; 3/4 of that with 32-bit values or
    // for uint64 keys, less again with wider payloads (registers and shared
    // memory scale with the bytes per key)
    return key_bytes <= 4 ? (vb == 0 ? RS_CL_ITEMS : vb == 4 ? RS_CL_ITEMS * 3 / 4 : RS_CL_ITEMS / 2)
                          : (vb == 0 ? RS_CL_ITEMS * 3 / 4 : vb == 4 ? RS_CL_ITEMS * 9 / 16 : RS_CL_ITEMS * 3 / 8);
}
constexpr size_t cluster_tile_keys(int key_bytes, int vb)
{
    return (size_t)kClusterThreads * cluster_items(key_bytes, vb);
}
constexpr size_t cluster_max_n(int key_bytes, int vb)
{
    return (size_t)kClusterMaxCtas * cluster_tile_keys(key_bytes, vb);
}

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int passes_for(int begin_bit, int end_bit, int radix_bits)
{
    return end_bit > begin_bit ? (end_bit - begin_bit + radix_bits - 1) / radix_bits : 0;
}

// Byte offsets of the regions of temp.  Every region starts on a 256-byte
// boundary; the meta block (and so the device error word) is always first.
struct TempLayout {
    size_t meta;       // kMetaWords uint32
    size_t alt_keys;   // n keys: the ping-pong partner of keys_out
    size_t alt_vals;   // n values (pairs only; 4 or 8 bytes each)
    size_t big;        // chained-scan tile status, or reduce-then-scan block counts
    size_t big_bytes;
    size_t total;
};

constexpr size_t status_bytes(size_t n, int key_bytes, int vb, int begin_bit, int end_bit,
                              int radix_bits)
{
    const size_t tk = (size_t)onesweep_threads(n, key_bytes, vb, radix_bits) * (size_t)tile_items(key_bytes, vb);
    size_t tiles = (n + tk - 1) / tk;
    return (size_t)passes_for(begin_bit, end_bit, radix_bits) * tiles * ((size_t)1 << radix_bits) * 4;
}

constexpr TempLayout temp_layout(int key_bytes, int vb, size_t n, int begin_bit, int end_bit)
{
    TempLayout t{};
    size_t off = 0;
    t.meta = off;
    off += align_up(kMetaWords * 4, 256);
    t.alt_keys = off;
    off += align_up(n * (size_t)key_bytes, 256);
    t.alt_vals = off;
    off += vb ? align_up(n * (size_t)vb, 256) : 0;
    t.big = off;
    size_t s8 = status_bytes(n, key_bytes, vb, begin_bit, end_bit, 8);
    size_t s4 = status_bytes(n, key_bytes, vb, begin_bit, end_bit, 4);
    size_t rts = (size_t)256 * kRtsMaxCtas * 4;
    size_t big = s8 > s4 ? s8 : s4;
    big = big > rts ? big : rts;
    t.big_bytes = align_up(big, 256);
    off += t.big_bytes;
    t.total = off;
    return t;
}

}  // namespace rs
