// rs_kernels.cuh -- device code of the GB300 LSD radix sort and its per-key-type
// host driver.  Included once per key type (rs_sort_<type>.cu), which
// instantiates run_sort<KT>.
//
// One digit pass ("Radix sort paralelo sobre el scan", section "Las tres fases
// de una pasada") is:
//   1. a digit histogram per block of keys,
//   2. an exclusive scan of those counts in digit-major order, so that entry
//      (d, b) is where block b starts writing digit d ("高性能计算：GPU上的基数
//      排序", section "GPU上的基数排序": position = P_d[n] + m),
//   3. a stable rank of every key among equal digits inside its tile,
//   4. a shuffle of the tile in shared memory so that each digit is one run,
//      and a scatter of the runs to global memory ("정렬: 라딕스와 머지소트",
//      13.4: coalescing through shared memory).
//
// Three schedules are built from the same tile code:
//   * chained scan (k_histogram once, then k_onesweep per pass): every tile
//     takes a ticket, publishes its digit counts, and looks back over its
//     predecessors' published counts for its global offsets (decoupled
//     look-back; Merrill & Garland 2016, Adinets & Merrill 2022).  Step 2 thus
//     runs inside the pass kernel and the keys are read once per pass, plus
//     once up front for all histograms.
//   * reduce-then-scan (k_upsweep, k_spine_scan, k_downsweep per pass): each
//     CTA owns a contiguous chunk of tiles; the spine scan is step 2 proper.
//     Full tiles of keys-only 32/16-bit sorts reach shared memory by 1-D bulk
//     copies (cp.async.bulk) one tile ahead.
//   * small sorts (k_cluster_sort): the whole sort in one launch on a
//     thread-block cluster whose CTAs keep their tiles in shared memory and
//     exchange counts and keys through distributed shared memory.
//
// Keys may be 32-, 64- or 16-bit, values absent, 32- or 64-bit (VB = value
// bytes), and the order ascending or descending (each digit XORed with its
// mask).
//
// The kernels of one sort are chained by programmatic dependent launch: every
// kernel after the first waits on the device (griddepcontrol.wait) for the
// one before it, so their launches overlap the previous kernel's drain.
//
// Pass skipping: the first read of the keys (k_histogram, or the first
// k_upsweep) also records which key bits differ between keys and whether the
// input is already in order, and its last CTA turns that into a plan of
// which passes run.  Every later kernel reads the plan: a pass whose digit is
// the same for every key, or every pass of an input already in order, returns
// at once, and the running passes take their buffers from the plan so that
// the result still lands in keys_out (section "pass skipping" below).
//
// Keys are carried with their original bit patterns.  The order-preserving
// map T (identity, sign flip for int32/int16, the NaN/Inf-aware flip for
// float32 and binary16) is applied when a digit is extracted, in every pass
// -- as the CPU code of "Radix sort を実装 & 測定してみた" (section 実装)
// does -- so no inverse map is needed and NaN/Inf payloads come back
// unchanged.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "rs.h"
#include "rs_config.h"

// RS_CHECKED 1 also records (in the device error word) any shuffle position
// that had to be clamped; the clamp itself and the scatter bounds check are
// always on.
#ifndef RS_CHECKED
#define RS_CHECKED 0
#endif

// Compile-time choices measured against each other (defaults = the faster):
//   RS_MATCH_BITS   how many high bits of a digit are compared with
//                   __match_any_sync; the remaining low bits are compared with
//                   one __ballot_sync each.  (match cost grows with the number
//                   of distinct values in a warp, ballot cost with the bits.)
//   RS_LOOKBACK_BATCH  predecessor statuses read at once while walking back.
//   RS_TILE_MIN_THREADS_PER_SM  resident threads per SM the tile kernels are
//                   compiled for (caps their registers: 1024 -> 64 each).
#ifndef RS_MATCH_BITS
#define RS_MATCH_BITS 3
#endif
#ifndef RS_LOOKBACK_BATCH
#define RS_LOOKBACK_BATCH 4
#endif
#ifndef RS_TILE_MIN_THREADS_PER_SM
#define RS_TILE_MIN_THREADS_PER_SM 1024
#endif
//   RS_TMA_TILES    1: the reduce-then-scan downsweep of keys-only 32- and
//                   16-bit sorts with 8-bit digits stages each full tile in
//                   shared memory with a 1-D bulk copy (cp.async.bulk,
//                   completion on an mbarrier) issued one tile ahead; 0: it
//                   prefetches the next tile into registers with plain loads.
//                   (2^28 keys: -0.4% for uint32, -3.2% for uint16; with
//                   4-bit digits it measured 2.5% slower, so those keep the
//                   register prefetch.)
#ifndef RS_TMA_TILES
#define RS_TMA_TILES 1
#endif

namespace rs {

enum : int { KU32 = 0, KI32 = 1, KF32 = 2, KU64 = 3, KU16 = 4, KI16 = 5, KF16 = 6 };
// The same 32- and 16-bit key types, for passes whose digit is one whole byte
// of the ordered key: the digit is then one byte permute instead of a shift
// and a mask.
enum : int { KU32B = 7, KI32B = 8, KF32B = 9, KU16B = 10, KI16B = 11, KF16B = 12 };

// ------------------------------------------------------------------ key maps

template <int KT> struct KeyOps;

template <> struct KeyOps<KU32> {
    using T = uint32_t;
    static __device__ __forceinline__ uint32_t ordered(uint32_t u) { return u; }
};

// "Radix sort paralelo sobre el scan", section "Claves con signo y en coma
// flotante": two's-complement ints order as unsigned once the sign bit flips.
template <> struct KeyOps<KI32> {
    using T = uint32_t;
    static __device__ __forceinline__ uint32_t ordered(uint32_t u) { return u ^ 0x80000000u; }
};

// "Radix sort を実装 & 測定してみた", section "符号付型、浮動小数点型に対する
// radix sort": NaN/+-Inf become the maximum; a set sign bit flips all bits; a
// clear one sets the MSB.  Branch-free: the arithmetic shift gives an all-ones
// mask for negatives.
template <> struct KeyOps<KF32> {
    using T = uint32_t;
    static __device__ __forceinline__ uint32_t ordered(uint32_t u)
    {
        uint32_t flip = (uint32_t)((int32_t)u >> 31) | 0x80000000u;
        uint32_t o = u ^ flip;
        return ((u & 0x7F800000u) == 0x7F800000u) ? 0xFFFFFFFFu : o;
    }
};

template <> struct KeyOps<KU64> {
    using T = uint64_t;
    static __device__ __forceinline__ uint64_t ordered(uint64_t u) { return u; }
};

// 16-bit keys sort "by the same procedure" ("Radix sort を実装 & 測定してみた",
// section 符号付型、浮動小数点型に対する radix sort): int16 flips its sign bit,
// binary16 takes the float rule at 16 bits (exponent field all ones -> the
// maximum; negative -> all bits flipped; positive -> MSB set).
template <> struct KeyOps<KU16> {
    using T = uint16_t;
    static __device__ __forceinline__ uint32_t ordered(uint16_t u) { return u; }
};
template <> struct KeyOps<KI16> {
    using T = uint16_t;
    static __device__ __forceinline__ uint32_t ordered(uint16_t u) { return (uint32_t)u ^ 0x8000u; }
};
template <> struct KeyOps<KF16> {
    using T = uint16_t;
    static __device__ __forceinline__ uint32_t ordered(uint16_t h)
    {
        const uint32_t u = h;
        const uint32_t flip = ((u & 0x8000u) ? 0xFFFFu : 0x8000u);
        return ((u & 0x7C00u) == 0x7C00u) ? 0xFFFFu : (u ^ flip);
    }
};

template <> struct KeyOps<KU32B> : KeyOps<KU32> { static constexpr bool kByte = true; };
template <> struct KeyOps<KI32B> : KeyOps<KI32> { static constexpr bool kByte = true; };
template <> struct KeyOps<KF32B> : KeyOps<KF32> { static constexpr bool kByte = true; };
template <> struct KeyOps<KU16B> : KeyOps<KU16> { static constexpr bool kByte = true; };
template <> struct KeyOps<KI16B> : KeyOps<KI16> { static constexpr bool kByte = true; };
template <> struct KeyOps<KF16B> : KeyOps<KF16> { static constexpr bool kByte = true; };

template <int KT, typename = void> struct IsByte { static constexpr bool value = false; };
template <int KT> struct IsByte<KT, decltype((void)KeyOps<KT>::kByte)> { static constexpr bool value = true; };

// The payload type by its byte count: 4 (uint32) or 8 (uint64); 0 = keys only.
template <int VB> struct ValType { using type = uint32_t; };
template <> struct ValType<8> { using type = uint64_t; };
template <int VB> using ValT = typename ValType<VB>::type;

// The digit of key u for a pass at `shift` of width mask; `flip` (mask for a
// descending sort, else 0) reverses the digit order.  The byte twins serve
// ascending sorts only.
template <int KT>
__device__ __forceinline__ uint32_t digit_of(typename KeyOps<KT>::T u, uint32_t shift, uint32_t mask,
                                             uint32_t flip)
{
    if constexpr (IsByte<KT>::value)  // byte (shift / 8) moved to the low byte, zeros above
        return __byte_perm((uint32_t)KeyOps<KT>::ordered(u), 0u, 0x4440u | (shift >> 3));
    else
        return ((uint32_t)(KeyOps<KT>::ordered(u) >> shift) & mask) ^ flip;
}

// ------------------------------------------------------------- small helpers

// Look-back status word: 2-bit flag | 30-bit count.
constexpr uint32_t kFlagAgg = 1u << 30;   // this tile's own digit count
constexpr uint32_t kFlagInc = 2u << 30;   // count of this tile and every earlier one
constexpr uint32_t kValMask = (1u << 30) - 1;

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A 64-bit L2 cache policy that marks lines evict-last.
__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <typename T>
__device__ __forceinline__ void st_keep(T* addr, T v, uint64_t pol)
{
    if constexpr (sizeof(T) == 8)
        asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(addr), "l"(v), "l"(pol) : "memory");
    else if constexpr (sizeof(T) == 4)
        asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(addr), "r"(v), "l"(pol) : "memory");
    else
        asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(addr), "h"(v), "l"(pol) : "memory");
}

// ---- 1-D bulk copies into shared memory, completed on an mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory
// before later async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// One thread: expect `bytes` on bar and copy them from global src to shared
// dst (both 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Waits for phase `parity` of bar to complete, at most `limit` polls (each
// poll may suspend the thread briefly); returns false if it ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// The device error word is a bit set of rs_status codes (bit = 1 << code),
// so a root cause (a timed-out wait) is never hidden by its consequences.
__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code) { atomicOr(err, 1u << code); }

// Programmatic dependent launch: every kernel of a sort after its first is
// launched as a dependent of the kernel before it in the stream, so its CTAs
// are set up as that kernel's last CTAs exit instead of after a full launch
// round trip.  wait_prior_grid() blocks until the kernel before has completed
// and its writes are visible (every earlier kernel completed before that one
// passed its own wait); it returns at once after a plain launch.  A kernel
// touches no global memory before its wait.  (The kernels do not signal
// their dependents early: measured on GB300, letting the next kernel's CTAs
// in while a kernel still runs was slower in graph replays.)
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Exclusive scan of one value per digit over the first BINS threads of the
// block (others pass 0).  Every thread must call it: it holds one barrier, and
// a second one unless TRAILING_SYNC is false.  `scratch` needs (BINS + 31) / 32
// words.  *total (if given) receives the sum.
template <int BINS, bool TRAILING_SYNC = true>
__device__ __forceinline__ uint32_t bins_exclusive_scan(uint32_t v, uint32_t* scratch, uint32_t* total)
{
    constexpr int SCAN_WARPS = (BINS + 31) / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t x = v;
    if (warp < SCAN_WARPS) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) scratch[warp] = x;
    }
    __syncthreads();
    uint32_t wp = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < SCAN_WARPS; ++w) {
        uint32_t s = scratch[w];
        wp += (w < warp) ? s : 0u;
        tot += s;
    }
    if (total) *total = tot;
    // Without the trailing barrier the caller must not reuse `scratch` before
    // another block-wide barrier.
    if (TRAILING_SYNC) __syncthreads();
    return (warp < SCAN_WARPS) ? x - v + wp : 0u;
}

// ------------------------------------------------------------ pass parameters

struct PassParams {
    // This pass's source and destination when every pass runs (the host's
    // plan); when the skip record drops a pass, the kernels work out the
    // actual ones from the sort-level buffers below (pass_buffers).
    const void* keys_in;
    void* keys_out;
    const void* vals_in;
    void* vals_out;
    const void* sort_keys_in;   // the sort's input and output
    void* sort_keys_out;
    const void* sort_vals_in;
    void* sort_vals_out;
    void* alt_keys;          // the ping-pong partner buffers in temp
    void* alt_vals;
    uint32_t* skip;          // the skip record in temp (see kSkipBase)
    uint32_t* plan;          // the pass plan in temp (see kPlanBase)
    uint32_t pass;           // this pass's index and the geometry of all passes
    uint32_t passes;
    uint32_t begin_bit;
    uint32_t end_bit;
    uint32_t in_place;       // keys_in == keys_out
    uint32_t n;
    uint32_t shift;          // lowest bit of this pass's digit in the ordered key
    uint32_t mask;           // digit mask (fewer bits on a final partial digit)
    uint32_t flip;           // mask for a descending sort, else 0
    uint32_t descending;
    uint32_t num_tiles;
    // chained scan
    uint32_t* status;        // [num_tiles][BINS] for this pass
    const uint32_t* ghist;   // [BINS] global histogram of this pass
    uint32_t* ticket;        // tile ticket of this pass
    uint32_t spin_limit;
    int32_t stall_tile;      // testing hook: tile index + 1 that never publishes
    // reduce-then-scan
    uint32_t* counts;        // [BINS][G] digit-major block counts (scanned in place)
    uint32_t G;
    uint32_t tiles_per_cta;
    uint32_t* err;
};

// Shared-memory layout of one tile (byte offsets, 16-byte aligned regions).
template <typename T, int RB, int THREADS, int ITEMS, int VB>
struct TileSmem {
    static constexpr int BINS = 1 << RB;
    static constexpr int WARPS = THREADS / 32;
    // Every tile kernel gives each digit its own thread for the per-digit
    // steps (counts, scans, starts, look-back), and the digit scan runs over
    // at most 32 warps.
    static_assert(THREADS >= BINS && THREADS % 32 == 0 && THREADS <= 1024,
                  "a tile needs at least one thread per digit");
    static constexpr int TILE = THREADS * ITEMS;
    static constexpr int WH = BINS + 1;  // per-array counters + one dummy slot for tail lanes
    // The shuffled tile: slot s holds a key and its value.  A 32-bit key and
    // a 32-bit value share one 8-byte slot (one shared-memory store and one
    // load per pair instead of two each); other shapes keep two arrays.
    static constexpr bool PAIRED = sizeof(T) == 4 && VB == 4;
    static constexpr size_t keys_off = 0;
    static constexpr size_t vals_off = PAIRED ? 0 : align_up(sizeof(T) * TILE, 16);
    static constexpr size_t wh_off = PAIRED ? align_up(8 * (size_t)TILE, 16)
                                            : vals_off + (VB ? align_up(sizeof(ValT<VB>) * (size_t)TILE, 16) : 0);
    static constexpr size_t base_off = wh_off + align_up(4 * (size_t)WARPS * WH, 16);
    static constexpr size_t scan_off = base_off + 4 * BINS;
    static constexpr size_t misc_off = scan_off + 4 * 32;
    static constexpr size_t io_off = misc_off + 16;  // this pass's 4 buffer pointers
    static constexpr size_t bytes = io_off + 32;
};

// Slot s of the shuffled tile (TileSmem::keys_off / vals_off, or the paired
// slots): store a key and its value, and read them back.
template <typename S, typename T, int VB>
__device__ __forceinline__ void slot_put(unsigned char* smem, uint32_t s, T key, ValT<VB> val)
{
    if constexpr (S::PAIRED) {
        reinterpret_cast<uint2*>(smem + S::keys_off)[s] = make_uint2((uint32_t)key, (uint32_t)val);
    } else {
        reinterpret_cast<T*>(smem + S::keys_off)[s] = key;
        if constexpr (VB != 0) reinterpret_cast<ValT<VB>*>(smem + S::vals_off)[s] = val;
    }
}

template <typename S, typename T, int VB>
__device__ __forceinline__ void slot_get(const unsigned char* smem, uint32_t s, T& key, ValT<VB>& val)
{
    if constexpr (S::PAIRED) {
        const uint2 kv = reinterpret_cast<const uint2*>(smem + S::keys_off)[s];
        key = (T)kv.x;
        val = kv.y;
    } else {
        key = reinterpret_cast<const T*>(smem + S::keys_off)[s];
        if constexpr (VB != 0) val = reinterpret_cast<const ValT<VB>*>(smem + S::vals_off)[s];
    }
}

// ------------------------------------------------------------ pass skipping
//
// The first read of the keys (the first upsweep, or the all-pass histogram)
// records two facts about the ordered keys in temp: `diff`, the OR over all
// keys of ordered(key) ^ ordered(keys[0]), whose clear bits are the bits that
// every key shares; and whether some adjacent pair is out of order in the
// sorted bit range.  A pass whose digit bits are all clear in diff leaves every
// key where it is (every key has the same digit and the pass is stable), so it
// is skipped, and an input that is already in order skips every pass (the
// early exit of "高性能计算：GPU上的基数排序", section 基数排序在GPU上的具体实现).
// Every kernel of a pass reads the record itself, so the decision needs no
// host round trip and a captured graph replays it.

// The pass plan from the finished record: pass q runs iff the input is not
// already in order and some bit of its digit differs between keys; its word
// holds runs | j << 8 | E << 16 (j = running passes before it, E = all
// running passes).
template <int RB>
__device__ __forceinline__ void write_plan(uint32_t diff_lo, uint32_t diff_hi, uint32_t unsorted,
                                           uint32_t* plan, uint32_t passes, uint32_t begin_bit, uint32_t end_bit)
{
    const uint64_t diff = ((uint64_t)diff_hi << 32) | diff_lo;
    uint32_t E = 0;
    for (uint32_t q = 0; q < passes; ++q) {
        const uint32_t shift = begin_bit + q * RB;
        const uint32_t width = min((uint32_t)RB, end_bit - shift);
        E += (unsorted != 0u && ((diff >> shift) & ((1ull << width) - 1ull)) != 0ull) ? 1u : 0u;
    }
    uint32_t j = 0;
    for (uint32_t q = 0; q < passes; ++q) {
        const uint32_t shift = begin_bit + q * RB;
        const uint32_t width = min((uint32_t)RB, end_bit - shift);
        const uint32_t run = (unsorted != 0u && ((diff >> shift) & ((1ull << width) - 1ull)) != 0ull) ? 1u : 0u;
        plan[q] = run | (j << 8) | (E << 16);
        j += run;
    }
}

// One thread's share of the record.  The order check compares the ordered
// keys masked to the sorted bit range in place (no shift needed: masking
// keeps the order of the range's value); MASKED = false when the range is the
// whole key.
template <int KT, bool MASKED = true>
struct SkipAcc {
    using T = typename KeyOps<KT>::T;
    T ref;          // ordered(keys[0])
    T rmask;        // bits [begin_bit, end_bit)
    T vflip;        // for a descending sort the check runs on complemented values
    T diff = 0;
    bool unsorted = false;

    __device__ __forceinline__ SkipAcc(const T* keys, uint32_t begin_bit, uint32_t end_bit, bool descending)
        : ref((T)KeyOps<KT>::ordered(keys[0])),
          rmask((T)((end_bit - begin_bit >= 64 ? ~0ull : (1ull << (end_bit - begin_bit)) - 1ull) << begin_bit)),
          vflip(descending ? (MASKED ? rmask : (T)~0ull) : T(0)) {}

    // Folds one key into diff and returns its value for the order check.
    __device__ __forceinline__ T visit(T k)
    {
        const T o = (T)KeyOps<KT>::ordered(k);
        diff |= o ^ ref;
        return MASKED ? (T)((o & rmask) ^ vflip) : (T)(o ^ vflip);
    }
    __device__ __forceinline__ T value(T k) const
    {
        const T o = (T)KeyOps<KT>::ordered(k);
        return MASKED ? (T)((o & rmask) ^ vflip) : (T)(o ^ vflip);
    }
    __device__ __forceinline__ void pair(T a, T b) { unsorted |= a > b; }

    // The keys of one 16-byte vector, checked in order; returns the values
    // of the first and the last.
    template <int VEC>
    __device__ __forceinline__ void vector(const T (&k)[VEC], T& first, T& last)
    {
        T prev = visit(k[0]);
        first = prev;
#pragma unroll
        for (int j = 1; j < VEC; ++j) {
            const T v = visit(k[j]);
            pair(prev, v);
            prev = v;
        }
        last = prev;
    }

    // Every thread of the block calls this once at the end, between two
    // barriers: each warp ORs its share into the block's words `blk` (3
    // words, zeroed before the first barrier); flush_block then adds the
    // block's to the record with one atomic per word, so that the CTAs do not
    // all queue on the record's line warp by warp.
    __device__ __forceinline__ void flush_warp(uint32_t* blk)
    {
        const uint64_t d = (uint64_t)diff;
        const uint32_t lo = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)d);
        const uint32_t hi = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)(d >> 32));
        const bool un = __any_sync(0xFFFFFFFFu, unsorted);
        if ((threadIdx.x & 31) == 0) {
            if (lo) atomicOr(blk + 0, lo);
            if (hi) atomicOr(blk + 1, hi);
            if (un) atomicOr(blk + 2, 1u);
        }
    }
    // Thread 0 of the last CTA to add its share also writes the pass plan.
    template <int RB>
    static __device__ __forceinline__ void flush_block(const uint32_t* blk, uint32_t* skip, uint32_t* plan,
                                                       uint32_t passes, uint32_t begin_bit, uint32_t end_bit)
    {
        if (threadIdx.x == 0) {
            if (blk[0]) atomicOr(skip + 0, blk[0]);
            if (blk[1]) atomicOr(skip + 1, blk[1]);
            if (blk[2]) atomicOr(skip + 2, 1u);
            __threadfence();
            if (atomicAdd(skip + 3, 1u) == gridDim.x - 1) {
                __threadfence();
                write_plan<RB>(ld_relaxed_gpu(skip + 0), ld_relaxed_gpu(skip + 1), ld_relaxed_gpu(skip + 2),
                               plan, passes, begin_bit, end_bit);
            }
        }
    }
};

// Which passes run: `run` for this pass, `j` = how many running passes come
// before it, `E` = how many run in all.
struct PassRole {
    bool run;
    uint32_t j;
    uint32_t E;
};

__device__ __forceinline__ PassRole decode_plan(uint32_t w)
{
    return PassRole{(w & 1u) != 0u, (w >> 8) & 0xFFu, (w >> 16) & 0xFFu};
}

// This pass's plan word, read by one thread per CTA.
__device__ __forceinline__ uint32_t load_plan(const PassParams& p) { return p.plan[p.pass]; }

struct RoleShared {
    uint32_t run, j, E;
};

__device__ __forceinline__ void publish_role(RoleShared* sh, const PassRole& r)
{
    sh->run = r.run ? 1u : 0u;
    sh->j = r.j;
    sh->E = r.E;
}

__device__ __forceinline__ PassRole read_role(const RoleShared* sh)
{
    return PassRole{sh->run != 0u, sh->j, sh->E};
}

// Thread 0 reads the plan; every thread returns it (holds a barrier).
__device__ __forceinline__ PassRole block_pass_role(const PassParams& p, RoleShared* sh)
{
    if (threadIdx.x == 0) publish_role(sh, decode_plan(load_plan(p)));
    __syncthreads();
    return read_role(sh);
}

// Buffer i of the chain of running passes: i = 0 is the sort's input.  Out of
// place, buffers 1..E alternate so that buffer E is keys_out.  In place, even
// i is keys_out (= keys_in) and odd i the partner, so with E odd the result
// ends in the partner and k_chain_copy moves it back.  (The host plans the
// every-pass-runs case with the same rule.)
__host__ __device__ __forceinline__ bool chain_is_out(uint32_t i, uint32_t E, bool in_place)
{
    return in_place ? (i % 2u == 0u) : ((E - i) % 2u == 0u);
}

// This pass's source and destination for role r.
template <int VB>
__device__ __forceinline__ void pass_buffers(PassParams& p, const PassRole& r)
{
    const bool ip = p.in_place != 0u;
    const bool src_out = chain_is_out(r.j, r.E, ip), dst_out = chain_is_out(r.j + 1, r.E, ip);
    p.keys_in = r.j == 0 ? p.sort_keys_in : (src_out ? p.sort_keys_out : p.alt_keys);
    p.keys_out = dst_out ? p.sort_keys_out : p.alt_keys;
    if constexpr (VB != 0) {
        p.vals_in = r.j == 0 ? p.sort_vals_in : (src_out ? p.sort_vals_out : p.alt_vals);
        p.vals_out = dst_out ? p.sort_vals_out : p.alt_vals;
    }
}

// Copy elements [lo, hi) of the keys (and values), thread t of `stride`.
template <typename T, int VB>
__device__ __forceinline__ void copy_span(const T* src, T* dst, const void* vsrc, void* vdst,
                                          size_t lo, size_t hi, size_t t, size_t stride)
{
    for (size_t i = lo + t; i < hi; i += stride) {
        dst[i] = src[i];
        if constexpr (VB != 0) static_cast<ValT<VB>*>(vdst)[i] = static_cast<const ValT<VB>*>(vsrc)[i];
    }
}

// When no pass runs, the last pass's kernel copies the input to the output
// (out of place); its CTAs cover [lo, hi) each.
template <typename T, int VB>
__device__ __forceinline__ void copy_if_no_pass_runs(const PassParams& p, const PassRole& r, size_t lo, size_t hi)
{
    if (r.E == 0u && p.pass + 1u == p.passes && p.in_place == 0u)
        copy_span<T, VB>(static_cast<const T*>(p.sort_keys_in), static_cast<T*>(p.sort_keys_out),
                           p.sort_vals_in, p.sort_vals_out, lo, hi < p.n ? hi : p.n, threadIdx.x, blockDim.x);
}

// --------------------------------------------------------------- tile pieces

// Load ITEMS keys per thread in warp-striped order: lane l of warp w holds
// positions seg + k*32 + l, so every load instruction of a warp covers 32
// consecutive keys and the processing order (k, lane) is the input order.
template <bool FULL, typename T, int ITEMS>
__device__ __forceinline__ void load_striped(const T* __restrict__ src, uint32_t seg, uint32_t n,
                                             int lane, T (&v)[ITEMS])
{
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t i = seg + k * 32 + lane;
        if (FULL) v[k] = src[i];
        else v[k] = i < n ? src[i] : T(0);
    }
}

// When a pass was skipped, the buffers of the passes after it live in shared
// memory (PassIO, written once per CTA by set_pass_io) rather than in
// registers, which the tile loop has none to spare for; each use reloads them.
struct PassIO {
    const void* keys_in;
    void* keys_out;
    const void* vals_in;
    void* vals_out;
};

__device__ __forceinline__ void* lds_ptr(const void* slot)
{
    uint64_t v;
    asm volatile("ld.volatile.shared.u64 %0, [%1];"
                 : "=l"(v)
                 : "r"((uint32_t)__cvta_generic_to_shared(slot)));
    return reinterpret_cast<void*>(v);
}

template <typename S>
__device__ __forceinline__ void set_pass_io(unsigned char* smem, const PassParams& p)
{
    if (threadIdx.x == 0) {
        PassIO* io = reinterpret_cast<PassIO*>(smem + S::io_off);
        io->keys_in = p.keys_in;
        io->keys_out = p.keys_out;
        io->vals_in = p.vals_in;
        io->vals_out = p.vals_out;
    }
}

template <typename S, typename T>
__device__ __forceinline__ const T* io_keys_in(const unsigned char* smem)
{
    return static_cast<const T*>(lds_ptr(&reinterpret_cast<const PassIO*>(smem + S::io_off)->keys_in));
}
template <typename S, typename T>
__device__ __forceinline__ T* io_keys_out(const unsigned char* smem)
{
    return static_cast<T*>(lds_ptr(&reinterpret_cast<const PassIO*>(smem + S::io_off)->keys_out));
}
template <typename S, typename V>
__device__ __forceinline__ const V* io_vals_in(const unsigned char* smem)
{
    return static_cast<const V*>(lds_ptr(&reinterpret_cast<const PassIO*>(smem + S::io_off)->vals_in));
}
template <typename S, typename V>
__device__ __forceinline__ V* io_vals_out(const unsigned char* smem)
{
    return static_cast<V*>(lds_ptr(&reinterpret_cast<const PassIO*>(smem + S::io_off)->vals_out));
}

// Keys (and values) of one tile in warp-striped order; a tile that runs past
// n is guarded lane by lane.  The source is the pass's planned buffer
// (p.keys_in), or with DYN the one in the PassIO slots.
template <int KT, int RB, int THREADS, int ITEMS, int VB, bool DYN>
__device__ __forceinline__ void load_tile(const PassParams& p, const unsigned char* smem, uint32_t tile,
                                          typename KeyOps<KT>::T (&key)[ITEMS],
                                          ValT<VB> (&val)[VB ? ITEMS : 1])
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    constexpr uint32_t TILE = THREADS * ITEMS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t seg = tile * TILE + (uint32_t)warp * (32u * ITEMS);
    const T* kin = DYN ? io_keys_in<S, T>(smem) : static_cast<const T*>(p.keys_in);
    if ((tile + 1) * TILE <= p.n) {
        load_striped<true, T, ITEMS>(kin, seg, p.n, lane, key);
        if constexpr (VB != 0)
            load_striped<true, ValT<VB>, ITEMS>(DYN ? io_vals_in<S, ValT<VB>>(smem)
                                                    : static_cast<const ValT<VB>*>(p.vals_in),
                                                seg, p.n, lane, val);
    } else {
        load_striped<false, T, ITEMS>(kin, seg, p.n, lane, key);
        if constexpr (VB != 0)
            load_striped<false, ValT<VB>, ITEMS>(DYN ? io_vals_in<S, ValT<VB>>(smem)
                                                     : static_cast<const ValT<VB>*>(p.vals_in),
                                                 seg, p.n, lane, val);
    }
}

// Mask of the lanes of this warp whose value equals this lane's (the low
// BITS bits of v are compared; higher bits must be zero).  The top
// RS_MATCH_BITS of the digit (and any bit above it) go through
// __match_any_sync, the rest through one __ballot_sync per bit.
template <int BITS, int RB>
__device__ __forceinline__ uint32_t warp_peers(uint32_t v)
{
    constexpr int BALLOT_BITS = (RB - RS_MATCH_BITS) < 0 ? 0 : (RB - RS_MATCH_BITS);
    uint32_t peers = (BITS > BALLOT_BITS) ? __match_any_sync(0xFFFFFFFFu, v >> BALLOT_BITS) : 0xFFFFFFFFu;
#pragma unroll
    for (int b = 0; b < (BITS < BALLOT_BITS ? BITS : BALLOT_BITS); ++b) {
        const uint32_t bit = (v >> b) & 1u;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, bit);
        peers &= bal ^ (bit - 1u);  // bit - 1 is all ones exactly when the bit is clear
    }
    return peers;
}

// Stable rank of each key among equal digits within its warp's segment.
// For each step k the lanes holding the same digit (peers) are found; a key's
// rank is the warp's running count for its digit plus the number of peers
// below it, and all peers then store the same advanced count (no branch).
// Ranks (< 2^16) are packed two per register: rank[k/2] holds step k in its
// low half when k is even, in its high half when k is odd.  On a partial
// tile, lanes past the end get digit BINS, which has its own dummy counter.
template <bool FULL, int KT, int RB, int ITEMS>
__device__ __forceinline__ uint32_t step_digit(const typename KeyOps<KT>::T (&key)[ITEMS], int k, uint32_t seg,
                                               uint32_t n, uint32_t shift, uint32_t mask, uint32_t flip,
                                               int lane)
{
    const uint32_t d = digit_of<KT>(key[k], shift, mask, flip);
    return (FULL || seg + k * 32 + lane < n) ? d : (1u << RB);
}

template <bool FULL, int KT, int RB, int ITEMS>
__device__ __forceinline__ void rank_in_warp(const typename KeyOps<KT>::T (&key)[ITEMS], uint32_t seg,
                                             uint32_t n, uint32_t shift, uint32_t mask, uint32_t flip,
                                             uint32_t* cnt, int lane, uint32_t (&rank)[(ITEMS + 1) / 2])
{
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < (ITEMS + 1) / 2; ++i) rank[i] = 0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t d = step_digit<FULL, KT, RB, ITEMS>(key, k, seg, n, shift, mask, flip, lane);
        const uint32_t peers = warp_peers<FULL ? RB : RB + 1, RB>(d);
        const uint32_t prior = cnt[d];
        cnt[d] = prior + __popc(peers);
        const uint32_t r = prior + __popc(peers & lt);
        rank[k / 2] |= (k & 1) ? (r << 16) : r;
        __syncwarp();
    }
}

// Zero the tile's digit counters (the caller synchronises before ranking).
template <typename S>
__device__ __forceinline__ void zero_counters(unsigned char* smem, int threads)
{
    uint32_t* whist = reinterpret_cast<uint32_t*>(smem + S::wh_off);
    for (int i = threadIdx.x; i < S::WARPS * S::WH; i += threads) whist[i] = 0;
}

// Zero this warp's own digit counters, after the warp has read its digit
// starts from them in the shuffle.  Only this warp touches them again before
// the next ranking barrier, so a warp barrier suffices.
template <typename S>
__device__ __forceinline__ void zero_warp_counters(unsigned char* smem)
{
    uint32_t* wh = reinterpret_cast<uint32_t*>(smem + S::wh_off) + (threadIdx.x >> 5) * S::WH;
    for (int i = threadIdx.x & 31; i < S::WH; i += 32) wh[i] = 0;
    __syncwarp();
}

// Everything of one tile, whose keys are in registers, up to the point where
// its global digit offsets are needed: rank, per-digit counts, tile-local
// digit starts, shuffle into shared memory.  Returns, for thread d < BINS,
// the tile's count of digit d in *cnt and its tile-local start in *start.
// `publish(d, cnt)` runs for every digit as soon as the count is known (the
// chained scan publishes it there).  The key/value registers are free again
// on return (the downsweep loads its next tile into them).
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, int VB, typename Publish>
__device__ __forceinline__ void tile_rank_and_shuffle(const PassParams& p, unsigned char* smem,
                                                      uint32_t tile,
                                                      const typename KeyOps<KT>::T (&key)[ITEMS],
                                                      const ValT<VB> (&val)[VB ? ITEMS : 1],
                                                      uint32_t* cnt_out, uint32_t* start_out,
                                                      Publish publish)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    constexpr int BINS = S::BINS, TILE = S::TILE, WH = S::WH, WARPS = S::WARPS;
    uint32_t* whist = reinterpret_cast<uint32_t*>(smem + S::wh_off);
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tile_base = tile * (uint32_t)TILE;
    const uint32_t seg = tile_base + (uint32_t)warp * (32u * ITEMS);

    // (the caller has zeroed the counters and synchronised)
    uint32_t rank[(ITEMS + 1) / 2];
    rank_in_warp<FULL, KT, RB, ITEMS>(key, seg, p.n, p.shift, p.mask, p.flip, whist + warp * WH, lane, rank);
    __syncthreads();

    // Per digit: the tile count, and after the scan each warp's start for the
    // digit inside the tile (the warps' counts are read twice rather than
    // held in registers).
    uint32_t cnt = 0;
    if (tid < BINS) {
#pragma unroll
        for (int w = 0; w < WARPS; ++w) cnt += whist[w * WH + tid];
        publish(tid, cnt);
    }
    const uint32_t start = bins_exclusive_scan<BINS, false>(tid < BINS ? cnt : 0u, sscan + 16, nullptr);
    if (tid < BINS) {
        uint32_t run = start;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const uint32_t c = whist[w * WH + tid];
            whist[w * WH + tid] = run;
            run += c;
        }
    }
    __syncthreads();

    // Shuffle: each digit becomes one contiguous run of the tile.  pos < TILE
    // holds by construction; the clamp keeps a violation inside the tile.
    uint32_t bad = 0;
    const uint32_t* wbase = whist + warp * WH;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t d = step_digit<FULL, KT, RB, ITEMS>(key, k, seg, p.n, p.shift, p.mask, p.flip, lane);
        const uint32_t r = (k & 1) ? (rank[k / 2] >> 16) : (rank[k / 2] & 0xFFFFu);
        uint32_t pos = wbase[d] + r;
#if RS_CHECKED
        bad |= pos >= (uint32_t)TILE;
#endif
        pos = min(pos, (uint32_t)TILE - 1u);
        if (FULL || d < (uint32_t)BINS) {
            if constexpr (VB != 0) slot_put<S, T, VB>(smem, pos, key[k], val[k]);
            else slot_put<S, T, VB>(smem, pos, key[k], 0u);
        }
    }
    if (bad) record_error(p.err, RS_ERR_CHECK_FAILED);
    *cnt_out = cnt;
    *start_out = start;
}

// Scatter the shuffled tile: slot s holds a key of digit d, whose global
// position is sbase[d] + s (sbase = global offset of the digit's run minus
// its tile-local start).  Consecutive slots mostly share a digit, so each
// warp store covers few, contiguous segments.  Positions are bounds-checked
// (a failure is recorded and the store skipped).  KEEP marks the stored lines
// evict-last in L2: in reduce-then-scan the next tile of the same CTA soon
// fills the rest of each digit run's last, half-written line; the chained
// scan's neighbouring tiles run on other CTAs at other times, and there the
// hint measured slower (2^28 uint32 keys: 1.10 vs 1.14 ms per pass).
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, int VB, bool KEEP = true>
__device__ __forceinline__ void tile_scatter(const PassParams& p, unsigned char* smem, uint32_t tile,
                                             typename KeyOps<KT>::T* out, ValT<VB>* vout)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    constexpr int TILE = S::TILE;
    const uint32_t* sbase = reinterpret_cast<const uint32_t*>(smem + S::base_off);
    const uint32_t tile_base = tile * (uint32_t)TILE;
    const uint32_t valid = FULL ? (uint32_t)TILE : p.n - tile_base;
    uint32_t bad = 0;
    const uint64_t pol = KEEP ? l2_evict_last_policy() : 0ull;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t s = (uint32_t)(k * THREADS) + threadIdx.x;
        if (FULL || s < valid) {
            T kk;
            ValT<VB> vv;
            slot_get<S, T, VB>(smem, s, kk, vv);
            const uint32_t idx = sbase[digit_of<KT>(kk, p.shift, p.mask, p.flip)] + s;
            const bool ok = idx < p.n;
            bad |= !ok;
            if (ok) {
                if constexpr (KEEP) {
                    st_keep(out + idx, kk, pol);
                    if constexpr (VB != 0) st_keep(vout + idx, vv, pol);
                } else {
                    out[idx] = kk;
                    if constexpr (VB != 0) vout[idx] = vv;
                }
            }
        }
    }
    if (bad) record_error(p.err, RS_ERR_CHECK_FAILED);
}

// Decoupled look-back for digit d of `tile` (one thread per digit): sum the
// predecessors' published counts, newest first, until one that already holds
// an inclusive sum.  RS_LOOKBACK_BATCH statuses are read per round trip; an
// unpublished status stops the round and is polled again, at most spin_limit
// times in a row, after which the timeout is recorded and the sum so far
// returned.
// The first RS_LOOKBACK_BATCH statuses are read early (pre[], issued before
// the tile's shuffle so that their latency overlaps it); the walk then goes
// on from where they leave off.
template <int B>
__device__ __forceinline__ void lookback_preload(const PassParams& p, uint32_t tile, uint32_t d,
                                                 uint32_t bins, uint32_t (&pre)[B])
{
    const int32_t t = (int32_t)tile - 1;
#pragma unroll
    for (int j = 0; j < B; ++j)
        pre[j] = (t - j >= 0) ? ld_relaxed_gpu(p.status + (size_t)(t - j) * bins + d) : 0u;
}

template <int B>
__device__ __forceinline__ uint32_t lookback(const PassParams& p, uint32_t tile, uint32_t d, uint32_t bins,
                                             const uint32_t (&pre)[B])
{
    uint32_t excl = 0;
    int32_t t = (int32_t)tile - 1;
    uint32_t spins = 0, sleep_ns = 0;
    uint32_t s[B];
#pragma unroll
    for (int j = 0; j < B; ++j) s[j] = pre[j];
    while (true) {
        // Consume the newest-first batch up to an unpublished status or an
        // inclusive one.
        int consumed = 0;
        bool stop = false, inclusive = false;
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (!stop) {
                const uint32_t f = s[j] & ~kValMask;
                if (f == 0u) {
                    stop = true;
                } else {
                    excl += s[j] & kValMask;
                    ++consumed;
                    if (f == kFlagInc) stop = inclusive = true;
                }
            }
        }
        if (inclusive) return excl;
        t -= consumed;
        if (t < 0) break;  // ran past tile 0, which always publishes an inclusive sum
        if (consumed == 0) {
            // The nearest unread status is not published yet: poll it alone.
            if (++spins >= p.spin_limit) break;
            if (sleep_ns) __nanosleep(sleep_ns);
            sleep_ns = sleep_ns ? min(sleep_ns * 2, 256u) : 16u;
            s[0] = ld_relaxed_gpu(p.status + (size_t)t * bins + d);
#pragma unroll
            for (int j = 1; j < B; ++j) s[j] = 0u;
            continue;
        }
        spins = 0;
        sleep_ns = 0;
#pragma unroll
        for (int j = 0; j < B; ++j)
            s[j] = (t - j >= 0) ? ld_relaxed_gpu(p.status + (size_t)(t - j) * bins + d) : 0u;
    }
    record_error(p.err, RS_ERR_DEVICE_TIMEOUT);
    __threadfence();
    return excl;
}

// ------------------------------------------------------------------ kernels

// One tile of a chained-scan pass.
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, int VB>
__device__ __forceinline__ void onesweep_tile(const PassParams& p, unsigned char* smem, uint32_t tile,
                                              const typename KeyOps<KT>::T (&key)[ITEMS],
                                              const ValT<VB> (&val)[VB ? ITEMS : 1])
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    constexpr int BINS = S::BINS;
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem + S::base_off);
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);
    const int tid = threadIdx.x;
    const bool stalled = (int32_t)tile + 1 == p.stall_tile;
    uint32_t* my_status = p.status + (size_t)tile * BINS;

    // Tile 0 needs the pass's global digit starts: an exclusive scan of the
    // histogram.  Its published value is then already inclusive and absolute.
    uint32_t gexcl = 0;
    if (tile == 0) gexcl = bins_exclusive_scan<BINS>(tid < BINS ? p.ghist[tid] : 0u, sscan, nullptr);

    uint32_t cnt, start;
    uint32_t pre[RS_LOOKBACK_BATCH];
    tile_rank_and_shuffle<FULL, KT, RB, THREADS, ITEMS, VB>(
        p, smem, tile, key, val, &cnt, &start, [&](int d, uint32_t c) {
            if (!stalled) {
                if (tile == 0) st_relaxed_gpu(my_status + d, kFlagInc | ((gexcl + c) & kValMask));
                else st_relaxed_gpu(my_status + d, kFlagAgg | (c & kValMask));
            }
            if (tile > 0) lookback_preload<RS_LOOKBACK_BATCH>(p, tile, d, BINS, pre);
        });
    if (tid < BINS) {
        uint32_t excl = gexcl;
        if (tile > 0) {
            excl = lookback<RS_LOOKBACK_BATCH>(p, tile, tid, BINS, pre);
            if (!stalled) st_relaxed_gpu(my_status + tid, kFlagInc | ((excl + cnt) & kValMask));
        }
        sbase[tid] = excl - start;
    }
    T* out = io_keys_out<S, T>(smem);
    ValT<VB>* vout = VB ? io_vals_out<S, ValT<VB>>(smem) : nullptr;
    __syncthreads();
    tile_scatter<FULL, KT, RB, THREADS, ITEMS, VB, false>(p, smem, tile, out, vout);
}

// Chained-scan pass: one tile per CTA, in the order of an atomic ticket, so
// every tile a CTA waits on belongs to a CTA that already runs.
template <int KT, int RB, int THREADS, int ITEMS, int VB>
__global__ void __launch_bounds__(THREADS, RS_TILE_MIN_THREADS_PER_SM / THREADS) k_onesweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* smisc = reinterpret_cast<uint32_t*>(smem + S::misc_off);
    const int tid = threadIdx.x;
    RoleShared* rsh = reinterpret_cast<RoleShared*>(smisc + 1);
    zero_counters<S>(smem, THREADS);
    wait_prior_grid();
    if (tid == 0) {
        // The skip record is read and the ticket taken together, so the two
        // round trips overlap (a skipped pass leaves its tickets unused).
        const uint32_t w = load_plan(p);
        smisc[0] = atomicAdd(p.ticket, 1u);
        const PassRole r = decode_plan(w);
        publish_role(rsh, r);
        if (r.run) {
            PassParams q = p;
            pass_buffers<VB>(q, r);
            set_pass_io<S>(smem, q);
        }
    }
    __syncthreads();
    const PassRole role = read_role(rsh);
    if (!role.run) {
        const size_t lo = (size_t)blockIdx.x * S::TILE;
        copy_if_no_pass_runs<T, VB>(p, role, lo, lo + S::TILE);
        return;
    }
    const uint32_t tile = smisc[0];
    if (tile >= p.num_tiles) return;
    T key[ITEMS];
    ValT<VB> val[VB ? ITEMS : 1];
    load_tile<KT, RB, THREADS, ITEMS, VB, true>(p, smem, tile, key, val);
    if ((tile + 1) * (uint32_t)S::TILE <= p.n)
        onesweep_tile<true, KT, RB, THREADS, ITEMS, VB>(p, smem, tile, key, val);
    else
        onesweep_tile<false, KT, RB, THREADS, ITEMS, VB>(p, smem, tile, key, val);
}

// Reduce-then-scan, step 1: digit histogram of each CTA's chunk, written
// digit-major (counts[d * G + g]) so that one exclusive scan of the whole
// array yields every (digit, CTA) start ("Radix sort paralelo sobre el scan",
// section "Las tres fases de una pasada").
// The first upsweep (FIRST) also writes the pass-skip record (FULLRANGE: the
// sorted bits are the whole key, so its order check needs no mask); every
// later one runs only if its pass does.
template <int KT, int RB, int THREADS, int TILE, bool FIRST, bool FULLRANGE = false>
__global__ void __launch_bounds__(THREADS) k_upsweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    constexpr int BINS = 1 << RB;
    constexpr int COLS = 32;          // lane-private counter columns: hist[bin][lane]
    constexpr int VEC = 16 / sizeof(T);
    constexpr int U = 4;              // vectors in flight per thread
    __shared__ uint32_t hist[BINS * COLS];
    __shared__ RoleShared rsh;
    __shared__ uint32_t skip_blk[3];
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t col = lane;
    for (int i = tid; i < BINS * COLS; i += THREADS) hist[i] = 0;
    if (FIRST && tid < 3) skip_blk[tid] = 0;
    wait_prior_grid();
    if constexpr (!FIRST) {
        const PassRole role = block_pass_role(p, &rsh);  // (its barrier also covers the zeroing)
        if (!role.run) return;
        pass_buffers<false>(p, role);
    } else {
        __syncthreads();
    }
    const uint32_t g = blockIdx.x;
    const uint64_t lo64 = (uint64_t)g * p.tiles_per_cta * TILE;
    const uint32_t lo = lo64 < p.n ? (uint32_t)lo64 : p.n;
    const uint64_t hi64 = lo64 + (uint64_t)p.tiles_per_cta * TILE;
    const uint32_t hi = hi64 < p.n ? (uint32_t)hi64 : p.n;
    const T* src = static_cast<const T*>(p.keys_in);
    auto count = [&](T k) { atomicAdd(&hist[digit_of<KT>(k, p.shift, p.mask, p.flip) * COLS + col], 1u); };
    SkipAcc<KT, !FULLRANGE> acc(src, p.begin_bit, p.end_bit, p.descending != 0u);
    // lo is a multiple of TILE, so lo * sizeof(T) is 16-byte aligned whenever the base is.
    uint32_t i = lo;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const uint32_t nvec = (hi - lo) / VEC;
        const uint4* sv = reinterpret_cast<const uint4*>(src + lo);
        // Full rounds (U vectors per thread, the same trip count in every
        // warp), then what is left.  Thread v + 1 holds the vector after
        // thread v's, so a shuffle brings the next key for the order check.
        const uint32_t per_round = U * THREADS, rounds = nvec / per_round;
        for (uint32_t r = 0; r < rounds; ++r) {
            uint4 w[U];
            T nb[FIRST ? U : 1];  // lane 31: the key after its vector, loaded with the round
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t v = r * per_round + u * THREADS + tid;
                w[u] = __ldcs(sv + v);
                if constexpr (FIRST) nb[u] = (lane == 31 && v + 1 < nvec) ? src[lo + (v + 1) * VEC] : T(0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                T k[VEC];
                memcpy(k, &w[u], 16);
#pragma unroll
                for (int j = 0; j < VEC; ++j) count(k[j]);
                if constexpr (FIRST) {
                    const uint32_t v = r * per_round + u * THREADS + tid;
                    T first, last;
                    acc.vector(k, first, last);
                    T next = __shfl_down_sync(0xFFFFFFFFu, first, 1);
                    if (lane == 31) next = v + 1 < nvec ? acc.value(nb[u]) : last;
                    acc.pair(last, next);
                }
            }
        }
        for (uint32_t v = rounds * per_round + tid; v < nvec; v += THREADS) {
            const uint4 w = __ldcs(sv + v);
            T k[VEC];
            memcpy(k, &w, 16);
#pragma unroll
            for (int j = 0; j < VEC; ++j) count(k[j]);
            if constexpr (FIRST) {
                T first, last;
                acc.vector(k, first, last);
                if (v + 1 < nvec) acc.pair(last, acc.value(src[lo + (v + 1) * VEC]));
            }
        }
        i = lo + nvec * VEC;
    }
    for (i += tid; i < hi; i += THREADS) {
        const T k = src[i];
        count(k);
        if constexpr (FIRST) {
            const T v = acc.visit(k);
            if (i > 0) acc.pair(acc.value(src[i - 1]), v);
        }
    }
    if constexpr (FIRST) {
        if (tid == 0 && lo > 0 && lo < hi) acc.pair(acc.value(src[lo - 1]), acc.value(src[lo]));
        acc.flush_warp(skip_blk);
    }
    __syncthreads();
    if constexpr (FIRST)
        SkipAcc<KT, !FULLRANGE>::template flush_block<RB>(skip_blk, p.skip, p.plan, p.passes, p.begin_bit,
                                                          p.end_bit);
    for (int d = tid; d < BINS; d += THREADS) {
        uint32_t c = 0;
#pragma unroll 8
        for (int j = 0; j < COLS; ++j) c += hist[d * COLS + ((j + d) & (COLS - 1))];
        p.counts[(size_t)d * p.G + g] = c;
    }
}

// Reduce-then-scan, step 2: exclusive scan of the digit-major counts.  CTA d
// scans row d (its G per-CTA counts) in place and writes the row total; the
// downsweep adds the exclusive scan of the row totals (the digit starts).
template <int RB, int THREADS>
__global__ void __launch_bounds__(THREADS) k_spine_scan(PassParams p, uint32_t* row_total)
{
    // Each thread owns PER consecutive counts (G <= kRtsMaxCtas): all its
    // loads are issued at once, together with the plan read, so the kernel
    // pays about one memory latency before the scan and one after.
    constexpr uint32_t PER = (kRtsMaxCtas + THREADS - 1) / THREADS;
    __shared__ uint32_t sscan[32];
    __shared__ RoleShared rsh;
    const int tid = threadIdx.x;
    const uint32_t G = p.G;
    uint32_t* row = p.counts + (size_t)blockIdx.x * G;
    const uint32_t per = (G + THREADS - 1) / THREADS;
    const uint32_t lo = min(G, tid * per), hi = min(G, lo + per);
    wait_prior_grid();
    uint32_t c[PER];
#pragma unroll
    for (uint32_t j = 0; j < PER; ++j) c[j] = lo + j < hi ? row[lo + j] : 0u;
    if (!block_pass_role(p, &rsh).run) return;  // (a skipped pass's counts are stale, unused)
    uint32_t sum = 0;
#pragma unroll
    for (uint32_t j = 0; j < PER; ++j) sum += c[j];
    uint32_t total;
    uint32_t run = bins_exclusive_scan<THREADS>(sum, sscan, &total);
#pragma unroll
    for (uint32_t j = 0; j < PER; ++j) {
        if (lo + j < hi) row[lo + j] = run;
        run += c[j];
    }
    if (tid == 0) row_total[blockIdx.x] = total;
}

// Shared memory of a downsweep CTA: the tile layout, then (when the tiles are
// staged by bulk copies) the stage and its mbarrier.
template <typename T, int RB, int THREADS, int ITEMS, int VB>
struct DownsweepSmem {
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    static constexpr bool kStaged = RS_TMA_TILES && VB == 0 && sizeof(T) <= 4 && RB == 8;
    static constexpr size_t stage_off = align_up(S::bytes, 128);
    static constexpr size_t bar_off = stage_off + sizeof(T) * (size_t)S::TILE;
    static constexpr size_t bytes = kStaged ? bar_off + 16 : S::bytes;
};

// Reduce-then-scan, step 3: each CTA walks its chunk tile by tile, keeping a
// running global offset per digit.
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, int VB, bool DYN, bool STAGED = false>
__device__ __forceinline__ void downsweep_tile(const PassParams& p, unsigned char* smem, uint32_t tile,
                                               uint32_t next, uint32_t& running,
                                               typename KeyOps<KT>::T (&key)[ITEMS],
                                               ValT<VB> (&val)[VB ? ITEMS : 1])
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    constexpr int BINS = S::BINS;
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem + S::base_off);
    const int tid = threadIdx.x;
    uint32_t cnt, start;
    tile_rank_and_shuffle<FULL, KT, RB, THREADS, ITEMS, VB>(p, smem, tile, key, val, &cnt, &start,
                                                               [](int, uint32_t) {});
    if constexpr (STAGED) {
        // The ranking barrier above means every thread has moved the stage
        // into registers: refill it with the next full tile.
        if (tid == 0 && next != 0xFFFFFFFFu) {
            using D = DownsweepSmem<T, RB, THREADS, ITEMS, VB>;
            const T* src = DYN ? io_keys_in<S, T>(smem) : static_cast<const T*>(p.keys_in);
            fence_proxy_async_smem();
            bulk_load(smem + D::stage_off, src + (size_t)next * S::TILE, (uint32_t)(sizeof(T) * S::TILE),
                      reinterpret_cast<uint64_t*>(smem + D::bar_off));
        }
    } else if (next != 0xFFFFFFFFu) {
        load_tile<KT, RB, THREADS, ITEMS, VB, DYN>(p, smem, next, key, val);
    }
    T* out = DYN ? io_keys_out<S, T>(smem) : static_cast<T*>(p.keys_out);
    ValT<VB>* vout = VB ? (DYN ? io_vals_out<S, ValT<VB>>(smem) : static_cast<ValT<VB>*>(p.vals_out)) : nullptr;
    if (tid < BINS) {
        sbase[tid] = running - start;
        running += cnt;
    }
    __syncthreads();
    if constexpr (VB == 0 && sizeof(T) <= 4 && (IsByte<KT>::value || RB == 4)) {
        // Keys only, 32- or 16-bit, byte digits or 4-bit digits: no block
        // barrier after the scatter.  The next tile's first shared-memory
        // writes outside this warp's counters (digit starts, the shuffle, the
        // scatter bases, the stage refill) all come after its ranking barrier,
        // which every thread reaches only after this scatter.  (Measured on
        // GB300, 2^28 keys: -0.8% per uint32 and uint16 pass, -1.4% per 4-bit
        // pass.  The tiles with values or 64-bit keys ran 4-6% slower without
        // it, and the general 8-bit digit kernel spills 7x more registers
        // without it, so those keep it.)
        zero_warp_counters<S>(smem);  // for the next tile; the scatter does not read them
        tile_scatter<FULL, KT, RB, THREADS, ITEMS, VB>(p, smem, tile, out, vout);
        __syncwarp();
    } else {
        zero_counters<S>(smem, THREADS);  // for the next tile; the scatter does not read them
        tile_scatter<FULL, KT, RB, THREADS, ITEMS, VB>(p, smem, tile, out, vout);
        __syncthreads();  // the next tile reuses shared memory
    }
}

// The tile loop of one downsweep CTA.  DYN: the pass's buffers come from the
// PassIO slots (some earlier pass was skipped) instead of the host's plan.
template <int KT, int RB, int THREADS, int ITEMS, int VB, bool DYN>
__device__ __forceinline__ void downsweep_loop(const PassParams& p, unsigned char* smem, uint32_t running)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    const uint32_t t0 = blockIdx.x * p.tiles_per_cta;
    const uint32_t t1 = min(p.num_tiles, t0 + p.tiles_per_cta);
    if (t0 >= t1) return;
    T key[ITEMS];
    ValT<VB> val[VB ? ITEMS : 1];
    load_tile<KT, RB, THREADS, ITEMS, VB, DYN>(p, smem, t0, key, val);
    for (uint32_t tile = t0; tile < t1; ++tile) {
        const uint32_t next = tile + 1 < t1 ? tile + 1 : 0xFFFFFFFFu;
        if ((tile + 1) * (uint32_t)S::TILE <= p.n)
            downsweep_tile<true, KT, RB, THREADS, ITEMS, VB, DYN>(p, smem, tile, next, running, key, val);
        else
            downsweep_tile<false, KT, RB, THREADS, ITEMS, VB, DYN>(p, smem, tile, next, running, key, val);
    }
}


// The tile loop with every full tile staged in shared memory by a bulk copy
// issued while the previous tile is ranked and scattered; keys then move from
// the stage into registers warp-striped, as load_tile would place them.  A
// partial last tile is loaded directly.  Source must be 16-byte aligned.
template <int KT, int RB, int THREADS, int ITEMS, bool DYN>
__device__ __forceinline__ void downsweep_loop_staged(const PassParams& p, unsigned char* smem, uint32_t running)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, 0>;
    using D = DownsweepSmem<T, RB, THREADS, ITEMS, 0>;
    constexpr uint32_t TILE = S::TILE, BYTES = (uint32_t)(sizeof(T) * S::TILE);
    const uint32_t t0 = blockIdx.x * p.tiles_per_cta;
    const uint32_t t1 = min(p.num_tiles, t0 + p.tiles_per_cta);
    if (t0 >= t1) return;
    const uint32_t tf = min(t1, p.n / TILE);  // tiles [t0, tf) are full
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T* src = DYN ? io_keys_in<S, T>(smem) : static_cast<const T*>(p.keys_in);
    const T* stage = reinterpret_cast<const T*>(smem + D::stage_off);
    (void)BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + D::bar_off);
    if (tid == 0 && t0 < tf) bulk_load(smem + D::stage_off, src + (size_t)t0 * TILE, BYTES, bar);
    uint32_t parity = 0;
    T key[ITEMS];
    uint32_t none[1];
    for (uint32_t tile = t0; tile < t1; ++tile) {
        if (tile < tf) {
            if (!mbar_wait(bar, parity, p.spin_limit)) record_error(p.err, RS_ERR_DEVICE_TIMEOUT);
            parity ^= 1u;
#pragma unroll
            for (int k = 0; k < ITEMS; ++k) key[k] = stage[warp * (32 * ITEMS) + k * 32 + lane];
            downsweep_tile<true, KT, RB, THREADS, ITEMS, 0, DYN, true>(p, smem, tile,
                                                                      tile + 1 < tf ? tile + 1 : 0xFFFFFFFFu,
                                                                      running, key, none);
        } else {
            load_tile<KT, RB, THREADS, ITEMS, 0, DYN>(p, smem, tile, key, none);
            downsweep_tile<false, KT, RB, THREADS, ITEMS, 0, DYN>(p, smem, tile, 0xFFFFFFFFu, running, key, none);
        }
    }
}

template <int KT, int RB, int THREADS, int ITEMS, int VB>
__global__ void __launch_bounds__(THREADS, RS_TILE_MIN_THREADS_PER_SM / THREADS) k_downsweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    constexpr int BINS = S::BINS;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);
    RoleShared* rsh = reinterpret_cast<RoleShared*>(smem + S::misc_off + 4);
    const int tid = threadIdx.x;
    const uint32_t g = blockIdx.x;
    zero_counters<S>(smem, THREADS);
    wait_prior_grid();
    // This CTA's digit totals and block offsets are read while thread 0
    // reads the skip record (for a skipped pass they are dropped).
    const uint32_t total = tid < BINS ? p.ghist[tid] : 0u;
    const uint32_t block_off = tid < BINS ? p.counts[(size_t)tid * p.G + g] : 0u;
    if (tid == 0) {
        const PassRole r = decode_plan(load_plan(p));
        publish_role(rsh, r);
        if (r.run && r.E != p.passes) {
            PassParams q = p;
            pass_buffers<VB>(q, r);
            set_pass_io<S>(smem, q);
        }
    }
    // The scan's barriers also publish the role, the PassIO slots and the zeroed counters.
    const uint32_t dstart = bins_exclusive_scan<BINS>(total, sscan, nullptr);
    const PassRole role = read_role(rsh);
    if (!role.run) {
        const size_t lo = (size_t)g * p.tiles_per_cta * S::TILE;
        copy_if_no_pass_runs<T, VB>(p, role, lo, lo + (size_t)p.tiles_per_cta * S::TILE);
        return;
    }
    const uint32_t running = tid < BINS ? dstart + block_off : 0u;
    const bool dyn = role.E != p.passes;  // some pass was skipped: buffers from PassIO
    if constexpr (DownsweepSmem<T, RB, THREADS, ITEMS, VB>::kStaged) {
        using D = DownsweepSmem<T, RB, THREADS, ITEMS, VB>;
        const void* src = dyn ? io_keys_in<S, T>(smem) : p.keys_in;
        if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
            if (tid == 0) mbar_init(reinterpret_cast<uint64_t*>(smem + D::bar_off), 1);
            __syncthreads();
            if (dyn)
                downsweep_loop_staged<KT, RB, THREADS, ITEMS, true>(p, smem, running);
            else
                downsweep_loop_staged<KT, RB, THREADS, ITEMS, false>(p, smem, running);
            return;
        }
    }
    if (!dyn)  // every pass runs: the host's plan holds
        downsweep_loop<KT, RB, THREADS, ITEMS, VB, false>(p, smem, running);
    else
        downsweep_loop<KT, RB, THREADS, ITEMS, VB, true>(p, smem, running);
}

// In place with an odd number of running passes the result ends in the
// partner buffer (see chain_is_out): copy it back to keys_out.
template <int RB, typename T, int VB>
__global__ void __launch_bounds__(256) k_chain_copy(PassParams p)
{
    __shared__ RoleShared rsh;
    wait_prior_grid();
    const PassRole role = block_pass_role(p, &rsh);
    if (p.in_place == 0u || role.E % 2u == 0u) return;
    copy_span<T, VB>(static_cast<const T*>(p.alt_keys), static_cast<T*>(p.sort_keys_out), p.alt_vals,
                       p.sort_vals_out, 0, p.n, (size_t)blockIdx.x * blockDim.x + threadIdx.x,
                       (size_t)gridDim.x * blockDim.x);
}

// ------------------------------------------------------------ small sorts
//
// A sort of at most kClusterMaxCtas tiles runs as ONE kernel on a thread-block
// cluster: CTA c holds positions [c*TILE, (c+1)*TILE) of the current order in
// its shared memory, for every pass.  A pass ranks and shuffles the CTA's tile
// exactly as a chained-scan tile does; the CTAs then exchange their digit
// counts through distributed shared memory -- the start of digit d in CTA c
// is every CTA's count of smaller digits plus CTA 0..c-1's count of d, the
// digit-major exclusive scan ("Radix sort paralelo sobre el scan", section
// "Las tres fases de una pasada") over C blocks -- and every key is stored
// straight into the shared memory of the CTA that owns its new position (the
// last running pass writes keys_out).  Two cluster barriers per pass; global
// memory is read once and written once.

struct ClusterParams {
    const void* keys_in;
    void* keys_out;
    const void* vals_in;
    void* vals_out;
    uint32_t n;
    uint32_t passes;
    uint32_t begin_bit;
    uint32_t end_bit;
    uint32_t* err;
    uint32_t* skip;   // the skip record, for rs_skip_record
    uint32_t descending;
};

template <typename T, int RB, int THREADS, int ITEMS, int VB>
struct ClusterSmem {
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    static constexpr size_t next_keys_off = align_up(S::bytes, 16);  // this CTA's keys of the next pass
    static constexpr size_t next_vals_off = next_keys_off + align_up(sizeof(T) * S::TILE, 16);
    static constexpr size_t cnt_off = next_vals_off + (VB ? align_up(sizeof(ValT<VB>) * (size_t)S::TILE, 16) : 0);
    static constexpr size_t rec_off = cnt_off + 4 * S::BINS;  // this CTA's share of the skip record
    static constexpr size_t plan_off = rec_off + 16;          // run mask, running passes
    static constexpr size_t bytes = plan_off + 16;
};

template <int KT, int RB, int THREADS, int ITEMS, int VB>
__global__ void __launch_bounds__(THREADS, 1) k_cluster_sort(ClusterParams cp)
{
    namespace cg = cooperative_groups;
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    using CS = ClusterSmem<T, RB, THREADS, ITEMS, VB>;
    constexpr int BINS = S::BINS;
    constexpr uint32_t M = S::TILE;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem + S::base_off);
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);
    T* nkeys = reinterpret_cast<T*>(smem + CS::next_keys_off);
    ValT<VB>* nvals = reinterpret_cast<ValT<VB>*>(smem + CS::next_vals_off);
    uint32_t* cnts = reinterpret_cast<uint32_t*>(smem + CS::cnt_off);
    uint32_t* rec = reinterpret_cast<uint32_t*>(smem + CS::rec_off);
    uint32_t* plan = reinterpret_cast<uint32_t*>(smem + CS::plan_off);

    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t c = cluster.block_rank(), C = cluster.num_blocks();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t lo = c * M;
    const uint32_t valid = cp.n > lo ? min(cp.n - lo, M) : 0u;
    const uint32_t seg = (uint32_t)warp * (32u * ITEMS);
    const T* gin = static_cast<const T*>(cp.keys_in);
    PassParams p{};
    p.n = valid;  // the tile code guards positions against its tile's key count
    p.err = cp.err;

    // 1. This CTA's keys, warp-striped (as load_tile), from global memory.
    T key[ITEMS];
    ValT<VB> val[VB ? ITEMS : 1];
    if (valid == M) {
        load_striped<true, T, ITEMS>(gin + lo, seg, valid, lane, key);
        if constexpr (VB != 0)
            load_striped<true, ValT<VB>, ITEMS>(static_cast<const ValT<VB>*>(cp.vals_in) + lo, seg, valid, lane, val);
    } else {
        load_striped<false, T, ITEMS>(gin + lo, seg, valid, lane, key);
        if constexpr (VB != 0)
            load_striped<false, ValT<VB>, ITEMS>(static_cast<const ValT<VB>*>(cp.vals_in) + lo, seg, valid, lane, val);
    }

    // 2. The skip record: each CTA's share of diff and of the order check
    // (pairs inside the tile from registers, across warps and CTAs from
    // global memory), then every CTA combines all shares into the same plan.
    if (tid < 4) rec[tid] = 0u;
    __syncthreads();
    {
        SkipAcc<KT> acc(gin, cp.begin_bit, cp.end_bit, cp.descending != 0u);
        T v[ITEMS];
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
            const uint32_t pos = seg + k * 32 + lane;
            v[k] = pos < valid ? acc.visit(key[k]) : T(0);
        }
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
            const uint32_t pos = seg + k * 32 + lane;
            T nx = __shfl_down_sync(0xFFFFFFFFu, v[k], 1);
            if (k + 1 < ITEMS) {
                const T first_next = __shfl_sync(0xFFFFFFFFu, v[k + 1 < ITEMS ? k + 1 : k], 0);
                if (lane == 31) nx = first_next;
            } else if (lane == 31 && pos + 1 < valid) {
                nx = acc.value(gin[lo + pos + 1]);
            }
            if (pos + 1 < valid) acc.pair(v[k], nx);
        }
        if (tid == 0 && lo > 0 && valid > 0) acc.pair(acc.value(gin[lo - 1]), acc.value(gin[lo]));
        acc.flush_warp(rec);
    }
    __syncthreads();
    cluster.sync();  // every CTA's share is complete
    if (tid == 0) {
        uint32_t d_lo = 0, d_hi = 0, un = 0;
#pragma unroll
        for (uint32_t r = 0; r < (uint32_t)kClusterMaxCtas; ++r) {
            if (r < C) {
                const uint32_t* rr = cluster.map_shared_rank(rec, r);
                d_lo |= rr[0];
                d_hi |= rr[1];
                un |= rr[2];
            }
        }
        uint32_t words[kMaxPasses];
        write_plan<RB>(d_lo, d_hi, un, words, cp.passes, cp.begin_bit, cp.end_bit);
        uint32_t mask = 0;
        for (uint32_t q = 0; q < cp.passes; ++q) mask |= (words[q] & 1u) << q;
        plan[0] = mask;
        plan[1] = cp.passes ? (words[0] >> 16) & 0xFFu : 0u;
        if (c == 0) {
            cp.skip[0] = d_lo;
            cp.skip[1] = d_hi;
            cp.skip[2] = un ? 1u : 0u;
        }
    }
    __syncthreads();
    const uint32_t run_mask = plan[0], E = plan[1];
    // A CTA's shared memory must not be read after it exits: with no pass to
    // run, wait here until every CTA has read the others' shares (otherwise
    // the first pass's barrier does).
    if (E == 0u) cluster.sync();

    // 3. The running passes.
    uint32_t j = 0;
    for (uint32_t q = 0; q < cp.passes; ++q) {
        if (!((run_mask >> q) & 1u)) continue;
        if (j > 0) {  // this CTA's keys of this pass, left by the previous one
            if (valid == M) {
                load_striped<true, T, ITEMS>(nkeys, seg, valid, lane, key);
                if constexpr (VB != 0) load_striped<true, ValT<VB>, ITEMS>(nvals, seg, valid, lane, val);
            } else {
                load_striped<false, T, ITEMS>(nkeys, seg, valid, lane, key);
                if constexpr (VB != 0) load_striped<false, ValT<VB>, ITEMS>(nvals, seg, valid, lane, val);
            }
        }
        p.shift = cp.begin_bit + q * RB;
        p.mask = (1u << min((uint32_t)RB, cp.end_bit - p.shift)) - 1u;
        p.flip = cp.descending ? p.mask : 0u;
        zero_counters<S>(smem, THREADS);
        __syncthreads();
        uint32_t cnt, start;
        if (valid == M)
            tile_rank_and_shuffle<true, KT, RB, THREADS, ITEMS, VB>(p, smem, 0, key, val, &cnt, &start,
                                                                      [](int, uint32_t) {});
        else
            tile_rank_and_shuffle<false, KT, RB, THREADS, ITEMS, VB>(p, smem, 0, key, val, &cnt, &start,
                                                                       [](int, uint32_t) {});
        if (tid < BINS) cnts[tid] = cnt;
        // Counts published; every CTA has also read its keys of this pass, so
        // the next-pass buffers may be written from here on.
        cluster.sync();
        uint32_t tot = 0, before = 0;
        if (tid < BINS) {
            // All C remote reads are issued before any is summed (unrolled to
            // the largest cluster), so they cost one round trip, not C.
            uint32_t x[kClusterMaxCtas];
#pragma unroll
            for (uint32_t r = 0; r < (uint32_t)kClusterMaxCtas; ++r)
                x[r] = r < C ? *cluster.map_shared_rank(cnts + tid, r) : 0u;
#pragma unroll
            for (uint32_t r = 0; r < (uint32_t)kClusterMaxCtas; ++r) {
                tot += x[r];
                before += r < c ? x[r] : 0u;
            }
        }
        const uint32_t dstart = bins_exclusive_scan<BINS>(tid < BINS ? tot : 0u, sscan, nullptr);
        if (tid < BINS) sbase[tid] = dstart + before - start;
        __syncthreads();
        const bool last = j + 1 == E;
        T* gout = static_cast<T*>(cp.keys_out);
        uint32_t bad = 0;
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
            const uint32_t s = (uint32_t)(k * THREADS) + tid;
            if (s < valid) {
                T kk;
                ValT<VB> vv;
                slot_get<S, T, VB>(smem, s, kk, vv);
                const uint32_t g = sbase[digit_of<KT>(kk, p.shift, p.mask, p.flip)] + s;
                if (g >= cp.n) {
                    bad = 1;
                    continue;
                }
                if (last) {
                    gout[g] = kk;
                    if constexpr (VB != 0) static_cast<ValT<VB>*>(cp.vals_out)[g] = vv;
                } else {
                    const uint32_t dst = g / M, off = g - dst * M;
                    *cluster.map_shared_rank(nkeys + off, dst) = kk;
                    if constexpr (VB != 0) *cluster.map_shared_rank(nvals + off, dst) = vv;
                }
            }
        }
        if (bad) record_error(cp.err, RS_ERR_CHECK_FAILED);
        cluster.sync();  // the next pass's keys are in place; cnts may be reused
        ++j;
    }
    // No pass runs: the input is the result.
    if (E == 0u && cp.keys_in != cp.keys_out)
        copy_span<T, VB>(gin, static_cast<T*>(cp.keys_out), cp.vals_in, cp.vals_out, lo, lo + valid, tid,
                           THREADS);
}

// Chained scan, the one upfront read: the digit histograms of ALL passes,
// accumulated in shared memory and added to the global ones; the same kernel
// zeroes the look-back status words of every pass.
struct HistParams {
    const void* keys;
    uint32_t n;
    uint32_t begin_bit;
    uint32_t end_bit;
    uint32_t passes;
    uint32_t* ghist;        // [passes][BINS]
    uint4* zero;            // status region to clear
    size_t zero_vec4;       // its size in 16-byte words
    int aligned16;          // keys pointer is 16-byte aligned
    uint32_t* skip;         // the pass-skip record
    uint32_t* plan;         // the pass plan
    uint32_t descending;
};

// Counters are lane-private columns, hist[pass][bin][col] with col = lane %
// COLS, so the COLS lanes of a warp that share no column hit distinct banks:
// the shared atomics of one warp instruction do not conflict (the warps of
// the CTA still share the columns, which the atomics make safe).
// BYTES: every pass's digit is one whole byte of the ordered key (8-bit
// digits over the full key, ascending), so all MAXP passes run, each digit is
// one byte permute and each counter address a constant offset from the
// byte's: the kernel is issue-bound, and this halves its instructions.
template <int KT, int RB, int THREADS, int COLS, bool FULLRANGE, bool BYTES = false>
__global__ void __launch_bounds__(THREADS) k_histogram(HistParams h)
{
    using T = typename KeyOps<KT>::T;
    constexpr int BINS = 1 << RB;
    constexpr int VEC = 16 / sizeof(T);
    constexpr int U = 4;  // vectors in flight per thread
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem);
    __shared__ uint32_t skip_blk[3];
    const int tid = threadIdx.x;
    const uint32_t col = tid % COLS;
    const uint32_t words = h.passes * BINS * COLS;
    for (uint32_t i = tid; i < words; i += THREADS) hist[i] = 0;
    if (tid < 3) skip_blk[tid] = 0;
    __syncthreads();

    // Each pass's shift, digit mask and flip, worked out once; the key loop
    // below is unrolled over the most passes this key type can have.
    constexpr int MAXP = (8 * (int)sizeof(T) + RB - 1) / RB;
    uint32_t sh[MAXP], mk[MAXP], fl[MAXP];
#pragma unroll
    for (int q = 0; q < MAXP; ++q) {
        sh[q] = min(h.begin_bit + q * RB, 8u * (uint32_t)sizeof(T) - 1u);
        const uint32_t width = (uint32_t)q < h.passes ? min((uint32_t)RB, h.end_bit - sh[q]) : 0u;
        mk[q] = (1u << width) - 1u;
        fl[q] = h.descending ? mk[q] : 0u;
    }
    static_assert(!BYTES || (RB == 8 && FULLRANGE), "byte digits need 8-bit digits over the whole key");
    uint32_t* const hcol = hist + col;
    auto count = [&](T k) {
        const auto o = KeyOps<KT>::ordered(k);
        if constexpr (BYTES) {
#pragma unroll
            for (int q = 0; q < MAXP; ++q) {
                const uint32_t word = (uint32_t)((uint64_t)o >> (32 * (q / 4)));
                const uint32_t d = __byte_perm(word, 0u, 0x4440u | (uint32_t)(q & 3));
                atomicAdd(hcol + (q * BINS) * COLS + d * COLS, 1u);
            }
        } else {
#pragma unroll
            for (int q = 0; q < MAXP; ++q) {
                if ((uint32_t)q < h.passes) {
                    const uint32_t d = ((uint32_t)(o >> sh[q]) & mk[q]) ^ fl[q];
                    atomicAdd(hist + (q * BINS + d) * COLS + col, 1u);
                }
            }
        }
    };

    const size_t gthreads = (size_t)gridDim.x * THREADS;
    const size_t gid = (size_t)blockIdx.x * THREADS + tid;
    const int lane = tid & 31;
    const T* keys = static_cast<const T*>(h.keys);
    SkipAcc<KT, !FULLRANGE> acc(keys, h.begin_bit, h.end_bit, h.descending != 0u);
    size_t done = 0;
    if (h.aligned16) {
        const size_t nvec = h.n / VEC;
        const uint4* kv = reinterpret_cast<const uint4*>(keys);
        // Full rounds (U vectors per thread, the same trip count everywhere),
        // then what is left.  Thread gid + 1 holds the vector after thread
        // gid's, so a shuffle brings the next key for the order check.
        const size_t per_round = U * gthreads, rounds = nvec / per_round;
        for (size_t r = 0; r < rounds; ++r) {
            uint4 w[U];
            T nb[U];  // lane 31: the key after its vector, loaded with the round
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t v = r * per_round + u * gthreads + gid;
                w[u] = __ldcs(kv + v);
                nb[u] = (lane == 31 && v + 1 < nvec) ? keys[(v + 1) * VEC] : T(0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                T k[VEC];
                memcpy(k, &w[u], 16);
#pragma unroll
                for (int j = 0; j < VEC; ++j) count(k[j]);
                const size_t v = r * per_round + u * gthreads + gid;
                T first, last;
                acc.vector(k, first, last);
                T next = __shfl_down_sync(0xFFFFFFFFu, first, 1);
                if (lane == 31) next = v + 1 < nvec ? acc.value(nb[u]) : last;
                acc.pair(last, next);
            }
        }
        for (size_t v = rounds * per_round + gid; v < nvec; v += gthreads) {
            const uint4 w = __ldcs(kv + v);
            T k[VEC];
            memcpy(k, &w, 16);
#pragma unroll
            for (int j = 0; j < VEC; ++j) count(k[j]);
            T first, last;
            acc.vector(k, first, last);
            if (v + 1 < nvec) acc.pair(last, acc.value(keys[(v + 1) * VEC]));
        }
        done = nvec * VEC;
    }
    for (size_t i = done + gid; i < h.n; i += gthreads) {
        const T k = keys[i];
        count(k);
        const T v = acc.visit(k);
        if (i > 0) acc.pair(acc.value(keys[i - 1]), v);
    }
    acc.flush_warp(skip_blk);
    __syncthreads();
    SkipAcc<KT, !FULLRANGE>::template flush_block<RB>(skip_blk, h.skip, h.plan, h.passes, h.begin_bit, h.end_bit);
    for (uint32_t i = tid; i < h.passes * BINS; i += THREADS) {
        uint32_t c = 0;
#pragma unroll 8
        for (int j = 0; j < COLS; ++j) c += hist[i * COLS + ((j + i) % COLS)];
        if (c) atomicAdd(&h.ghist[i], c);
    }
    for (size_t i = gid; i < h.zero_vec4; i += gthreads) h.zero[i] = make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------- host driver

// Everything run_sort needs, resolved from the public descriptor.
struct Plan {
    int kt;
    bool vals;
    int vb;           // value bytes: 0, 4 or 8
    size_t n;
    int begin_bit, end_bit;
    int algo;         // RS_ALGO_ONESWEEP or RS_ALGO_REDUCE_SCAN (resolved)
    int radix_bits;   // 4 or 8
    bool descending;
    int passes;
    const void* keys_in;
    void* keys_out;
    const void* vals_in;
    void* vals_out;
    unsigned char* temp;
    TempLayout lay;
    cudaStream_t stream;
    uint32_t spin_limit;
    int32_t stall_tile;
    // profiling (optional)
    cudaEvent_t const* events;
    unsigned event_flags;  // cudaEventRecordExternal while the stream is being captured
    int max_events;
    int launched;
    int* kinds;
    bool count_only;   // only count kernels, launch nothing
    bool auto_chosen;  // the schedule came from RS_ALGO_AUTO
    bool launch_failed = false;
};

enum KernelKind { kKindHistogram = 1, kKindOnesweep = 2, kKindUpsweep = 3, kKindSpine = 4,
                  kKindDownsweep = 5, kKindCopy = 6, kKindCluster = 7 };

// After every launch: check it, and record the next profiling event.
inline rs_status after_launch(Plan& pl, int kind)
{
    if (pl.count_only) { pl.launched++; return RS_OK; }
    if (cudaGetLastError() != cudaSuccess || pl.launch_failed) return RS_ERR_CUDA;
    if (pl.kinds && pl.launched < pl.max_events) pl.kinds[pl.launched] = kind;
    pl.launched++;
    if (pl.events && pl.launched < pl.max_events)
        if (cudaEventRecordWithFlags(pl.events[pl.launched], pl.stream, pl.event_flags) != cudaSuccess)
            return RS_ERR_CUDA;
    return RS_OK;
}

// Launch `kernel` on the plan's stream (nothing when only counting).  With
// `dependent`, as a programmatic dependent of the kernel before it in the
// stream (see wait_prior_grid); the first kernel of a sort is launched
// plainly, so it waits for everything the caller enqueued before the sort.
template <typename... KArgs, typename... Args>
inline void launch(Plan& pl, bool dependent, void (*kernel)(KArgs...), unsigned grid, unsigned block,
                   size_t smem, Args... args)
{
    if (pl.count_only) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = pl.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) pl.launch_failed = true;
}

inline int device_sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = v;
    }
    return cache[dev];
}

// Opt a kernel into more than 48 KB of dynamic shared memory (a host-side
// function attribute of the current device; not a stream operation).
template <typename K>
inline bool set_smem(K kernel, size_t bytes)
{
    if (bytes <= 48 * 1024) return true;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
}

// The byte-digit twin of a 32-bit key type (the type itself otherwise).
template <int KT> struct ByteTwin { static constexpr int value = KT; };
template <> struct ByteTwin<KU32> { static constexpr int value = KU32B; };
template <> struct ByteTwin<KI32> { static constexpr int value = KI32B; };
template <> struct ByteTwin<KF32> { static constexpr int value = KF32B; };
template <> struct ByteTwin<KU16> { static constexpr int value = KU16B; };
template <> struct ByteTwin<KI16> { static constexpr int value = KI16B; };
template <> struct ByteTwin<KF16> { static constexpr int value = KF16B; };

template <int KT, int RB, int VB>
rs_status run_passes(Plan& pl)
{
    using T = typename KeyOps<KT>::T;
    constexpr int KB = sizeof(T);
    constexpr int ITEMS = tile_items(KB, VB);
    constexpr int BINS = 1 << RB;
    const uint32_t n = (uint32_t)pl.n;
    uint32_t* meta = reinterpret_cast<uint32_t*>(pl.temp + pl.lay.meta);
    uint32_t* big = reinterpret_cast<uint32_t*>(pl.temp + pl.lay.big);
    T* alt_keys = reinterpret_cast<T*>(pl.temp + pl.lay.alt_keys);
    void* alt_vals = pl.temp + pl.lay.alt_vals;
    const int P = pl.passes;

    // The host plans each pass's buffers for the case where every pass runs
    // (chain_is_out with E = P); a pass kernel that finds some pass skipped
    // works out its own from the sort-level buffers (pass_buffers).
    const bool in_place = pl.keys_in == pl.keys_out;
    PassParams base{};
    base.sort_keys_in = pl.keys_in;
    base.sort_keys_out = pl.keys_out;
    base.sort_vals_in = (VB != 0) ? pl.vals_in : nullptr;
    base.sort_vals_out = (VB != 0) ? pl.vals_out : nullptr;
    base.alt_keys = alt_keys;
    base.alt_vals = (VB != 0) ? alt_vals : nullptr;
    base.skip = meta + kSkipBase;
    base.plan = meta + kPlanBase;
    base.passes = (uint32_t)P;
    base.begin_bit = (uint32_t)pl.begin_bit;
    base.end_bit = (uint32_t)pl.end_bit;
    base.in_place = in_place ? 1u : 0u;
    base.descending = pl.descending ? 1u : 0u;
    base.n = n;
    base.err = meta + kErrWord;
    base.spin_limit = pl.spin_limit;
    base.stall_tile = pl.stall_tile;
    const int sms = pl.count_only ? 1 : device_sm_count();

    auto plan_buffers = [&](PassParams& pp, int q) {
        const uint32_t E = (uint32_t)P, j = (uint32_t)q;
        const bool src_out = chain_is_out(j, E, in_place), dst_out = chain_is_out(j + 1, E, in_place);
        pp.keys_in = j == 0 ? pl.keys_in : (src_out ? pl.keys_out : static_cast<const void*>(alt_keys));
        pp.keys_out = dst_out ? pl.keys_out : static_cast<void*>(alt_keys);
        if (VB != 0) {
            pp.vals_in = j == 0 ? pl.vals_in : (src_out ? static_cast<const void*>(pl.vals_out) : alt_vals);
            pp.vals_out = dst_out ? pl.vals_out : alt_vals;
        }
    };

    // In place, a final copy (k_chain_copy) runs when an odd number of passes ran.
    auto finish = [&]() -> rs_status {
        if (!in_place) return RS_OK;
        launch(pl, true, k_chain_copy<RB, T, VB>, 4 * sms, 256, 0, base);
        return after_launch(pl, kKindCopy);
    };

    // The chained scan on tiles of THREADS x ITEMS keys (threads_c carries
    // THREADS: onesweep_threads() picks it from n).
    auto run_onesweep = [&](auto threads_c) -> rs_status {
        constexpr int THREADS = decltype(threads_c)::value;
        constexpr int TILE = THREADS * ITEMS;
        using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
        const uint32_t num_tiles = (n + TILE - 1) / TILE;
        base.num_tiles = num_tiles;
        constexpr int MAXP = (8 * KB + RB - 1) / RB;
        constexpr int HCOLS = (MAXP * (1 << RB) * 32 * 4 <= 160 * 1024) ? 32 : 16;
        const bool full_range = pl.begin_bit == 0 && pl.end_bit == 8 * KB;
        auto hk = !full_range                    ? k_histogram<KT, RB, 1024, HCOLS, false>
                  : (RB == 8 && !pl.descending) ? k_histogram<KT, RB, 1024, HCOLS, true, RB == 8>
                                                : k_histogram<KT, RB, 1024, HCOLS, true>;
        auto pk = k_onesweep<KT, RB, THREADS, ITEMS, VB>;
        auto pkb = k_onesweep<ByteTwin<KT>::value, RB, THREADS, ITEMS, VB>;
        if (!pl.count_only && (!set_smem(pk, S::bytes) || !set_smem(pkb, S::bytes))) return RS_ERR_CUDA;
        const size_t status_words = (size_t)P * num_tiles * BINS;
        HistParams h{};
        h.keys = pl.keys_in;
        h.n = n;
        h.begin_bit = pl.begin_bit;
        h.end_bit = pl.end_bit;
        h.passes = P;
        h.ghist = meta + kGhistBase;
        h.zero = reinterpret_cast<uint4*>(big);
        h.zero_vec4 = status_words / 4;
        h.aligned16 = (reinterpret_cast<uintptr_t>(pl.keys_in) % 16) == 0;
        h.descending = pl.descending ? 1u : 0u;
        h.skip = meta + kSkipBase;
        h.plan = meta + kPlanBase;
        const size_t want = (n + 1024 * 16 - 1) / (1024 * 16);
        const int hgrid = (int)std::max<size_t>(1, std::min<size_t>(want, (size_t)sms));
        const size_t hsmem = (size_t)P * BINS * HCOLS * 4;
        if (!pl.count_only && !set_smem(hk, hsmem)) return RS_ERR_CUDA;
        launch(pl, false, hk, hgrid, 1024, hsmem, h);
        rs_status st = after_launch(pl, kKindHistogram);
        if (st != RS_OK) return st;
        for (int q = 0; q < P; ++q) {
            PassParams pp = base;
            pp.pass = (uint32_t)q;
            plan_buffers(pp, q);
            pp.shift = pl.begin_bit + q * RB;
            const uint32_t width = std::min(RB, pl.end_bit - (int)pp.shift);
            pp.mask = (1u << width) - 1u;
            pp.flip = pl.descending ? pp.mask : 0u;
            pp.status = big + (size_t)q * num_tiles * BINS;
            pp.ghist = meta + kGhistBase + q * BINS;
            pp.ticket = meta + kTicketBase + q;
            const bool byte_digit = (RB == 8) && (pp.shift % 8 == 0) && (pp.mask == 0xFFu) && !pl.descending;
            launch(pl, true, byte_digit ? pkb : pk, num_tiles, THREADS, S::bytes, pp);
            st = after_launch(pl, kKindOnesweep);
            if (st != RS_OK) return st;
        }
        return finish();
    };
    if (pl.algo == RS_ALGO_ONESWEEP) {
        if constexpr (RB == 8) {
            if (onesweep_threads(n, KB, VB, RB) == RS_OS_THREADS_SMALL)
                return run_onesweep(std::integral_constant<int, RS_OS_THREADS_SMALL>{});
        }
        return run_onesweep(std::integral_constant<int, RS_OS_THREADS>{});
    }

    // Reduce-then-scan.
    constexpr int THREADS = tile_threads(kAlgoReduceScan, KB, VB);
    constexpr int TILE = THREADS * ITEMS;
    using S = TileSmem<T, RB, THREADS, ITEMS, VB>;
    const uint32_t num_tiles = (n + TILE - 1) / TILE;
    base.num_tiles = num_tiles;
    const bool full_range = pl.begin_bit == 0 && pl.end_bit == 8 * KB;
    auto uk0 = full_range ? k_upsweep<KT, RB, 512, TILE, true, true> : k_upsweep<KT, RB, 512, TILE, true, false>;
    auto uk = k_upsweep<KT, RB, 512, TILE, false>;
    auto dk = k_downsweep<KT, RB, THREADS, ITEMS, VB>;
    auto dkb = k_downsweep<ByteTwin<KT>::value, RB, THREADS, ITEMS, VB>;
    constexpr size_t DSMEM = DownsweepSmem<T, RB, THREADS, ITEMS, VB>::bytes;
    if (!pl.count_only && (!set_smem(dk, DSMEM) || !set_smem(dkb, DSMEM))) return RS_ERR_CUDA;
    uint32_t G = 1;
    if (!pl.count_only) {
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dk, THREADS, DSMEM) != cudaSuccess || occ < 1)
            occ = 1;
        G = (uint32_t)std::min<size_t>((size_t)sms * occ, (size_t)kRtsMaxCtas);
    }
    G = std::max<uint32_t>(1, std::min<uint32_t>(G, num_tiles));
    const uint32_t tpc = (num_tiles + G - 1) / G;
    G = (num_tiles + tpc - 1) / tpc;
    for (int q = 0; q < P; ++q) {
        PassParams pp = base;
        pp.pass = (uint32_t)q;
        plan_buffers(pp, q);
        pp.shift = pl.begin_bit + q * RB;
        const uint32_t width = std::min(RB, pl.end_bit - (int)pp.shift);
        pp.mask = (1u << width) - 1u;
        pp.flip = pl.descending ? pp.mask : 0u;
        pp.counts = big;
        pp.G = G;
        pp.tiles_per_cta = tpc;
        launch(pl, q != 0, q == 0 ? uk0 : uk, G, 512, 0, pp);
        rs_status st = after_launch(pl, kKindUpsweep);
        if (st != RS_OK) return st;
        pp.ghist = meta + kGhistBase + q * BINS;  // row totals of this pass
        launch(pl, true, k_spine_scan<RB, 256>, BINS, 256, 0, pp, meta + kGhistBase + q * BINS);
        st = after_launch(pl, kKindSpine);
        if (st != RS_OK) return st;
        const bool byte_digit = (RB == 8) && (pp.shift % 8 == 0) && (pp.mask == 0xFFu) && !pl.descending;
        launch(pl, true, byte_digit ? dkb : dk, G, THREADS, DSMEM, pp);
        st = after_launch(pl, kKindDownsweep);
        if (st != RS_OK) return st;
    }
    return finish();
}

// The largest cluster of k_cluster_sort<...> the current device schedules
// (queried once per device; kClusterMaxCtas when no device is visible, as
// when only counting kernels on a machine without a GPU).
template <typename K>
inline unsigned max_cluster_ctas(K kernel, int threads, size_t smem_bytes)
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return kClusterMaxCtas;
    }
    if (cache[dev] == 0) {
        int size = 0;
        if (!set_smem(kernel, smem_bytes) ||
            cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            cudaGetLastError();
            size = 1;
        } else {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(kClusterMaxCtas, 1, 1);
            cfg.blockDim = dim3(threads, 1, 1);
            cfg.dynamicSmemBytes = smem_bytes;
            if (cudaOccupancyMaxPotentialClusterSize(&size, kernel, &cfg) != cudaSuccess || size < 1) {
                cudaGetLastError();
                size = 1;
            }
        }
        cache[dev] = std::min(size, kClusterMaxCtas);
    }
    return (unsigned)cache[dev];
}

// CTAs the cluster sort of n keys needs, or 0 if this device cannot run it.
template <int KT, int RB, int VB>
unsigned cluster_ctas_for(size_t n)
{
    using T = typename KeyOps<KT>::T;
    constexpr int KB = sizeof(T);
    constexpr int ITEMS = cluster_items(KB, VB);
    using CS = ClusterSmem<T, RB, kClusterThreads, ITEMS, VB>;
    const size_t tile = cluster_tile_keys(KB, VB);
    const size_t ctas = (n + tile - 1) / tile;
    if (ctas < 1 || ctas > (size_t)kClusterMaxCtas) return 0;
    if (ctas <= 8) return (unsigned)ctas;  // the portable size always schedules
    const unsigned cap = max_cluster_ctas(k_cluster_sort<KT, RB, kClusterThreads, ITEMS, VB>,
                                          kClusterThreads, CS::bytes);
    return ctas <= cap ? (unsigned)ctas : 0u;
}

// The whole sort as one launch on a cluster of ceil(n / tile) CTAs.
template <int KT, int RB, int VB>
rs_status run_cluster(Plan& pl)
{
    using T = typename KeyOps<KT>::T;
    constexpr int KB = sizeof(T);
    constexpr int ITEMS = cluster_items(KB, VB);
    constexpr int THREADS = kClusterThreads;
    using CS = ClusterSmem<T, RB, THREADS, ITEMS, VB>;
    const unsigned ctas = cluster_ctas_for<KT, RB, VB>(pl.n);
    if (ctas == 0) return RS_ERR_UNSUPPORTED;
    if (pl.count_only) return after_launch(pl, kKindCluster);
    auto kernel = k_cluster_sort<KT, RB, THREADS, ITEMS, VB>;
    if (!set_smem(kernel, CS::bytes)) return RS_ERR_CUDA;
    if (ctas > 8 && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return RS_ERR_CUDA;
    uint32_t* meta = reinterpret_cast<uint32_t*>(pl.temp + pl.lay.meta);
    ClusterParams cp{};
    cp.keys_in = pl.keys_in;
    cp.keys_out = pl.keys_out;
    cp.vals_in = (VB != 0) ? pl.vals_in : nullptr;
    cp.vals_out = (VB != 0) ? pl.vals_out : nullptr;
    cp.n = (uint32_t)pl.n;
    cp.passes = (uint32_t)pl.passes;
    cp.begin_bit = (uint32_t)pl.begin_bit;
    cp.end_bit = (uint32_t)pl.end_bit;
    cp.descending = pl.descending ? 1u : 0u;
    cp.err = meta + kErrWord;
    cp.skip = meta + kSkipBase;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = CS::bytes;
    cfg.stream = pl.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, cp) != cudaSuccess) return RS_ERR_CUDA;
    return after_launch(pl, kKindCluster);
}

// The instantiation for this request's digit width and value bytes.
template <int KT, int VB>
rs_status run_sort_vb(Plan& pl)
{
    if (pl.algo == RS_ALGO_CLUSTER) {
        const unsigned ctas = pl.radix_bits == 4 ? cluster_ctas_for<KT, 4, VB>(pl.n)
                                                 : cluster_ctas_for<KT, 8, VB>(pl.n);
        if (ctas == 0 && pl.auto_chosen) {
            pl.algo = RS_ALGO_ONESWEEP;  // this device cannot schedule the cluster
        } else {
            return pl.radix_bits == 4 ? run_cluster<KT, 4, VB>(pl) : run_cluster<KT, 8, VB>(pl);
        }
    }
    return pl.radix_bits == 4 ? run_passes<KT, 4, VB>(pl) : run_passes<KT, 8, VB>(pl);
}

template <int KT>
rs_status run_sort(Plan& pl)
{
    switch (pl.vb) {
    case 0: return run_sort_vb<KT, 0>(pl);
    case 8: return run_sort_vb<KT, 8>(pl);
    default: return run_sort_vb<KT, 4>(pl);
    }
}

}  // namespace rs
