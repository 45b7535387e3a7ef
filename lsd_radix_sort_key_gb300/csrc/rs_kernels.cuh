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
// Two schedules are built from the same tile code:
//   * chained scan (k_histogram once, then k_onesweep per pass): every tile
//     takes a ticket, publishes its digit counts, and looks back over its
//     predecessors' published counts for its global offsets (decoupled
//     look-back; Merrill & Garland 2016, Adinets & Merrill 2022).  Step 2 thus
//     runs inside the pass kernel and the keys are read once per pass, plus
//     once up front for all histograms.
//   * reduce-then-scan (k_upsweep, k_spine_scan, k_downsweep per pass): each
//     CTA owns a contiguous chunk of tiles; the spine scan is step 2 proper.
//
// Keys are carried with their original bit patterns.  The order-preserving
// map T (identity, sign flip for int32, the NaN/Inf-aware flip for float32)
// is applied when a digit is extracted, in every pass -- as the CPU code of
// "Radix sort を実装 & 測定してみた" (section 実装) does -- so no inverse map
// is needed and NaN/Inf payloads come back unchanged.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>

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
#ifndef RS_BALLOT_XOR
#define RS_BALLOT_XOR 1
#endif
#ifndef RS_LOOKBACK_BATCH
#define RS_LOOKBACK_BATCH 4
#endif
#ifndef RS_TILE_MIN_THREADS_PER_SM
#define RS_TILE_MIN_THREADS_PER_SM 1024
#endif
//   RS_CHAINS       each warp's segment is split into this many contiguous
//                   parts with separate digit counters ("virtual warps"),
//                   ranked interleaved: independent dependency chains.
#ifndef RS_CHAINS
#define RS_CHAINS 1
#endif
//   RS_RANK_ATOMIC  1: one leader lane per digit advances the counter with a
//                   shared atomic and hands the old count to its peers with a
//                   shuffle; 0: every lane reads the counter and the peers
//                   store the advanced count.
#ifndef RS_RANK_ATOMIC
#define RS_RANK_ATOMIC 0
#endif
//   RS_LOAD_STREAM  1: tile loads are streaming (evict-first) loads.
//   RS_STORE_KEEP   1: scatter stores carry an L2 evict-last policy, so lines
//                   that a digit run leaves half written stay resident until
//                   the next tile completes them.
#ifndef RS_LOAD_STREAM
#define RS_LOAD_STREAM 0
#endif
#ifndef RS_STORE_KEEP
#define RS_STORE_KEEP 1
#endif
//   RS_OS_PERSISTENT   1: chained-scan CTAs loop over tiles and prefetch the
//                   next one; 0: one tile per CTA.
#ifndef RS_OS_PERSISTENT
#define RS_OS_PERSISTENT 0
#endif

namespace rs {

enum : int { KU32 = 0, KI32 = 1, KF32 = 2, KU64 = 3 };
// The same 32-bit key types, for passes whose digit is one whole byte of the
// ordered key: the digit is then one byte permute instead of a shift and a mask.
enum : int { KU32B = 4, KI32B = 5, KF32B = 6 };

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

template <> struct KeyOps<KU32B> : KeyOps<KU32> { static constexpr bool kByte = true; };
template <> struct KeyOps<KI32B> : KeyOps<KI32> { static constexpr bool kByte = true; };
template <> struct KeyOps<KF32B> : KeyOps<KF32> { static constexpr bool kByte = true; };

template <int KT, typename = void> struct IsByte { static constexpr bool value = false; };
template <int KT> struct IsByte<KT, decltype((void)KeyOps<KT>::kByte)> { static constexpr bool value = true; };

template <int KT>
__device__ __forceinline__ uint32_t digit_of(typename KeyOps<KT>::T u, uint32_t shift, uint32_t mask)
{
    if constexpr (IsByte<KT>::value)  // byte (shift / 8) moved to the low byte, zeros above
        return __byte_perm((uint32_t)KeyOps<KT>::ordered(u), 0u, 0x4440u | (shift >> 3));
    else
        return (uint32_t)(KeyOps<KT>::ordered(u) >> shift) & mask;
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
    else
        asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(addr), "r"(v), "l"(pol) : "memory");
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
    const void* keys_in;
    void* keys_out;
    const uint32_t* vals_in;
    uint32_t* vals_out;
    uint32_t n;
    uint32_t shift;          // lowest bit of this pass's digit in the ordered key
    uint32_t mask;           // digit mask (fewer bits on a final partial digit)
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
template <typename T, int RB, int THREADS, int ITEMS, bool VALS>
struct TileSmem {
    static constexpr int BINS = 1 << RB;
    static constexpr int WARPS = THREADS / 32;
    static constexpr int CHAINS = (ITEMS % RS_CHAINS == 0) ? RS_CHAINS : 1;
    static constexpr int VWARPS = WARPS * CHAINS;  // counter arrays ("virtual warps")
    static constexpr int TILE = THREADS * ITEMS;
    static constexpr int WH = BINS + 1;  // per-array counters + one dummy slot for tail lanes
    static constexpr size_t keys_off = 0;
    static constexpr size_t vals_off = align_up(sizeof(T) * TILE, 16);
    static constexpr size_t wh_off = vals_off + (VALS ? align_up(4 * (size_t)TILE, 16) : 0);
    static constexpr size_t base_off = wh_off + align_up(4 * (size_t)VWARPS * WH, 16);
    static constexpr size_t scan_off = base_off + 4 * BINS;
    static constexpr size_t misc_off = scan_off + 4 * 32;
    static constexpr size_t bytes = misc_off + 16;
};

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
#if RS_LOAD_STREAM
        if (FULL) v[k] = __ldcs(src + i);
        else v[k] = i < n ? __ldcs(src + i) : T(0);
#else
        if (FULL) v[k] = src[i];
        else v[k] = i < n ? src[i] : T(0);
#endif
    }
}

// Keys (and values) of one tile in warp-striped order; a tile that runs past
// n is guarded lane by lane.
template <int KT, int THREADS, int ITEMS, bool VALS>
__device__ __forceinline__ void load_tile(const PassParams& p, uint32_t tile,
                                          typename KeyOps<KT>::T (&key)[ITEMS],
                                          uint32_t (&val)[VALS ? ITEMS : 1])
{
    using T = typename KeyOps<KT>::T;
    constexpr uint32_t TILE = THREADS * ITEMS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t seg = tile * TILE + (uint32_t)warp * (32u * ITEMS);
    if ((tile + 1) * TILE <= p.n) {
        load_striped<true, T, ITEMS>(static_cast<const T*>(p.keys_in), seg, p.n, lane, key);
        if constexpr (VALS) load_striped<true, uint32_t, ITEMS>(p.vals_in, seg, p.n, lane, val);
    } else {
        load_striped<false, T, ITEMS>(static_cast<const T*>(p.keys_in), seg, p.n, lane, key);
        if constexpr (VALS) load_striped<false, uint32_t, ITEMS>(p.vals_in, seg, p.n, lane, val);
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
#if RS_BALLOT_XOR
        peers &= bal ^ (bit - 1u);  // bit - 1 is all ones exactly when the bit is clear
#else
        peers &= bit ? bal : ~bal;
#endif
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
                                               uint32_t n, uint32_t shift, uint32_t mask, int lane)
{
    const uint32_t d = digit_of<KT>(key[k], shift, mask);
    return (FULL || seg + k * 32 + lane < n) ? d : (1u << RB);
}

template <bool FULL, int KT, int RB, int ITEMS, int CHAINS, int WH>
__device__ __forceinline__ void rank_in_warp(const typename KeyOps<KT>::T (&key)[ITEMS], uint32_t seg,
                                             uint32_t n, uint32_t shift, uint32_t mask, uint32_t* wh,
                                             int lane, uint32_t (&rank)[(ITEMS + 1) / 2])
{
    // Part c holds steps [c*L, (c+1)*L) and counts into wh + c*WH; the parts
    // are visited interleaved (j-th step of every part, then the next j).
    constexpr int L = ITEMS / CHAINS;
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < (ITEMS + 1) / 2; ++i) rank[i] = 0;
#pragma unroll
    for (int j = 0; j < L; ++j) {
#pragma unroll
        for (int c = 0; c < CHAINS; ++c) {
            const int k = c * L + j;
            uint32_t* cnt = wh + c * WH;
            const uint32_t d = step_digit<FULL, KT, RB, ITEMS>(key, k, seg, n, shift, mask, lane);
            const uint32_t peers = warp_peers<FULL ? RB : RB + 1, RB>(d);
#if RS_RANK_ATOMIC
            const int leader = 31 - __clz(peers);
            uint32_t old = 0;
            if (leader == lane) old = atomicAdd(cnt + d, (uint32_t)__popc(peers));
            const uint32_t prior = __shfl_sync(0xFFFFFFFFu, old, leader);
#else
            const uint32_t prior = cnt[d];
            cnt[d] = prior + __popc(peers);
#endif
            const uint32_t r = prior + __popc(peers & lt);
            rank[k / 2] |= (k & 1) ? (r << 16) : r;
        }
        __syncwarp();
    }
}

// Zero the tile's digit counters (the caller synchronises before ranking).
template <typename S>
__device__ __forceinline__ void zero_counters(unsigned char* smem, int threads)
{
    uint32_t* whist = reinterpret_cast<uint32_t*>(smem + S::wh_off);
    for (int i = threadIdx.x; i < S::VWARPS * S::WH; i += threads) whist[i] = 0;
}

// Everything of one tile, whose keys are in registers, up to the point where
// its global digit offsets are needed: rank, per-digit counts, tile-local
// digit starts, shuffle into shared memory.  Returns, for thread d < BINS,
// the tile's count of digit d in *cnt and its tile-local start in *start.
// `publish(d, cnt)` runs for every digit as soon as the count is known (the
// chained scan publishes it there).  The key/value registers are free again
// on return (the caller prefetches the next tile into them).
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, bool VALS, typename Publish>
__device__ __forceinline__ void tile_rank_and_shuffle(const PassParams& p, unsigned char* smem,
                                                      uint32_t tile,
                                                      const typename KeyOps<KT>::T (&key)[ITEMS],
                                                      const uint32_t (&val)[VALS ? ITEMS : 1],
                                                      uint32_t* cnt_out, uint32_t* start_out,
                                                      Publish publish)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    constexpr int BINS = S::BINS, TILE = S::TILE, WH = S::WH, CHAINS = S::CHAINS, VWARPS = S::VWARPS;
    T* skeys = reinterpret_cast<T*>(smem + S::keys_off);
    uint32_t* svals = reinterpret_cast<uint32_t*>(smem + S::vals_off);
    uint32_t* whist = reinterpret_cast<uint32_t*>(smem + S::wh_off);
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tile_base = tile * (uint32_t)TILE;
    const uint32_t seg = tile_base + (uint32_t)warp * (32u * ITEMS);

    // (the caller has zeroed the counters and synchronised)
    uint32_t rank[(ITEMS + 1) / 2];
    rank_in_warp<FULL, KT, RB, ITEMS, CHAINS, WH>(key, seg, p.n, p.shift, p.mask,
                                                  whist + warp * CHAINS * WH, lane, rank);
    __syncthreads();

    // Per digit: the tile count, and after the scan each warp's start for the
    // digit inside the tile (the warps' counts are read twice rather than
    // held in registers).
    uint32_t cnt = 0;
    if (tid < BINS) {
#pragma unroll
        for (int w = 0; w < VWARPS; ++w) cnt += whist[w * WH + tid];
        publish(tid, cnt);
    }
    const uint32_t start = bins_exclusive_scan<BINS, false>(tid < BINS ? cnt : 0u, sscan + 16, nullptr);
    if (tid < BINS) {
        uint32_t run = start;
#pragma unroll
        for (int w = 0; w < VWARPS; ++w) {
            const uint32_t c = whist[w * WH + tid];
            whist[w * WH + tid] = run;
            run += c;
        }
    }
    __syncthreads();

    // Shuffle: each digit becomes one contiguous run of the tile.  pos < TILE
    // holds by construction; the clamp keeps a violation inside the tile.
    uint32_t bad = 0;
    const uint32_t* wbase = whist + warp * CHAINS * WH;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t d = step_digit<FULL, KT, RB, ITEMS>(key, k, seg, p.n, p.shift, p.mask, lane);
        const uint32_t r = (k & 1) ? (rank[k / 2] >> 16) : (rank[k / 2] & 0xFFFFu);
        uint32_t pos = wbase[(k / (ITEMS / CHAINS)) * WH + d] + r;
#if RS_CHECKED
        bad |= pos >= (uint32_t)TILE;
#endif
        pos = min(pos, (uint32_t)TILE - 1u);
        if (FULL || d < (uint32_t)BINS) {
            skeys[pos] = key[k];
            if constexpr (VALS) svals[pos] = val[k];
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
// (a failure is recorded and the store skipped).
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, bool VALS>
__device__ __forceinline__ void tile_scatter(const PassParams& p, unsigned char* smem, uint32_t tile)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    constexpr int TILE = S::TILE;
    const T* skeys = reinterpret_cast<const T*>(smem + S::keys_off);
    const uint32_t* svals = reinterpret_cast<const uint32_t*>(smem + S::vals_off);
    const uint32_t* sbase = reinterpret_cast<const uint32_t*>(smem + S::base_off);
    T* out = static_cast<T*>(p.keys_out);
    const uint32_t tile_base = tile * (uint32_t)TILE;
    const uint32_t valid = FULL ? (uint32_t)TILE : p.n - tile_base;
    uint32_t bad = 0;
#if RS_STORE_KEEP
    const uint64_t pol = l2_evict_last_policy();
#endif
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t s = (uint32_t)(k * THREADS) + threadIdx.x;
        if (FULL || s < valid) {
            const T kk = skeys[s];
            const uint32_t idx = sbase[digit_of<KT>(kk, p.shift, p.mask)] + s;
            const bool ok = idx < p.n;
            bad |= !ok;
            if (ok) {
#if RS_STORE_KEEP
                st_keep(out + idx, kk, pol);
                if constexpr (VALS) st_keep(p.vals_out + idx, svals[s], pol);
#else
                out[idx] = kk;
                if constexpr (VALS) p.vals_out[idx] = svals[s];
#endif
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

// One tile of a chained-scan pass.  `next` is the ticket this CTA already
// holds for its following tile; that tile's keys are loaded into the freed
// registers while this tile looks back and scatters.
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, bool VALS>
__device__ __forceinline__ void onesweep_tile(const PassParams& p, unsigned char* smem, uint32_t tile,
                                              uint32_t next, typename KeyOps<KT>::T (&key)[ITEMS],
                                              uint32_t (&val)[VALS ? ITEMS : 1])
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
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
    tile_rank_and_shuffle<FULL, KT, RB, THREADS, ITEMS, VALS>(
        p, smem, tile, key, val, &cnt, &start, [&](int d, uint32_t c) {
            if (!stalled) {
                if (tile == 0) st_relaxed_gpu(my_status + d, kFlagInc | ((gexcl + c) & kValMask));
                else st_relaxed_gpu(my_status + d, kFlagAgg | (c & kValMask));
            }
            if (tile > 0) lookback_preload<RS_LOOKBACK_BATCH>(p, tile, d, BINS, pre);
        });
    if (next < p.num_tiles) load_tile<KT, THREADS, ITEMS, VALS>(p, next, key, val);

    if (tid < BINS) {
        uint32_t excl = gexcl;
        if (tile > 0) {
            excl = lookback<RS_LOOKBACK_BATCH>(p, tile, tid, BINS, pre);
            if (!stalled) st_relaxed_gpu(my_status + tid, kFlagInc | ((excl + cnt) & kValMask));
        }
        sbase[tid] = excl - start;
    }
    __syncthreads();
    tile_scatter<FULL, KT, RB, THREADS, ITEMS, VALS>(p, smem, tile);
}

// Chained-scan pass, persistent: each CTA takes tiles by an atomic ticket
// until none is left.  Tickets are handed out in order, so every tile a CTA
// waits on belongs to a CTA that already runs (and that CTA finishes the
// tile it holds before the one it prefetches).
template <int KT, int RB, int THREADS, int ITEMS, bool VALS>
__global__ void __launch_bounds__(THREADS, RS_TILE_MIN_THREADS_PER_SM / THREADS) k_onesweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* smisc = reinterpret_cast<uint32_t*>(smem + S::misc_off);
    const int tid = threadIdx.x;
    if (tid == 0) smisc[0] = atomicAdd(p.ticket, 1u);
    zero_counters<S>(smem, THREADS);
    __syncthreads();
    uint32_t tile = smisc[0];
    if (tile >= p.num_tiles) return;
    T key[ITEMS];
    uint32_t val[VALS ? ITEMS : 1];
    load_tile<KT, THREADS, ITEMS, VALS>(p, tile, key, val);
    while (true) {
#if RS_OS_PERSISTENT == 1
        __syncthreads();  // the previous tile's scatter is done with shared memory
        if (tid == 0) smisc[1] = atomicAdd(p.ticket, 1u);
        zero_counters<S>(smem, THREADS);
        __syncthreads();
        const uint32_t next = smisc[1];
#else
        const uint32_t next = 0xFFFFFFFFu;
#endif
        if ((tile + 1) * (uint32_t)S::TILE <= p.n)
            onesweep_tile<true, KT, RB, THREADS, ITEMS, VALS>(p, smem, tile, next, key, val);
        else
            onesweep_tile<false, KT, RB, THREADS, ITEMS, VALS>(p, smem, tile, next, key, val);
#if RS_OS_PERSISTENT == 2
        // take the next ticket only now, so no tile waits on a held ticket
        __syncthreads();
        if (tid == 0) smisc[1] = atomicAdd(p.ticket, 1u);
        zero_counters<S>(smem, THREADS);
        __syncthreads();
        tile = smisc[1];
        if (tile >= p.num_tiles) break;
        load_tile<KT, THREADS, ITEMS, VALS>(p, tile, key, val);
#else
        if (next >= p.num_tiles) break;
        tile = next;
#endif
    }
}

// Reduce-then-scan, step 1: digit histogram of each CTA's chunk, written
// digit-major (counts[d * G + g]) so that one exclusive scan of the whole
// array yields every (digit, CTA) start ("Radix sort paralelo sobre el scan",
// section "Las tres fases de una pasada").
template <int KT, int RB, int THREADS, int TILE>
__global__ void __launch_bounds__(THREADS) k_upsweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    constexpr int BINS = 1 << RB;
    constexpr int COLS = 32;          // lane-private counter columns: hist[bin][lane]
    constexpr int VEC = 16 / sizeof(T);
    __shared__ uint32_t hist[BINS * COLS];
    const int tid = threadIdx.x;
    const uint32_t col = tid & 31;
    for (int i = tid; i < BINS * COLS; i += THREADS) hist[i] = 0;
    __syncthreads();
    const uint32_t g = blockIdx.x;
    const uint64_t lo64 = (uint64_t)g * p.tiles_per_cta * TILE;
    const uint32_t lo = lo64 < p.n ? (uint32_t)lo64 : p.n;
    const uint64_t hi64 = lo64 + (uint64_t)p.tiles_per_cta * TILE;
    const uint32_t hi = hi64 < p.n ? (uint32_t)hi64 : p.n;
    const T* src = static_cast<const T*>(p.keys_in);
    auto count = [&](T k) { atomicAdd(&hist[digit_of<KT>(k, p.shift, p.mask) * COLS + col], 1u); };
    // lo is a multiple of TILE, so lo * sizeof(T) is 16-byte aligned whenever the base is.
    uint32_t i = lo;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        constexpr int U = 4;
        const uint32_t nvec = (hi - lo) / VEC;
        const uint4* sv = reinterpret_cast<const uint4*>(src + lo);
        uint32_t v = tid;
        for (; v + (U - 1) * THREADS < nvec; v += U * THREADS) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) w[u] = __ldcs(sv + v + u * THREADS);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                T k[VEC];
                memcpy(k, &w[u], 16);
#pragma unroll
                for (int j = 0; j < VEC; ++j) count(k[j]);
            }
        }
        for (; v < nvec; v += THREADS) {
            const uint4 w = __ldcs(sv + v);
            T k[VEC];
            memcpy(k, &w, 16);
#pragma unroll
            for (int j = 0; j < VEC; ++j) count(k[j]);
        }
        i = lo + nvec * VEC;
    }
    for (i += tid; i < hi; i += THREADS) count(src[i]);
    __syncthreads();
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
template <int THREADS>
__global__ void __launch_bounds__(THREADS) k_spine_scan(uint32_t* counts, uint32_t G, uint32_t* row_total)
{
    __shared__ uint32_t sscan[32];
    const int tid = threadIdx.x;
    uint32_t* row = counts + (size_t)blockIdx.x * G;
    const uint32_t per = (G + THREADS - 1) / THREADS;
    const uint32_t lo = min(G, tid * per), hi = min(G, lo + per);
    uint32_t sum = 0;
    for (uint32_t i = lo; i < hi; ++i) sum += row[i];
    uint32_t total;
    uint32_t run = bins_exclusive_scan<THREADS>(sum, sscan, &total);
    for (uint32_t i = lo; i < hi; ++i) {
        const uint32_t c = row[i];
        row[i] = run;
        run += c;
    }
    if (tid == 0) row_total[blockIdx.x] = total;
}

// Reduce-then-scan, step 3: each CTA walks its chunk tile by tile, keeping a
// running global offset per digit.
template <bool FULL, int KT, int RB, int THREADS, int ITEMS, bool VALS>
__device__ __forceinline__ void downsweep_tile(const PassParams& p, unsigned char* smem, uint32_t tile,
                                               uint32_t next, uint32_t& running,
                                               typename KeyOps<KT>::T (&key)[ITEMS],
                                               uint32_t (&val)[VALS ? ITEMS : 1])
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    constexpr int BINS = S::BINS;
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem + S::base_off);
    const int tid = threadIdx.x;
    uint32_t cnt, start;
    tile_rank_and_shuffle<FULL, KT, RB, THREADS, ITEMS, VALS>(p, smem, tile, key, val, &cnt, &start,
                                                               [](int, uint32_t) {});
    if (next != 0xFFFFFFFFu) load_tile<KT, THREADS, ITEMS, VALS>(p, next, key, val);
    if (tid < BINS) {
        sbase[tid] = running - start;
        running += cnt;
    }
    __syncthreads();
    zero_counters<S>(smem, THREADS);  // for the next tile; the scatter does not read them
    tile_scatter<FULL, KT, RB, THREADS, ITEMS, VALS>(p, smem, tile);
    __syncthreads();  // the next tile reuses shared memory
}

template <int KT, int RB, int THREADS, int ITEMS, bool VALS>
__global__ void __launch_bounds__(THREADS, RS_TILE_MIN_THREADS_PER_SM / THREADS) k_downsweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    constexpr int BINS = S::BINS;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);
    const int tid = threadIdx.x;
    const uint32_t g = blockIdx.x;
    zero_counters<S>(smem, THREADS);  // made visible by the scan's barriers
    const uint32_t dstart = bins_exclusive_scan<BINS>(tid < BINS ? p.ghist[tid] : 0u, sscan, nullptr);
    uint32_t running = tid < BINS ? dstart + p.counts[(size_t)tid * p.G + g] : 0u;
    const uint32_t t0 = g * p.tiles_per_cta;
    const uint32_t t1 = min(p.num_tiles, t0 + p.tiles_per_cta);
    if (t0 >= t1) return;
    T key[ITEMS];
    uint32_t val[VALS ? ITEMS : 1];
    load_tile<KT, THREADS, ITEMS, VALS>(p, t0, key, val);
    for (uint32_t tile = t0; tile < t1; ++tile) {
        const uint32_t next = tile + 1 < t1 ? tile + 1 : 0xFFFFFFFFu;
        if ((tile + 1) * (uint32_t)S::TILE <= p.n)
            downsweep_tile<true, KT, RB, THREADS, ITEMS, VALS>(p, smem, tile, next, running, key, val);
        else
            downsweep_tile<false, KT, RB, THREADS, ITEMS, VALS>(p, smem, tile, next, running, key, val);
    }
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
};

// Counters are lane-private columns, hist[pass][bin][col] with col = lane %
// COLS, so the COLS lanes of a warp that share no column hit distinct banks:
// the shared atomics of one warp instruction do not conflict (the warps of
// the CTA still share the columns, which the atomics make safe).
template <int KT, int RB, int THREADS, int COLS>
__global__ void __launch_bounds__(THREADS) k_histogram(HistParams h)
{
    using T = typename KeyOps<KT>::T;
    constexpr int BINS = 1 << RB;
    constexpr int VEC = 16 / sizeof(T);
    constexpr int U = 4;  // vectors in flight per thread
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem);
    const int tid = threadIdx.x;
    const uint32_t col = tid % COLS;
    const uint32_t words = h.passes * BINS * COLS;
    for (uint32_t i = tid; i < words; i += THREADS) hist[i] = 0;
    __syncthreads();

    auto count = [&](T k) {
        const auto o = KeyOps<KT>::ordered(k);
        uint32_t shift = h.begin_bit;
        uint32_t* row = hist + col;
        for (uint32_t q = 0; q < h.passes; ++q, shift += RB, row += BINS * COLS) {
            const uint32_t width = min((uint32_t)RB, h.end_bit - shift);
            const uint32_t d = (uint32_t)(o >> shift) & ((1u << width) - 1u);
            atomicAdd(row + d * COLS, 1u);
        }
    };

    const size_t gthreads = (size_t)gridDim.x * THREADS;
    const size_t gid = (size_t)blockIdx.x * THREADS + tid;
    const T* keys = static_cast<const T*>(h.keys);
    size_t done = 0;
    if (h.aligned16) {
        const size_t nvec = h.n / VEC;
        const uint4* kv = reinterpret_cast<const uint4*>(keys);
        size_t v = gid;
        for (; v + (U - 1) * gthreads < nvec; v += U * gthreads) {
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u) w[u] = __ldcs(kv + v + u * gthreads);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                T k[VEC];
                memcpy(k, &w[u], 16);
#pragma unroll
                for (int j = 0; j < VEC; ++j) count(k[j]);
            }
        }
        for (; v < nvec; v += gthreads) {
            const uint4 w = __ldcs(kv + v);
            T k[VEC];
            memcpy(k, &w, 16);
#pragma unroll
            for (int j = 0; j < VEC; ++j) count(k[j]);
        }
        done = nvec * VEC;
    }
    for (size_t i = done + gid; i < h.n; i += gthreads) count(keys[i]);
    __syncthreads();
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
    size_t n;
    int begin_bit, end_bit;
    int algo;         // RS_ALGO_ONESWEEP or RS_ALGO_REDUCE_SCAN (resolved)
    int radix_bits;   // 4 or 8
    int passes;
    const void* keys_in;
    void* keys_out;
    const uint32_t* vals_in;
    uint32_t* vals_out;
    unsigned char* temp;
    TempLayout lay;
    cudaStream_t stream;
    uint32_t spin_limit;
    int32_t stall_tile;
    // profiling (optional)
    cudaEvent_t const* events;
    int max_events;
    int launched;
    int* kinds;
    bool count_only;   // only count kernels, launch nothing
};

enum KernelKind { kKindHistogram = 1, kKindOnesweep = 2, kKindUpsweep = 3, kKindSpine = 4,
                  kKindDownsweep = 5, kKindCopy = 6 };

// After every launch: check it, and record the next profiling event.
inline rs_status after_launch(Plan& pl, int kind)
{
    if (pl.count_only) { pl.launched++; return RS_OK; }
    if (cudaGetLastError() != cudaSuccess) return RS_ERR_CUDA;
    if (pl.kinds && pl.launched < pl.max_events) pl.kinds[pl.launched] = kind;
    pl.launched++;
    if (pl.events && pl.launched < pl.max_events)
        if (cudaEventRecord(pl.events[pl.launched], pl.stream) != cudaSuccess) return RS_ERR_CUDA;
    return RS_OK;
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

template <int KT, int RB, bool VALS>
rs_status run_passes(Plan& pl)
{
    using T = typename KeyOps<KT>::T;
    constexpr int KB = sizeof(T);
    constexpr int ITEMS = tile_items(KB, VALS);
    constexpr int BINS = 1 << RB;
    const uint32_t n = (uint32_t)pl.n;
    uint32_t* meta = reinterpret_cast<uint32_t*>(pl.temp + pl.lay.meta);
    uint32_t* big = reinterpret_cast<uint32_t*>(pl.temp + pl.lay.big);
    T* alt_keys = reinterpret_cast<T*>(pl.temp + pl.lay.alt_keys);
    uint32_t* alt_vals = reinterpret_cast<uint32_t*>(pl.temp + pl.lay.alt_vals);
    const int P = pl.passes;

    // Destination of pass q: the final pass writes keys_out.
    auto dst_keys = [&](int q) -> T* { return ((P - 1 - q) % 2 == 0) ? static_cast<T*>(pl.keys_out) : alt_keys; };
    auto dst_vals = [&](int q) -> uint32_t* { return ((P - 1 - q) % 2 == 0) ? pl.vals_out : alt_vals; };

    const T* src_keys0 = static_cast<const T*>(pl.keys_in);
    const uint32_t* src_vals0 = pl.vals_in;
    // In place with an odd number of passes: pass 0 would overwrite keys it
    // has not read yet, so start from a copy in the ping-pong buffer.
    const bool copy_first = (pl.keys_in == pl.keys_out) && (P % 2 == 1);
    if (copy_first) {
        if (!pl.count_only) {
            if (cudaMemcpyAsync(alt_keys, pl.keys_in, pl.n * KB, cudaMemcpyDeviceToDevice, pl.stream) != cudaSuccess)
                return RS_ERR_CUDA;
            if (VALS && cudaMemcpyAsync(alt_vals, pl.vals_in, pl.n * 4, cudaMemcpyDeviceToDevice, pl.stream) != cudaSuccess)
                return RS_ERR_CUDA;
        }
        src_keys0 = alt_keys;
        src_vals0 = alt_vals;
    }
    // With copy_first, pass 0 (reading alt) writes keys_out because P is odd.

    PassParams base{};
    base.n = n;
    base.err = meta + kErrWord;
    base.spin_limit = pl.spin_limit;
    base.stall_tile = pl.stall_tile;

    if (pl.algo == RS_ALGO_ONESWEEP) {
        constexpr int THREADS = tile_threads(kAlgoOnesweep, KB, VALS);
        constexpr int TILE = THREADS * ITEMS;
        using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
        const uint32_t num_tiles = (n + TILE - 1) / TILE;
        base.num_tiles = num_tiles;
        constexpr int MAXP = (8 * KB + RB - 1) / RB;
        constexpr int HCOLS = (MAXP * (1 << RB) * 32 * 4 <= 160 * 1024) ? 32 : 16;
        auto hk = k_histogram<KT, RB, 1024, HCOLS>;
        auto pk = k_onesweep<KT, RB, THREADS, ITEMS, VALS>;
        auto pkb = k_onesweep<ByteTwin<KT>::value, RB, THREADS, ITEMS, VALS>;
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
        const int sms = pl.count_only ? 1 : device_sm_count();
        const size_t want = (n + 1024 * 16 - 1) / (1024 * 16);
        const int hgrid = (int)std::max<size_t>(1, std::min<size_t>(want, (size_t)sms));
        const size_t hsmem = (size_t)P * BINS * HCOLS * 4;
        if (!pl.count_only && !set_smem(hk, hsmem)) return RS_ERR_CUDA;
        if (!pl.count_only) hk<<<hgrid, 1024, hsmem, pl.stream>>>(h);
        rs_status st = after_launch(pl, kKindHistogram);
        if (st != RS_OK) return st;
        uint32_t os_grid = num_tiles;
        if (!pl.count_only) {
            int occ = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, pk, THREADS, S::bytes) != cudaSuccess || occ < 1)
                occ = 1;
            os_grid = RS_OS_PERSISTENT ? (uint32_t)std::min<size_t>((size_t)sms * occ, num_tiles) : num_tiles;
            (void)pkb;
        }
        for (int q = 0; q < P; ++q) {
            PassParams pp = base;
            pp.keys_in = q == 0 ? (const void*)src_keys0 : (const void*)dst_keys(q - 1);
            pp.keys_out = dst_keys(q);
            pp.vals_in = VALS ? (q == 0 ? src_vals0 : dst_vals(q - 1)) : nullptr;
            pp.vals_out = VALS ? dst_vals(q) : nullptr;
            pp.shift = pl.begin_bit + q * RB;
            const uint32_t width = std::min(RB, pl.end_bit - (int)pp.shift);
            pp.mask = (1u << width) - 1u;
            pp.status = big + (size_t)q * num_tiles * BINS;
            pp.ghist = meta + kGhistBase + q * BINS;
            pp.ticket = meta + kTicketBase + q;
            const bool byte_digit = (RB == 8) && (pp.shift % 8 == 0) && (pp.mask == 0xFFu);
            if (!pl.count_only) (byte_digit ? pkb : pk)<<<os_grid, THREADS, S::bytes, pl.stream>>>(pp);
            st = after_launch(pl, kKindOnesweep);
            if (st != RS_OK) return st;
        }
        return RS_OK;
    }

    // Reduce-then-scan.
    constexpr int THREADS = tile_threads(kAlgoReduceScan, KB, VALS);
    constexpr int TILE = THREADS * ITEMS;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    const uint32_t num_tiles = (n + TILE - 1) / TILE;
    base.num_tiles = num_tiles;
    auto uk = k_upsweep<KT, RB, 512, TILE>;
    auto dk = k_downsweep<KT, RB, THREADS, ITEMS, VALS>;
    auto dkb = k_downsweep<ByteTwin<KT>::value, RB, THREADS, ITEMS, VALS>;
    if (!pl.count_only && (!set_smem(dk, S::bytes) || !set_smem(dkb, S::bytes))) return RS_ERR_CUDA;
    uint32_t G = 1;
    if (!pl.count_only) {
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dk, THREADS, S::bytes) != cudaSuccess || occ < 1)
            occ = 1;
        G = (uint32_t)std::min<size_t>((size_t)device_sm_count() * occ, (size_t)kRtsMaxCtas);
    }
    G = std::max<uint32_t>(1, std::min<uint32_t>(G, num_tiles));
    const uint32_t tpc = (num_tiles + G - 1) / G;
    G = (num_tiles + tpc - 1) / tpc;
    for (int q = 0; q < P; ++q) {
        PassParams pp = base;
        pp.keys_in = q == 0 ? (const void*)src_keys0 : (const void*)dst_keys(q - 1);
        pp.keys_out = dst_keys(q);
        pp.vals_in = VALS ? (q == 0 ? src_vals0 : dst_vals(q - 1)) : nullptr;
        pp.vals_out = VALS ? dst_vals(q) : nullptr;
        pp.shift = pl.begin_bit + q * RB;
        const uint32_t width = std::min(RB, pl.end_bit - (int)pp.shift);
        pp.mask = (1u << width) - 1u;
        pp.counts = big;
        pp.G = G;
        pp.tiles_per_cta = tpc;
        if (!pl.count_only) uk<<<G, 512, 0, pl.stream>>>(pp);
        rs_status st = after_launch(pl, kKindUpsweep);
        if (st != RS_OK) return st;
        pp.ghist = meta + kGhistBase + q * BINS;  // row totals of this pass
        if (!pl.count_only)
            k_spine_scan<256><<<BINS, 256, 0, pl.stream>>>(big, G, meta + kGhistBase + q * BINS);
        st = after_launch(pl, kKindSpine);
        if (st != RS_OK) return st;
        const bool byte_digit = (RB == 8) && (pp.shift % 8 == 0) && (pp.mask == 0xFFu);
        if (!pl.count_only) (byte_digit ? dkb : dk)<<<G, THREADS, S::bytes, pl.stream>>>(pp);
        st = after_launch(pl, kKindDownsweep);
        if (st != RS_OK) return st;
    }
    return RS_OK;
}

template <int KT>
rs_status run_sort(Plan& pl)
{
    if (pl.vals) {
        if (pl.radix_bits == 4) return run_passes<KT, 4, true>(pl);
        return run_passes<KT, 8, true>(pl);
    }
    if (pl.radix_bits == 4) return run_passes<KT, 4, false>(pl);
    return run_passes<KT, 8, false>(pl);
}

}  // namespace rs
