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

#ifndef RS_CHECKED
#define RS_CHECKED 1
#endif

namespace rs {

enum : int { KU32 = 0, KI32 = 1, KF32 = 2, KU64 = 3 };

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

template <int KT>
__device__ __forceinline__ uint32_t digit_of(typename KeyOps<KT>::T u, uint32_t shift, uint32_t mask)
{
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
// block (others pass 0).  Every thread must call it: it holds two barriers.
// `scratch` needs 32 words.  *total (if given) receives the sum.
template <int BINS>
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
    __syncthreads();
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
    static constexpr int TILE = THREADS * ITEMS;
    static constexpr int WH = BINS + 1;  // per-warp counters + one dummy slot for tail lanes
    static constexpr size_t keys_off = 0;
    static constexpr size_t vals_off = align_up(sizeof(T) * TILE, 16);
    static constexpr size_t wh_off = vals_off + (VALS ? align_up(4 * (size_t)TILE, 16) : 0);
    static constexpr size_t base_off = wh_off + align_up(4 * (size_t)WARPS * WH, 16);
    static constexpr size_t scan_off = base_off + 4 * BINS;
    static constexpr size_t misc_off = scan_off + 4 * 32;
    static constexpr size_t bytes = misc_off + 16;
};

// --------------------------------------------------------------- tile pieces

// Load ITEMS keys per thread in warp-striped order: lane l of warp w holds
// positions seg + k*32 + l, so every load instruction of a warp covers 32
// consecutive keys and the processing order (k, lane) is the input order.
template <typename T, int ITEMS>
__device__ __forceinline__ void load_striped(const T* __restrict__ src, uint32_t seg, uint32_t n,
                                             bool full, int lane, T (&v)[ITEMS])
{
    if (full) {
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) v[k] = src[seg + k * 32 + lane];
    } else {
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
            uint32_t i = seg + k * 32 + lane;
            v[k] = i < n ? src[i] : T(0);
        }
    }
}

// Stable rank of each key among equal digits within its warp's segment.
// __match_any_sync gives the lanes holding the same digit in this step; the
// key's rank is the warp's running count for that digit plus the number of
// such lanes below it; the highest of those lanes then advances the count.
// packed[k] = rank | digit << 16 (digit BINS marks a lane past the end).
template <int KT, int BINS, int ITEMS>
__device__ __forceinline__ void rank_in_warp(const typename KeyOps<KT>::T (&key)[ITEMS], uint32_t seg,
                                             uint32_t n, bool full, uint32_t shift, uint32_t mask,
                                             uint32_t* wh, int lane, uint32_t (&packed)[ITEMS])
{
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        uint32_t d = digit_of<KT>(key[k], shift, mask);
        if (!full && seg + k * 32 + lane >= n) d = BINS;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
        const uint32_t r = wh[d] + __popc(peers & lt);
        __syncwarp();
        if ((peers >> lane) == 1u) wh[d] = r + 1;
        __syncwarp();
        packed[k] = r | (d << 16);
    }
}

// Everything of one tile up to the point where its global digit offsets are
// needed: load, rank, per-digit counts, tile-local digit starts, shuffle into
// shared memory.  Returns, for thread d < BINS, the tile's count of digit d in
// *cnt and its tile-local start in *start.  `publish(d, cnt)` runs for every
// digit as soon as the count is known (the chained scan publishes it there).
template <int KT, int RB, int THREADS, int ITEMS, bool VALS, typename Publish>
__device__ __forceinline__ void tile_rank_and_shuffle(const PassParams& p, unsigned char* smem,
                                                      uint32_t tile, uint32_t* cnt_out,
                                                      uint32_t* start_out, Publish publish)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    constexpr int BINS = S::BINS, WARPS = S::WARPS, TILE = S::TILE, WH = S::WH;
    T* skeys = reinterpret_cast<T*>(smem + S::keys_off);
    uint32_t* svals = reinterpret_cast<uint32_t*>(smem + S::vals_off);
    uint32_t* whist = reinterpret_cast<uint32_t*>(smem + S::wh_off);
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem + S::base_off);
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t tile_base = tile * (uint32_t)TILE;
    const bool full = tile_base + (uint32_t)TILE <= p.n;
    const uint32_t seg = tile_base + (uint32_t)warp * (32u * ITEMS);

    for (int i = tid; i < WARPS * WH; i += THREADS) whist[i] = 0;

    T key[ITEMS];
    load_striped<T, ITEMS>(static_cast<const T*>(p.keys_in), seg, p.n, full, lane, key);
    uint32_t val[VALS ? ITEMS : 1];
    if constexpr (VALS) load_striped<uint32_t, ITEMS>(p.vals_in, seg, p.n, full, lane, val);
    __syncthreads();  // counters zeroed

    uint32_t packed[ITEMS];
    rank_in_warp<KT, BINS, ITEMS>(key, seg, p.n, full, p.shift, p.mask, whist + warp * WH, lane, packed);
    __syncthreads();

    // Per digit: turn the warps' counts into each warp's exclusive offset.
    uint32_t cnt = 0;
    if (tid < BINS) {
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            uint32_t c = whist[w * WH + tid];
            whist[w * WH + tid] = cnt;
            cnt += c;
        }
        publish(tid, cnt);
    }
    const uint32_t start = bins_exclusive_scan<BINS>(tid < BINS ? cnt : 0u, sscan, nullptr);
    if (tid < BINS) {
#pragma unroll
        for (int w = 0; w < WARPS; ++w) whist[w * WH + tid] += start;
    }
    __syncthreads();

    // Shuffle: each digit becomes one contiguous run of the tile.
    uint32_t bad = 0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t d = packed[k] >> 16;
        if (full || d < (uint32_t)BINS) {
            const uint32_t pos = whist[warp * WH + d] + (packed[k] & 0xFFFFu);
#if RS_CHECKED
            if (pos >= (uint32_t)TILE) { bad = 1; continue; }
#endif
            skeys[pos] = key[k];
            if constexpr (VALS) svals[pos] = val[k];
        }
    }
    if (bad) record_error(p.err, RS_ERR_CHECK_FAILED);
    *cnt_out = cnt;
    *start_out = start;
    (void)sbase;
}

// Scatter the shuffled tile: slot s holds a key of digit d, whose global
// position is sbase[d] + s (sbase = global offset of the digit's run minus
// its tile-local start).  Consecutive slots mostly share a digit, so each
// warp store covers few, contiguous segments.
template <int KT, int RB, int THREADS, int ITEMS, bool VALS>
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
    const uint32_t valid = p.n - tile_base < (uint32_t)TILE ? p.n - tile_base : (uint32_t)TILE;
    uint32_t bad = 0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const uint32_t s = (uint32_t)(k * THREADS) + threadIdx.x;
        if (s < valid) {
            const T kk = skeys[s];
            const uint32_t idx = sbase[digit_of<KT>(kk, p.shift, p.mask)] + s;
            if (idx < p.n) {
                out[idx] = kk;
                if constexpr (VALS) p.vals_out[idx] = svals[s];
            } else {
                bad = 1;
            }
        }
    }
    if (bad) record_error(p.err, RS_ERR_CHECK_FAILED);
}

// ------------------------------------------------------------------ kernels

// Chained-scan pass: one CTA per tile, tiles numbered by an atomic ticket so
// that every tile a CTA waits on belongs to a CTA that started earlier.
template <int KT, int RB, int THREADS, int ITEMS, bool VALS>
__global__ void __launch_bounds__(THREADS) k_onesweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    constexpr int BINS = S::BINS;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem + S::base_off);
    uint32_t* sscan = reinterpret_cast<uint32_t*>(smem + S::scan_off);
    uint32_t* smisc = reinterpret_cast<uint32_t*>(smem + S::misc_off);
    const int tid = threadIdx.x;

    if (tid == 0) smisc[0] = atomicAdd(p.ticket, 1u);
    __syncthreads();
    const uint32_t tile = smisc[0];
    const bool stalled = (int32_t)tile + 1 == p.stall_tile;
    uint32_t* my_status = p.status + (size_t)tile * BINS;

    // Tile 0 needs the pass's global digit starts: an exclusive scan of the
    // histogram.  Its published value is then already inclusive.
    uint32_t gexcl = 0;
    if (tile == 0) gexcl = bins_exclusive_scan<BINS>(tid < BINS ? p.ghist[tid] : 0u, sscan, nullptr);

    uint32_t cnt, start;
    tile_rank_and_shuffle<KT, RB, THREADS, ITEMS, VALS>(
        p, smem, tile, &cnt, &start, [&](int d, uint32_t c) {
            if (stalled) return;
            if (tile == 0) st_relaxed_gpu(my_status + d, kFlagInc | ((gexcl + c) & kValMask));
            else st_relaxed_gpu(my_status + d, kFlagAgg | (c & kValMask));
        });

    // Decoupled look-back, one thread per digit: walk back over predecessor
    // tiles adding their counts until one that already holds an inclusive sum.
    if (tid < BINS) {
        uint32_t excl = gexcl;
        if (tile > 0) {
            int32_t t = (int32_t)tile - 1;
            uint32_t spins = 0;
            bool timed_out = false;
            while (t >= 0) {
                const uint32_t s = ld_relaxed_gpu(p.status + (size_t)t * BINS + tid);
                const uint32_t f = s & ~kValMask;
                if (f == 0u) {
                    if (++spins >= p.spin_limit) { timed_out = true; break; }
                    continue;
                }
                excl += s & kValMask;
                if (f == kFlagInc) break;
                --t;
            }
            if (timed_out || t < 0) {
                record_error(p.err, RS_ERR_DEVICE_TIMEOUT);
                __threadfence();
            }
            if (!stalled) st_relaxed_gpu(my_status + tid, kFlagInc | ((excl + cnt) & kValMask));
        }
        sbase[tid] = excl - start;
    }
    __syncthreads();
    tile_scatter<KT, RB, THREADS, ITEMS, VALS>(p, smem, tile);
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
    __shared__ uint32_t hist[BINS];
    const int tid = threadIdx.x;
    for (int i = tid; i < BINS; i += THREADS) hist[i] = 0;
    __syncthreads();
    const uint32_t g = blockIdx.x;
    const uint64_t lo64 = (uint64_t)g * p.tiles_per_cta * TILE;
    const uint32_t lo = lo64 < p.n ? (uint32_t)lo64 : p.n;
    const uint64_t hi64 = lo64 + (uint64_t)p.tiles_per_cta * TILE;
    const uint32_t hi = hi64 < p.n ? (uint32_t)hi64 : p.n;
    const T* src = static_cast<const T*>(p.keys_in);
    constexpr int U = 4;
    uint32_t i = lo + tid;
    for (; i + (U - 1) * THREADS < hi; i += U * THREADS) {
        T k[U];
#pragma unroll
        for (int u = 0; u < U; ++u) k[u] = src[i + u * THREADS];
#pragma unroll
        for (int u = 0; u < U; ++u) atomicAdd(&hist[digit_of<KT>(k[u], p.shift, p.mask)], 1u);
    }
    for (; i < hi; i += THREADS) atomicAdd(&hist[digit_of<KT>(src[i], p.shift, p.mask)], 1u);
    __syncthreads();
    for (int d = tid; d < BINS; d += THREADS) p.counts[(size_t)d * p.G + g] = hist[d];
}

// Reduce-then-scan, step 2: exclusive scan, in place, of the m digit-major
// counts, by one CTA: per-thread segment sums, a block scan of the sums, then
// each thread rewrites its segment.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) k_spine_scan(uint32_t* counts, uint32_t m)
{
    __shared__ uint32_t part[THREADS];
    const int tid = threadIdx.x;
    const uint32_t per = (m + THREADS - 1) / THREADS;
    const uint32_t lo = min(m, tid * per), hi = min(m, lo + per);
    uint32_t sum = 0;
    for (uint32_t i = lo; i < hi; ++i) sum += counts[i];
    part[tid] = sum;
    __syncthreads();
    // Hillis-Steele scan of THREADS partial sums in shared memory (inclusive).
    for (int o = 1; o < THREADS; o <<= 1) {
        uint32_t v = tid >= o ? part[tid - o] : 0u;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    uint32_t run = part[tid] - sum;
    for (uint32_t i = lo; i < hi; ++i) {
        uint32_t c = counts[i];
        counts[i] = run;
        run += c;
    }
}

// Reduce-then-scan, step 3: each CTA walks its chunk tile by tile, keeping a
// running global offset per digit.
template <int KT, int RB, int THREADS, int ITEMS, bool VALS>
__global__ void __launch_bounds__(THREADS) k_downsweep(PassParams p)
{
    using T = typename KeyOps<KT>::T;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;
    constexpr int BINS = S::BINS;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem + S::base_off);
    const int tid = threadIdx.x;
    const uint32_t g = blockIdx.x;
    uint32_t running = tid < BINS ? p.counts[(size_t)tid * p.G + g] : 0u;
    const uint32_t t0 = g * p.tiles_per_cta;
    const uint32_t t1 = min(p.num_tiles, t0 + p.tiles_per_cta);
    for (uint32_t tile = t0; tile < t1; ++tile) {
        uint32_t cnt, start;
        tile_rank_and_shuffle<KT, RB, THREADS, ITEMS, VALS>(p, smem, tile, &cnt, &start,
                                                             [](int, uint32_t) {});
        if (tid < BINS) {
            sbase[tid] = running - start;
            running += cnt;
        }
        __syncthreads();
        tile_scatter<KT, RB, THREADS, ITEMS, VALS>(p, smem, tile);
        __syncthreads();  // the next tile reuses shared memory
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

template <int KT, int RB, int THREADS>
__global__ void __launch_bounds__(THREADS) k_histogram(HistParams h)
{
    using T = typename KeyOps<KT>::T;
    constexpr int BINS = 1 << RB;
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem);
    const int tid = threadIdx.x;
    const uint32_t words = h.passes * BINS;
    for (uint32_t i = tid; i < words; i += THREADS) hist[i] = 0;
    __syncthreads();

    auto count = [&](T k) {
        const auto o = KeyOps<KT>::ordered(k);
        uint32_t shift = h.begin_bit;
        for (uint32_t q = 0; q < h.passes; ++q, shift += RB) {
            const uint32_t width = min((uint32_t)RB, h.end_bit - shift);
            const uint32_t d = (uint32_t)(o >> shift) & ((1u << width) - 1u);
            atomicAdd(&hist[q * BINS + d], 1u);
        }
    };

    const size_t gthreads = (size_t)gridDim.x * THREADS;
    const size_t gid = (size_t)blockIdx.x * THREADS + tid;
    const T* keys = static_cast<const T*>(h.keys);
    size_t done = 0;
    if (h.aligned16) {
        const size_t nvec = h.n / VEC;
        const uint4* kv = reinterpret_cast<const uint4*>(keys);
        for (size_t v = gid; v < nvec; v += gthreads) {
            const uint4 w = kv[v];
            T k[VEC];
            memcpy(k, &w, 16);
#pragma unroll
            for (int j = 0; j < VEC; ++j) count(k[j]);
        }
        done = nvec * VEC;
    }
    for (size_t i = done + gid; i < h.n; i += gthreads) count(keys[i]);
    __syncthreads();
    for (uint32_t i = tid; i < words; i += THREADS) {
        const uint32_t c = hist[i];
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

template <int KT, int RB, bool VALS>
rs_status run_passes(Plan& pl)
{
    using T = typename KeyOps<KT>::T;
    constexpr int KB = sizeof(T);
    constexpr int THREADS = kTileThreads;
    constexpr int ITEMS = tile_items(KB, VALS);
    constexpr int TILE = THREADS * ITEMS;
    constexpr int BINS = 1 << RB;
    using S = TileSmem<T, RB, THREADS, ITEMS, VALS>;

    const uint32_t n = (uint32_t)pl.n;
    const uint32_t num_tiles = (n + TILE - 1) / TILE;
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
    base.num_tiles = num_tiles;
    base.err = meta + kErrWord;
    base.spin_limit = pl.spin_limit;
    base.stall_tile = pl.stall_tile;

    if (pl.algo == RS_ALGO_ONESWEEP) {
        auto hk = k_histogram<KT, RB, 512>;
        auto pk = k_onesweep<KT, RB, THREADS, ITEMS, VALS>;
        if (!pl.count_only && !set_smem(pk, S::bytes)) return RS_ERR_CUDA;
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
        const size_t want = (n + 512 * 16 - 1) / (512 * 16);
        const int hgrid = (int)std::max<size_t>(1, std::min<size_t>(want, (size_t)sms * 2));
        if (!pl.count_only) hk<<<hgrid, 512, (size_t)P * BINS * 4, pl.stream>>>(h);
        rs_status st = after_launch(pl, kKindHistogram);
        if (st != RS_OK) return st;
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
            if (!pl.count_only) pk<<<num_tiles, THREADS, S::bytes, pl.stream>>>(pp);
            st = after_launch(pl, kKindOnesweep);
            if (st != RS_OK) return st;
        }
        return RS_OK;
    }

    // Reduce-then-scan.
    auto uk = k_upsweep<KT, RB, 512, TILE>;
    auto dk = k_downsweep<KT, RB, THREADS, ITEMS, VALS>;
    if (!pl.count_only && !set_smem(dk, S::bytes)) return RS_ERR_CUDA;
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
        if (!pl.count_only) k_spine_scan<1024><<<1, 1024, 0, pl.stream>>>(big, (uint32_t)BINS * G);
        st = after_launch(pl, kKindSpine);
        if (st != RS_OK) return st;
        if (!pl.count_only) dk<<<G, THREADS, S::bytes, pl.stream>>>(pp);
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
