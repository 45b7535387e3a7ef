/*
 * rs.h -- C ABI of a stable least-significant-digit radix sort for NVIDIA
 * GB300 (sm_103a).
 *
 * What is computed.  For n keys of one type (uint32, int32, float32, uint64,
 * uint16, int16 or binary16) and a bit range [begin_bit, end_bit), the sort
 * returns the keys, and optionally one uint32 value per key, in the unique
 * STABLE order of
 *     D(i) = bits [begin_bit, end_bit) of T(key_i),
 * ascending (descending on request, rs_sort_desc.descending), ties kept in
 * input order either way.  T is the order-preserving map to an unsigned
 * integer:
 *   - uint32, uint64, uint16: identity;
 *   - int32, int16: flip the sign bit ("Radix sort paralelo sobre el scan",
 *     section "Claves con signo y en coma flotante");
 *   - float32: NaN (any payload, either sign) and +-Inf map to 0xFFFFFFFF;
 *     otherwise a set sign bit flips every bit and a clear one sets the MSB
 *     ("Radix sort を実装 & 測定してみた", section "符号付型、浮動小数点型に
 *     対する radix sort").  So -Inf, +Inf and all NaNs tie after every finite
 *     value, in input order, and -0.0 sorts just before +0.0;
 *   - binary16: the same rule at 16 bits (that section says other widths
 *     sort by the same procedure): exponent field all ones -> 0xFFFF.
 * The output keys are the ORIGINAL bit patterns (nothing is re-encoded).  Bits
 * outside [begin_bit, end_bit) of T(key) do not influence the order.
 *
 * Method.  Each pass sorts by one r-bit digit (r = 8 by default, 4 on
 * request), lowest digit first ("Radix sort paralelo sobre el scan", sections
 * "La idea y el requisito de estabilidad" and "Las tres fases de una pasada"):
 * a per-block digit histogram, an exclusive scan of the block counts laid out
 * digit-major, a block-local stable rank and shuffle in shared memory, and a
 * coalesced scatter ("정렬: 라딕스와 머지소트", 13.3-13.6).  Two schedules
 * exist: a three-kernel reduce-then-scan per pass, and a single-pass chained
 * scan with decoupled look-back that reads every key once up front for all
 * pass histograms.
 *
 * Pass skipping.  The first read of the keys also records which bits of T(key)
 * differ between keys and whether the input is already in order.  A pass
 * whose digit is the same for every key, and every pass of an input already
 * in order ("高性能计算：GPU上的基数排序", section 基数排序在GPU上的具体实现),
 * is skipped on the device: its kernels still launch (the launch sequence
 * depends on the shape only, so a captured graph stays valid) but return at
 * once, and the remaining passes re-route their buffers so the result still
 * lands in keys_out.  The output is the same as without skipping.
 *
 * Conventions for every entry point below.
 *   Pointers.  Key, value and temp pointers are DEVICE pointers (cudaMalloc,
 *     cudaMallocAsync or a framework allocator) unless a parameter says
 *     "host".  The caller owns all memory; the library allocates no device
 *     memory and keeps no device state outside `temp`.
 *   Alignment.  Keys and values must be aligned to their element size; temp
 *     must be 256-byte aligned.  16-byte-aligned keys take the vector-load
 *     path; others are still sorted correctly.
 *   Aliasing.  keys_out may equal keys_in exactly (in-place sort: one more
 *     kernel is launched, which copies the result back from temp when an odd
 *     number of passes ran), likewise vals_out and vals_in.  Any other
 *     overlap among the key, value and temp buffers is RS_ERR_ALIAS.
 *   Stream.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Calls only enqueue work: they do not synchronise,
 *     allocate or read device memory back, so they may be captured into a
 *     CUDA graph.  Inside one sort, every kernel after the first is launched
 *     as a programmatic dependent of the kernel before it (it waits on the
 *     device before touching memory); the first is an ordinary launch, so
 *     the sort starts after the work enqueued before it, and ordinary work
 *     enqueued after it starts after the sort's last kernel has finished.  RS_OK means "enqueued"; faults the device detects (a
 *     look-back wait that ran out, an index that failed its bounds check) are
 *     written to an error word inside `temp` and read by rs_device_status().
 *   Sizes.  n may be 0 (nothing is launched).  n must be at most
 *     2^32 - 2^16 (the chained-scan schedule needs n < 2^30; AUTO uses
 *     reduce-then-scan above that).  0 <= begin_bit <= end_bit <= 32 (64 for
 *     uint64); begin_bit == end_bit is a stable copy.
 *   Errors.  Invalid arguments return an error before anything is enqueued;
 *     RS_ERR_CUDA reports a failed launch or copy (cudaGetLastError).
 */
#ifndef RS_H
#define RS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest n any sort accepts (2^32 - 2^16; positions and tile indices stay in
 * 32 bits). */
#define RS_MAX_N 4294901760u

typedef enum rs_status {
    RS_OK = 0,
    RS_ERR_INVALID_ARG = 1,    /* null pointer, bad bit range, n too large, bad enum   */
    RS_ERR_TEMP_TOO_SMALL = 2, /* temp_bytes < rs_temp_bytes(...)                      */
    RS_ERR_ALIAS = 3,          /* partially overlapping buffers                        */
    RS_ERR_CUDA = 4,           /* a CUDA runtime call failed                           */
    RS_ERR_DEVICE_TIMEOUT = 5, /* a look-back wait ran out (device error word)         */
    RS_ERR_CHECK_FAILED = 6,   /* a device bounds check failed (device error word)     */
    RS_ERR_UNSUPPORTED = 7     /* valid request this library does not handle           */
} rs_status;

typedef enum rs_key_type {
    RS_U32 = 0, RS_I32 = 1, RS_F32 = 2, RS_U64 = 3,
    RS_U16 = 4, RS_I16 = 5, RS_F16 = 6  /* 16-bit keys; F16 = IEEE binary16 bit patterns */
} rs_key_type;

typedef enum rs_algo {
    RS_ALGO_AUTO = 0,        /* the cluster sort for n <= rs_cluster_max_n(),
                                reduce-then-scan for n >= 2^22 (2^23 for 32-bit
                                keys with values and for 64-bit keys alone;
                                never below 2^30 for 64-bit keys with 64-bit
                                values), the chained scan between (measured
                                on GB300)                                        */
    RS_ALGO_ONESWEEP = 1,    /* one upfront histogram read + one kernel per pass    */
    RS_ALGO_REDUCE_SCAN = 2, /* upsweep + spine scan + downsweep per pass           */
    RS_ALGO_CLUSTER = 3      /* the whole sort in ONE kernel on a thread-block
                                cluster, keys held in distributed shared memory
                                between passes; n <= rs_cluster_max_n(), else
                                RS_ERR_UNSUPPORTED                               */
} rs_algo;

/*
 * Bytes of device scratch ("temp") a sort of this shape needs, for every
 * schedule and digit width, so one temp buffer serves any rs_sort variant.
 * with_values: 0 keys only, 8 uint64 values, any other value uint32 values.
 * Pure host arithmetic: needs no GPU and never fails (0 for n == 0).
 * Returns (size_t)-1 for arguments every sort would reject.
 */
size_t rs_temp_bytes(rs_key_type key_type, int with_values, size_t n, int begin_bit, int end_bit);

/* Keys only.  keys_in: n keys (read only); keys_out: n keys (written). */
rs_status rs_sort_keys_u32(const uint32_t* keys_in, uint32_t* keys_out, size_t n,
                           int begin_bit, int end_bit, void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_keys_i32(const int32_t* keys_in, int32_t* keys_out, size_t n,
                           int begin_bit, int end_bit, void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_keys_f32(const float* keys_in, float* keys_out, size_t n,
                           int begin_bit, int end_bit, void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_keys_u64(const uint64_t* keys_in, uint64_t* keys_out, size_t n,
                           int begin_bit, int end_bit, void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_keys_u16(const uint16_t* keys_in, uint16_t* keys_out, size_t n,
                           int begin_bit, int end_bit, void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_keys_i16(const int16_t* keys_in, int16_t* keys_out, size_t n,
                           int begin_bit, int end_bit, void* temp, size_t temp_bytes, void* stream);
/* binary16 keys as their 16-bit patterns */
rs_status rs_sort_keys_f16(const uint16_t* keys_in, uint16_t* keys_out, size_t n,
                           int begin_bit, int end_bit, void* temp, size_t temp_bytes, void* stream);

/* Keys with one uint32 value each ("Radix sort paralelo sobre el scan": the
 * payload travels with its key).  vals_in / vals_out: n values. */
rs_status rs_sort_pairs_u32(const uint32_t* keys_in, uint32_t* keys_out, const uint32_t* vals_in,
                            uint32_t* vals_out, size_t n, int begin_bit, int end_bit,
                            void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_pairs_i32(const int32_t* keys_in, int32_t* keys_out, const uint32_t* vals_in,
                            uint32_t* vals_out, size_t n, int begin_bit, int end_bit,
                            void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_pairs_f32(const float* keys_in, float* keys_out, const uint32_t* vals_in,
                            uint32_t* vals_out, size_t n, int begin_bit, int end_bit,
                            void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_pairs_u64(const uint64_t* keys_in, uint64_t* keys_out, const uint32_t* vals_in,
                            uint32_t* vals_out, size_t n, int begin_bit, int end_bit,
                            void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_pairs_u16(const uint16_t* keys_in, uint16_t* keys_out, const uint32_t* vals_in,
                            uint32_t* vals_out, size_t n, int begin_bit, int end_bit,
                            void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_pairs_i16(const int16_t* keys_in, int16_t* keys_out, const uint32_t* vals_in,
                            uint32_t* vals_out, size_t n, int begin_bit, int end_bit,
                            void* temp, size_t temp_bytes, void* stream);
rs_status rs_sort_pairs_f16(const uint16_t* keys_in, uint16_t* keys_out, const uint32_t* vals_in,
                            uint32_t* vals_out, size_t n, int begin_bit, int end_bit,
                            void* temp, size_t temp_bytes, void* stream);

/*
 * The general entry point: every typed call above fills one of these.  Fields
 * have the meanings given in the conventions; vals_in / vals_out are both NULL
 * for a keys-only sort.
 */
typedef struct rs_sort_desc {
    rs_key_type key_type;
    const void* keys_in;
    void* keys_out;
    const void* vals_in;   /* n values of value_bytes each, or NULL (keys only) */
    void* vals_out;
    size_t n;
    int begin_bit;
    int end_bit;
    rs_algo algo;       /* schedule, RS_ALGO_AUTO by default                    */
    int radix_bits;     /* digit width: 0 = default (8), or 4 or 8              */
    void* temp;
    size_t temp_bytes;
    void* stream;
    /* Testing hooks, 0 in normal use.  spin_limit bounds each look-back wait
     * (0 = the default bound, about a second).  stall_tile = t + 1 makes tile
     * t of the chained-scan schedule never publish its digit counts, so the
     * waits behind it run out and the sort reports RS_ERR_DEVICE_TIMEOUT. */
    uint32_t spin_limit;
    int32_t stall_tile;
    /* 1: descending order of D (ties still in input order); 0: ascending. */
    int descending;
    /* Bytes per value: 0 or 4 = uint32 values, 8 = uint64 values (ignored
     * for keys only); value pointers must be aligned to it. */
    int value_bytes;
} rs_sort_desc;

rs_status rs_sort(const rs_sort_desc* desc);

/*
 * As rs_sort, and records CUDA events around every kernel: events[0] before
 * the first launch and events[i] after the i-th, on desc->stream.  `events`
 * holds max_events cudaEvent_t handles (as void*) created by the caller.  On
 * return *num_kernels is the number of kernels launched and kinds[i] (if
 * kinds != NULL, max_events entries) names kernel i+1's role:
 *   1 histogram (all passes), 2 chained-scan pass, 3 upsweep, 4 spine scan,
 *   5 downsweep, 6 copy, 7 cluster sort (the whole sort).
 * Returns RS_ERR_INVALID_ARG if max_events is smaller than kernels + 1.
 * While desc->stream is being captured into a CUDA graph the events are
 * recorded as external event nodes, so every replay of the graph records
 * them (per-kernel timing of a replayed graph).
 */
rs_status rs_sort_profiled(const rs_sort_desc* desc, void* const* events, int max_events,
                           int* num_kernels, int* kinds);

/*
 * Largest n the cluster schedule (RS_ALGO_CLUSTER) sorts: 16 CTAs x one tile
 * each -- 65536 32- or 16-bit keys, 49152 of them with uint32 values or
 * uint64 keys, 32768 with uint64 values or uint64 keys with uint32 values,
 * 24576 uint64 keys with uint64 values (with_values as for rs_temp_bytes).  Up to half of that runs on 8 CTAs
 * (the portable cluster size); above it the cluster needs 16, which a device
 * may not schedule: then RS_ALGO_CLUSTER returns RS_ERR_UNSUPPORTED and AUTO
 * takes the chained scan.  No CUDA call; 0 for an invalid key type.
 */
size_t rs_cluster_max_n(rs_key_type key_type, int with_values);

/*
 * Number of kernels rs_sort would launch for this descriptor (no launch).
 * Returns -1 for a descriptor rs_sort would reject.
 */
int rs_sort_kernel_count(const rs_sort_desc* desc);

/*
 * Waits for `stream`, then reads and clears the device error word in `temp`
 * (the last sort enqueued with this temp on this stream).  Returns RS_OK,
 * RS_ERR_DEVICE_TIMEOUT, RS_ERR_CHECK_FAILED, or RS_ERR_CUDA if the wait or
 * the copy fails.  This and rs_skip_record are the only entry points that
 * synchronise.
 */
rs_status rs_device_status(const void* temp, void* stream);

/*
 * Waits for `stream`, then reads the pass-skip record that the last sort
 * enqueued with this temp on this stream left in it (see "Pass skipping"
 * above): *differing_bits = the OR over all keys of T(key) ^ T(keys[0]), so a
 * clear bit is one that every key shares (the high 32 bits are 0 for 32-bit
 * keys); *unordered = 1 if some adjacent pair of keys is out of order in
 * [begin_bit, end_bit), 0 if the input was already sorted (then no pass ran).
 * A pass ran iff unordered and its digit's bits are not all clear.  The
 * record is meaningful after a sort with n > 0 and begin_bit < end_bit.
 * Returns RS_ERR_INVALID_ARG for a NULL pointer, RS_ERR_CUDA if the copy or
 * the wait fails.
 */
rs_status rs_skip_record(const void* temp, void* stream, uint64_t* differing_bits, int* unordered);

/* Static English text for a status code; never NULL. */
const char* rs_status_string(rs_status status);

/*
 * CUDA graph of one whole sort.  rs_graph_create captures rs_sort(desc) on
 * desc->stream (which must not be capturing already) and instantiates it;
 * the graph bakes in every pointer and size of `desc`.  rs_graph_launch
 * replays it on `stream`.  The graph object is host memory owned by the
 * caller until rs_graph_destroy.
 */
typedef struct rs_graph rs_graph;
rs_status rs_graph_create(const rs_sort_desc* desc, rs_graph** graph);
rs_status rs_graph_launch(const rs_graph* graph, void* stream);
void rs_graph_destroy(rs_graph* graph);

/*
 * End-to-end sort of HOST buffers.  h_keys_in / h_vals_in (host, read only,
 * page-locked for full copy speed) are copied to the device, sorted, and the
 * result copied to h_keys_out / h_vals_out (host), all enqueued on `stream`.
 * d_work is a caller-owned device buffer of rs_host_work_bytes(...) bytes
 * holding the device copies and the sort's temp.  The call returns once the
 * work is enqueued; the host outputs are valid after the stream completes.
 */
size_t rs_host_work_bytes(rs_key_type key_type, int with_values, size_t n, int begin_bit,
                          int end_bit);
rs_status rs_sort_host(rs_key_type key_type, const void* h_keys_in, void* h_keys_out,
                       const uint32_t* h_vals_in, uint32_t* h_vals_out, size_t n, int begin_bit,
                       int end_bit, void* d_work, size_t work_bytes, void* stream);

/*
 * End-to-end sort of a sequence of `batches` independent HOST batches of n
 * keys each (same key type and bit range), pipelined: while batch i is
 * sorted on the device, batch i+1 is copied in and batch i-1 copied out, so
 * the host link carries both directions at once.  Batch i reads
 * h_keys_in[i] (and h_vals_in[i]) and writes h_keys_out[i] (and
 * h_vals_out[i]); each result is the same as rs_sort_host's for that batch.
 * The pointer arrays are read during the call only; the host buffers must
 * stay valid (and page-locked for full copy speed) until `stream`
 * completes.  h_vals_in and h_vals_out are both NULL (keys only) or both
 * arrays of non-NULL pointers.  d_work is a caller-owned device buffer of
 * rs_host_batches_work_bytes(...) bytes (two slots of rs_host_work_bytes,
 * used alternately).
 * The work runs on three internal streams forked from and joined back into
 * `stream` (also when an enqueue fails), so the call returns once the work
 * is enqueued and the outputs are valid after `stream` completes.  Not
 * capturable: RS_ERR_UNSUPPORTED while `stream` is capturing.  Errors:
 * RS_ERR_INVALID_ARG (negative batches, a NULL pointer, a bad shape),
 * RS_ERR_TEMP_TOO_SMALL, RS_ERR_CUDA.
 */
size_t rs_host_batches_work_bytes(rs_key_type key_type, int with_values, size_t n, int begin_bit,
                                  int end_bit);
rs_status rs_sort_host_batches(rs_key_type key_type, int batches, const void* const* h_keys_in,
                               void* const* h_keys_out, const uint32_t* const* h_vals_in,
                               uint32_t* const* h_vals_out, size_t n, int begin_bit, int end_bit,
                               void* d_work, size_t work_bytes, void* stream);

/*
 * The binary radix tree over sorted Morton codes: the hierarchy of a linear
 * BVH, the consumer that "高性能计算：GPU上的基数排序" (opening sections)
 * names as the reason to sort on the GPU.  The page stops at the sort; the
 * tree follows the published per-node construction of Karras (2012).
 *
 * sorted_codes: n uint32 codes in ascending order on the device (for example
 * the keys_out of rs_sort_pairs_u32 over Morton codes, whose values_out then
 * maps leaf i back to its primitive).  Equal codes are allowed: leaves are
 * ordered by (code, position), i.e. the tree is the radix tree of the
 * distinct 64-bit keys (code << 32) | position.
 * Outputs (caller-owned device arrays, written in full):
 *   left[n-1], right[n-1]  children of internal node i: an internal node's
 *                          index, or a leaf's index with bit 31 set
 *                          (RS_LBVH_LEAF);
 *   first[n-1], last[n-1]  the leaf range [first, last] internal node i
 *                          covers; one end is always i, and node 0 (the root)
 *                          covers [0, n-1];
 *   leaf_parent[n]         the internal node above each leaf
 *                          (0xFFFFFFFF when n == 1);
 *   node_parent[n-1]       the internal node above each internal node
 *                          (0xFFFFFFFF for the root).
 * A node covering [first, last] splits after the last leaf whose key has a 0
 * in the highest bit where the keys of leaves first and last differ; its left
 * child covers [first, split] (internal node `split` unless that is one
 * leaf), its right child [split + 1, last] (internal node `split + 1` unless
 * one leaf).  One kernel of n - 1 threads, asynchronous on `stream`; no
 * allocation.  Unsorted codes give an unspecified tree, still written within
 * the arrays' bounds.  n == 0: RS_OK, nothing enqueued; n == 1: only
 * leaf_parent[0] is written (the other pointers may be NULL).  Errors:
 * RS_ERR_INVALID_ARG (n > RS_LBVH_MAX_N, a NULL pointer), RS_ERR_CUDA.
 */
#define RS_LBVH_LEAF 0x80000000u
#define RS_LBVH_MAX_N 2147483648u
rs_status rs_lbvh_build(const uint32_t* sorted_codes, size_t n, uint32_t* left, uint32_t* right,
                        uint32_t* first, uint32_t* last, uint32_t* leaf_parent, uint32_t* node_parent,
                        void* stream);

/*
 * Sort without any allocation.  The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory where they
 * sort: code running while a stream capture in global mode is active (where
 * cudaMalloc is not permitted), plugins whose host application owns the
 * device memory pool, and latency-critical loops where cudaMalloc/cudaFree
 * would synchronise the device.
 *
 * Same operation and arguments as rs_sort_keys_u32, but the scratch is a
 * fixed array of RS_NOALLOC_SCRATCH_BYTES (about 21 MiB) of device memory
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  n must be at most RS_NOALLOC_MAX_N (2^22 keys), else
 * RS_ERR_INVALID_ARG is returned and nothing is enqueued.  No cudaMalloc,
 * cudaFree or allocating library routine is called.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  The address is remembered together with the context it belongs
 * to: after cudaDeviceReset (or with another context current) the next call
 * looks it up again, so that call too should come before any capture.
 * Every call shares the one array per device, so calls that overlap on the
 * GPU (on different streams, or from different threads) race; each call
 * clears what must start at zero.  The device error word (a look-back wait
 * that ran out, a failed bounds check) lives in that array and cannot be read
 * back: callers that need that status sort with rs_sort_keys_u32 and their
 * own temp, and read it with rs_device_status.
 */
#define RS_NOALLOC_MAX_N 4194304
#define RS_NOALLOC_SCRATCH_BYTES 22020096
rs_status rs_sort_keys_u32_noalloc(const uint32_t* keys_in, uint32_t* keys_out, size_t n,
                                   int begin_bit, int end_bit, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RS_H */
