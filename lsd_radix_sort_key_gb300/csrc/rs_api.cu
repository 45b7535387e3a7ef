// rs_api.cu -- the extern "C" boundary declared in include/rs.h: argument
// checks, the temp layout, schedule choice, profiling events, CUDA graphs and
// the host-buffer path.  The kernels live in rs_kernels.cuh and are
// instantiated per key type in rs_sort_<type>.cu.
#include <cuda_runtime.h>
#include <stdint.h>

#include <new>

#include "rs.h"
#include "rs_config.h"
#include "rs_kernels.cuh"

// Instantiated in rs_sort_<type>.cu; not here.
namespace rs {
extern template rs_status run_sort<KU32>(Plan& pl);
extern template rs_status run_sort<KI32>(Plan& pl);
extern template rs_status run_sort<KF32>(Plan& pl);
extern template rs_status run_sort<KU64>(Plan& pl);
extern template rs_status run_sort<KU16>(Plan& pl);
extern template rs_status run_sort<KI16>(Plan& pl);
extern template rs_status run_sort<KF16>(Plan& pl);
}  // namespace rs

namespace {

constexpr size_t kMaxN = (size_t)RS_MAX_N;           // 2^32 - 2^16
constexpr size_t kOnesweepMaxN = ((size_t)1 << 30) - 1;
// AUTO's smallest reduce-then-scan size for kb-byte keys with vb-byte values
// (0: none), from graph-replay timings on GB300 (ms per sort, chained scan vs
// reduce-then-scan): 32-bit keys alone tie at 2^22 (0.105 either way);
// 32-bit keys with values and 64-bit keys alone lose with reduce-then-scan at
// 2^22 (u32 + u32: 0.132 vs 0.139; u32 + u64: 0.157 vs 0.161; u64: 0.249 vs
// 0.287) and win with it from 2^24 (0.419 vs 0.432; 0.541 vs 0.554; 0.800
// vs 0.828); 64-bit keys with 64-bit values win with the chained scan at every
// size from 2^24 on (2^28: 21.33 vs 21.86) and tie at 2^22.
size_t auto_reduce_scan_min_n(int kb, int vb)
{
    if (kb == 8 && vb == 8) return kOnesweepMaxN + 1;
    if ((kb == 8 && vb == 0) || (kb == 4 && vb != 0)) return (size_t)1 << 23;
    return (size_t)1 << 22;
}
constexpr uint32_t kDefaultSpinLimit = 1u << 20;      // each spin is one L2 round trip (~1 s in all)

int key_bytes(rs_key_type kt) { return kt == RS_U64 ? 8 : kt >= RS_U16 ? 2 : 4; }
int key_bits(rs_key_type kt) { return 8 * key_bytes(kt); }
bool valid_kt(int kt) { return kt >= RS_U32 && kt <= RS_F16; }
// rs_temp_bytes / rs_cluster_max_n take with_values: 0 none, 8 uint64, else uint32.
int value_bytes_of(int with_values) { return with_values == 0 ? 0 : with_values == 8 ? 8 : 4; }

bool ranges_overlap(const void* a, size_t abytes, const void* b, size_t bbytes)
{
    if (!a || !b || abytes == 0 || bbytes == 0) return false;
    uintptr_t a0 = (uintptr_t)a, a1 = a0 + abytes, b0 = (uintptr_t)b, b1 = b0 + bbytes;
    return a0 < b1 && b0 < a1;
}

rs_status check_shape(rs_key_type kt, size_t n, int begin_bit, int end_bit)
{
    if (!valid_kt(kt)) return RS_ERR_INVALID_ARG;
    if (n > kMaxN) return RS_ERR_INVALID_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > key_bits(kt)) return RS_ERR_INVALID_ARG;
    return RS_OK;
}

// Validates a descriptor and resolves it into a Plan (no CUDA call).
rs_status make_plan(const rs_sort_desc* d, rs::Plan* pl)
{
    if (!d) return RS_ERR_INVALID_ARG;
    rs_status st = check_shape(d->key_type, d->n, d->begin_bit, d->end_bit);
    if (st != RS_OK) return st;
    const bool vals = d->vals_in != nullptr || d->vals_out != nullptr;
    if (vals && (!d->vals_in || !d->vals_out)) return RS_ERR_INVALID_ARG;
    if (d->value_bytes != 0 && d->value_bytes != 4 && d->value_bytes != 8) return RS_ERR_INVALID_ARG;
    const int vb = vals ? (d->value_bytes == 8 ? 8 : 4) : 0;
    if (d->radix_bits != 0 && d->radix_bits != 4 && d->radix_bits != 8) return RS_ERR_INVALID_ARG;
    if (d->algo != RS_ALGO_AUTO && d->algo != RS_ALGO_ONESWEEP && d->algo != RS_ALGO_REDUCE_SCAN &&
        d->algo != RS_ALGO_CLUSTER)
        return RS_ERR_INVALID_ARG;
    if (d->stall_tile < 0) return RS_ERR_INVALID_ARG;
    if (d->descending != 0 && d->descending != 1) return RS_ERR_INVALID_ARG;
    const size_t n = d->n;
    const int kb = key_bytes(d->key_type);
    *pl = rs::Plan{};
    pl->kt = d->key_type;
    pl->vals = vals;
    pl->vb = vb;
    pl->n = n;
    pl->begin_bit = d->begin_bit;
    pl->end_bit = d->end_bit;
    pl->radix_bits = d->radix_bits == 0 ? 8 : d->radix_bits;
    pl->descending = d->descending != 0;
    pl->passes = rs::passes_for(d->begin_bit, d->end_bit, pl->radix_bits);
    pl->algo = d->algo;
    const size_t cluster_max = rs::cluster_max_n(kb, vb);
    if (pl->algo == RS_ALGO_AUTO) {
        // Chosen by measurement on GB300: one cluster kernel while the keys fit
        // in the cluster's shared memory; reduce-then-scan from 2^22 or 2^23
        // keys, by shape (from there on it beats the chained scan
        // host-launched and graph-replayed, its 12 kernels' launches hidden by
        // programmatic dependent launch; below, the chained scan's 5 kernels
        // win); the chained scan between.  The chained scan needs n < 2^30.
        const bool rts = n > kOnesweepMaxN || n >= auto_reduce_scan_min_n(kb, vb);
        pl->algo = n <= cluster_max ? RS_ALGO_CLUSTER : rts ? RS_ALGO_REDUCE_SCAN : RS_ALGO_ONESWEEP;
        pl->auto_chosen = true;
    }
    if (pl->algo == RS_ALGO_ONESWEEP && n > kOnesweepMaxN) return RS_ERR_UNSUPPORTED;
    if (pl->algo == RS_ALGO_CLUSTER && n > cluster_max) return RS_ERR_UNSUPPORTED;
    pl->keys_in = d->keys_in;
    pl->keys_out = d->keys_out;
    pl->vals_in = d->vals_in;
    pl->vals_out = d->vals_out;
    pl->temp = static_cast<unsigned char*>(d->temp);
    pl->stream = static_cast<cudaStream_t>(d->stream);
    pl->spin_limit = d->spin_limit ? d->spin_limit : kDefaultSpinLimit;
    pl->stall_tile = d->stall_tile;
    if (n == 0) return RS_OK;

    if (!d->keys_in || !d->keys_out || !d->temp) return RS_ERR_INVALID_ARG;
    if ((uintptr_t)d->keys_in % kb || (uintptr_t)d->keys_out % kb) return RS_ERR_INVALID_ARG;
    if (vals && ((uintptr_t)d->vals_in % vb || (uintptr_t)d->vals_out % vb)) return RS_ERR_INVALID_ARG;
    if ((uintptr_t)d->temp % 256) return RS_ERR_INVALID_ARG;
    pl->lay = rs::temp_layout(kb, vb, n, d->begin_bit, d->end_bit);
    if (d->temp_bytes < pl->lay.total) return RS_ERR_TEMP_TOO_SMALL;

    // Aliasing: exact in-place is allowed; any other overlap is rejected.
    const size_t kbytes = n * kb, vbytes = n * (size_t)vb;
    const void* bufs[5] = {d->keys_in, d->keys_out, d->vals_in, d->vals_out, d->temp};
    const size_t sizes[5] = {kbytes, kbytes, vals ? vbytes : 0, vals ? vbytes : 0, pl->lay.total};
    for (int i = 0; i < 5; ++i)
        for (int j = i + 1; j < 5; ++j) {
            const bool same_exact = bufs[i] == bufs[j] && sizes[i] == sizes[j];
            const bool allowed = same_exact && ((i == 0 && j == 1) || (i == 2 && j == 3));
            if (!allowed && ranges_overlap(bufs[i], sizes[i], bufs[j], sizes[j])) return RS_ERR_ALIAS;
        }
    if (vals && (d->keys_in == d->keys_out) != (d->vals_in == d->vals_out)) return RS_ERR_ALIAS;
    return RS_OK;
}

rs_status dispatch(rs::Plan& pl)
{
    switch (pl.kt) {
    case RS_U32: return rs::run_sort<rs::KU32>(pl);
    case RS_I32: return rs::run_sort<rs::KI32>(pl);
    case RS_F32: return rs::run_sort<rs::KF32>(pl);
    case RS_U16: return rs::run_sort<rs::KU16>(pl);
    case RS_I16: return rs::run_sort<rs::KI16>(pl);
    case RS_F16: return rs::run_sort<rs::KF16>(pl);
    default:     return rs::run_sort<rs::KU64>(pl);
    }
}

// Enqueue a whole sort described by `pl` (already validated).
rs_status enqueue(rs::Plan& pl)
{
    if (pl.n == 0) return RS_OK;
    if (pl.count_only) {
        if (pl.passes == 0) { pl.launched = 0; return RS_OK; }
        return dispatch(pl);
    }
    // Clear the error word, the tile tickets and the global histograms.
    if (cudaMemsetAsync(pl.temp + pl.lay.meta, 0, rs::kMetaWords * 4, pl.stream) != cudaSuccess)
        return RS_ERR_CUDA;
    if (pl.passes == 0) {  // empty bit range: a stable sort is the identity
        if (pl.keys_out != pl.keys_in &&
            cudaMemcpyAsync(pl.keys_out, pl.keys_in, pl.n * key_bytes((rs_key_type)pl.kt),
                            cudaMemcpyDeviceToDevice, pl.stream) != cudaSuccess)
            return RS_ERR_CUDA;
        if (pl.vals && pl.vals_out != pl.vals_in &&
            cudaMemcpyAsync(pl.vals_out, pl.vals_in, pl.n * (size_t)pl.vb, cudaMemcpyDeviceToDevice, pl.stream) !=
                cudaSuccess)
            return RS_ERR_CUDA;
        return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
    }
    return dispatch(pl);
}

}  // namespace

extern "C" {

size_t rs_temp_bytes(rs_key_type key_type, int with_values, size_t n, int begin_bit, int end_bit)
{
    if (check_shape(key_type, n, begin_bit, end_bit) != RS_OK) return (size_t)-1;
    if (n == 0) return 0;
    return rs::temp_layout(key_bytes(key_type), value_bytes_of(with_values), n, begin_bit, end_bit).total;
}

rs_status rs_sort(const rs_sort_desc* desc)
{
    rs::Plan pl;
    rs_status st = make_plan(desc, &pl);
    if (st != RS_OK) return st;
    return enqueue(pl);
}

int rs_sort_kernel_count(const rs_sort_desc* desc)
{
    if (!desc) return -1;
    // The count depends on the shape only: stand in distinct, never
    // dereferenced addresses for any missing buffer so the checks pass.
    rs_sort_desc d = *desc;
    const bool vals = d.vals_in || d.vals_out;
    if (!d.keys_in) d.keys_in = reinterpret_cast<const void*>((uintptr_t)1 << 40);
    if (!d.keys_out) d.keys_out = reinterpret_cast<void*>((uintptr_t)2 << 40);
    if (vals && !d.vals_in) d.vals_in = reinterpret_cast<const void*>((uintptr_t)3 << 40);
    if (vals && !d.vals_out) d.vals_out = reinterpret_cast<void*>((uintptr_t)4 << 40);
    if (!d.temp) {
        d.temp = reinterpret_cast<void*>((uintptr_t)5 << 40);
        d.temp_bytes = (size_t)1 << 40;
    }
    rs::Plan pl;
    if (make_plan(&d, &pl) != RS_OK) return -1;
    pl.count_only = true;
    if (enqueue(pl) != RS_OK) return -1;
    return pl.launched;
}

rs_status rs_sort_profiled(const rs_sort_desc* desc, void* const* events, int max_events,
                           int* num_kernels, int* kinds)
{
    if (!events || !num_kernels) return RS_ERR_INVALID_ARG;
    int need = rs_sort_kernel_count(desc);
    if (need < 0) return RS_ERR_INVALID_ARG;
    if (max_events < need + 1) return RS_ERR_INVALID_ARG;
    rs::Plan pl;
    rs_status st = make_plan(desc, &pl);
    if (st != RS_OK) return st;
    pl.events = reinterpret_cast<cudaEvent_t const*>(events);
    pl.max_events = max_events;
    pl.kinds = kinds;
    // Inside a stream capture a plain event record only orders the capture;
    // an external record becomes a graph node that records at every replay.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(pl.stream, &cs) != cudaSuccess) return RS_ERR_CUDA;
    pl.event_flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    if (cudaEventRecordWithFlags(pl.events[0], pl.stream, pl.event_flags) != cudaSuccess) return RS_ERR_CUDA;
    st = enqueue(pl);
    *num_kernels = pl.launched;
    return st;
}

#define RS_TYPED(NAME, KT, KTYPE)                                                                   \
    rs_status rs_sort_keys_##NAME(const KTYPE* keys_in, KTYPE* keys_out, size_t n, int begin_bit,   \
                                  int end_bit, void* temp, size_t temp_bytes, void* stream)         \
    {                                                                                               \
        rs_sort_desc d{};                                                                           \
        d.key_type = KT;                                                                            \
        d.keys_in = keys_in;                                                                        \
        d.keys_out = keys_out;                                                                      \
        d.n = n;                                                                                    \
        d.begin_bit = begin_bit;                                                                    \
        d.end_bit = end_bit;                                                                        \
        d.temp = temp;                                                                              \
        d.temp_bytes = temp_bytes;                                                                  \
        d.stream = stream;                                                                          \
        return rs_sort(&d);                                                                         \
    }                                                                                               \
    rs_status rs_sort_pairs_##NAME(const KTYPE* keys_in, KTYPE* keys_out, const uint32_t* vals_in,  \
                                   uint32_t* vals_out, size_t n, int begin_bit, int end_bit,        \
                                   void* temp, size_t temp_bytes, void* stream)                     \
    {                                                                                               \
        if (n > 0 && (!vals_in || !vals_out)) return RS_ERR_INVALID_ARG;                            \
        rs_sort_desc d{};                                                                           \
        d.key_type = KT;                                                                            \
        d.keys_in = keys_in;                                                                        \
        d.keys_out = keys_out;                                                                      \
        d.vals_in = vals_in;                                                                        \
        d.vals_out = vals_out;                                                                      \
        d.n = n;                                                                                    \
        d.begin_bit = begin_bit;                                                                    \
        d.end_bit = end_bit;                                                                        \
        d.temp = temp;                                                                              \
        d.temp_bytes = temp_bytes;                                                                  \
        d.stream = stream;                                                                          \
        return rs_sort(&d);                                                                         \
    }

RS_TYPED(u32, RS_U32, uint32_t)
RS_TYPED(i32, RS_I32, int32_t)
RS_TYPED(f32, RS_F32, float)
RS_TYPED(u64, RS_U64, uint64_t)
RS_TYPED(u16, RS_U16, uint16_t)
RS_TYPED(i16, RS_I16, int16_t)
RS_TYPED(f16, RS_F16, uint16_t)
#undef RS_TYPED

rs_status rs_device_status(const void* temp, void* stream)
{
    if (!temp) return RS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* err = reinterpret_cast<uint32_t*>(const_cast<void*>(temp)) + rs::kErrWord;
    uint32_t word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
    if (cudaMemcpyAsync(&word, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return RS_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess) return RS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
    if (word & (1u << RS_ERR_DEVICE_TIMEOUT)) return RS_ERR_DEVICE_TIMEOUT;
    if (word) return RS_ERR_CHECK_FAILED;
    return RS_OK;
}

size_t rs_cluster_max_n(rs_key_type key_type, int with_values)
{
    if (!valid_kt(key_type)) return 0;
    return rs::cluster_max_n(key_bytes(key_type), value_bytes_of(with_values));
}

rs_status rs_skip_record(const void* temp, void* stream, uint64_t* differing_bits, int* unordered)
{
    if (!temp || !differing_bits || !unordered) return RS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint32_t* rec = reinterpret_cast<const uint32_t*>(temp) + rs::kSkipBase;
    uint32_t w[3] = {0, 0, 0};
    if (cudaMemcpyAsync(w, rec, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess) return RS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
    *differing_bits = ((uint64_t)w[1] << 32) | w[0];
    *unordered = w[2] != 0u ? 1 : 0;
    return RS_OK;
}

const char* rs_status_string(rs_status status)
{
    switch (status) {
    case RS_OK: return "ok";
    case RS_ERR_INVALID_ARG: return "invalid argument";
    case RS_ERR_TEMP_TOO_SMALL: return "temp buffer smaller than rs_temp_bytes()";
    case RS_ERR_ALIAS: return "buffers overlap";
    case RS_ERR_CUDA: return "CUDA runtime call failed";
    case RS_ERR_DEVICE_TIMEOUT: return "device look-back wait ran out";
    case RS_ERR_CHECK_FAILED: return "device bounds check failed";
    case RS_ERR_UNSUPPORTED: return "unsupported request";
    }
    return "unknown status";
}

struct rs_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

rs_status rs_graph_create(const rs_sort_desc* desc, rs_graph** graph)
{
    if (!desc || !graph) return RS_ERR_INVALID_ARG;
    *graph = nullptr;
    rs::Plan pl;
    rs_status st = make_plan(desc, &pl);
    if (st != RS_OK) return st;
    cudaStream_t cap = nullptr;
    if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) return RS_ERR_CUDA;
    pl.stream = cap;
    rs_graph g{nullptr, nullptr};
    if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(cap);
        return RS_ERR_CUDA;
    }
    st = enqueue(pl);
    cudaError_t e = cudaStreamEndCapture(cap, &g.graph);
    cudaStreamDestroy(cap);
    if (st != RS_OK || e != cudaSuccess) {
        if (g.graph) cudaGraphDestroy(g.graph);
        return st != RS_OK ? st : RS_ERR_CUDA;
    }
    if (cudaGraphInstantiate(&g.exec, g.graph, 0) != cudaSuccess) {
        cudaGraphDestroy(g.graph);
        return RS_ERR_CUDA;
    }
    rs_graph* out = new (std::nothrow) rs_graph(g);
    if (!out) {
        cudaGraphExecDestroy(g.exec);
        cudaGraphDestroy(g.graph);
        return RS_ERR_CUDA;
    }
    *graph = out;
    return RS_OK;
}

rs_status rs_graph_launch(const rs_graph* graph, void* stream)
{
    if (!graph) return RS_ERR_INVALID_ARG;
    return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? RS_OK
                                                                                          : RS_ERR_CUDA;
}

void rs_graph_destroy(rs_graph* graph)
{
    if (!graph) return;
    cudaGraphExecDestroy(graph->exec);
    cudaGraphDestroy(graph->graph);
    delete graph;
}

// Host path work buffer: [temp][keys in][keys out][vals in][vals out].
static rs::TempLayout host_work_layout(rs_key_type kt, bool vals, size_t n, int begin_bit, int end_bit,
                                       size_t* kin, size_t* kout, size_t* vin, size_t* vout)
{
    rs::TempLayout t = rs::temp_layout(key_bytes(kt), vals ? 4 : 0, n, begin_bit, end_bit);
    size_t off = t.total;
    const size_t kb = rs::align_up(n * key_bytes(kt), 256), vb = vals ? rs::align_up(n * 4, 256) : 0;
    *kin = off; off += kb;
    *kout = off; off += kb;
    *vin = off; off += vb;
    *vout = off; off += vb;
    t.total = off;  // whole work buffer
    return t;
}

size_t rs_host_work_bytes(rs_key_type key_type, int with_values, size_t n, int begin_bit, int end_bit)
{
    if (check_shape(key_type, n, begin_bit, end_bit) != RS_OK) return (size_t)-1;
    if (n == 0) return 0;
    size_t a, b, c, d;
    return host_work_layout(key_type, with_values != 0, n, begin_bit, end_bit, &a, &b, &c, &d).total;
}

rs_status rs_sort_host(rs_key_type key_type, const void* h_keys_in, void* h_keys_out,
                       const uint32_t* h_vals_in, uint32_t* h_vals_out, size_t n, int begin_bit,
                       int end_bit, void* d_work, size_t work_bytes, void* stream)
{
    rs_status st = check_shape(key_type, n, begin_bit, end_bit);
    if (st != RS_OK) return st;
    if (n == 0) return RS_OK;
    const bool vals = h_vals_in || h_vals_out;
    if (!h_keys_in || !h_keys_out || !d_work || (vals && (!h_vals_in || !h_vals_out)))
        return RS_ERR_INVALID_ARG;
    size_t kin, kout, vin, vout;
    rs::TempLayout t = host_work_layout(key_type, vals, n, begin_bit, end_bit, &kin, &kout, &vin, &vout);
    if (work_bytes < t.total) return RS_ERR_TEMP_TOO_SMALL;
    unsigned char* w = static_cast<unsigned char*>(d_work);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t kb = n * key_bytes(key_type);
    if (cudaMemcpyAsync(w + kin, h_keys_in, kb, cudaMemcpyHostToDevice, s) != cudaSuccess) return RS_ERR_CUDA;
    if (vals && cudaMemcpyAsync(w + vin, h_vals_in, n * 4, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return RS_ERR_CUDA;
    rs_sort_desc d{};
    d.key_type = key_type;
    d.keys_in = w + kin;
    d.keys_out = w + kout;
    d.vals_in = vals ? static_cast<const void*>(w + vin) : nullptr;
    d.vals_out = vals ? static_cast<void*>(w + vout) : nullptr;
    d.n = n;
    d.begin_bit = begin_bit;
    d.end_bit = end_bit;
    d.temp = w;
    d.temp_bytes = rs::temp_layout(key_bytes(key_type), vals ? 4 : 0, n, begin_bit, end_bit).total;
    d.stream = stream;
    st = rs_sort(&d);
    if (st != RS_OK) return st;
    if (cudaMemcpyAsync(h_keys_out, w + kout, kb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return RS_ERR_CUDA;
    if (vals && cudaMemcpyAsync(h_vals_out, w + vout, n * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RS_ERR_CUDA;
    return RS_OK;
}

size_t rs_host_batches_work_bytes(rs_key_type key_type, int with_values, size_t n, int begin_bit,
                                  int end_bit)
{
    const size_t one = rs_host_work_bytes(key_type, with_values, n, begin_bit, end_bit);
    if (one == (size_t)-1 || one == 0) return one;
    return 2 * rs::align_up(one, 256);
}

}  // extern "C"

namespace {

// The streams and events of one rs_sort_host_batches call.  Destroying them
// while their work is still pending is allowed: CUDA releases them once the
// work completes.
struct BatchPipe {
    cudaStream_t sh = nullptr, sc = nullptr, sd = nullptr;  // copies in, sorts, copies out
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaEvent_t in_done[2] = {}, sort_done[2] = {}, out_done[2] = {};
    bool create()
    {
        const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&sh, sf) != cudaSuccess || cudaStreamCreateWithFlags(&sc, sf) != cudaSuccess ||
            cudaStreamCreateWithFlags(&sd, sf) != cudaSuccess)
            return false;
        if (cudaEventCreateWithFlags(&fork, ef) != cudaSuccess || cudaEventCreateWithFlags(&join, ef) != cudaSuccess)
            return false;
        for (int s = 0; s < 2; ++s)
            if (cudaEventCreateWithFlags(&in_done[s], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&sort_done[s], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&out_done[s], ef) != cudaSuccess)
                return false;
        return true;
    }
    ~BatchPipe()
    {
        for (cudaStream_t s : {sh, sc, sd})
            if (s) cudaStreamDestroy(s);
        for (cudaEvent_t e : {fork, join, in_done[0], in_done[1], sort_done[0], sort_done[1], out_done[0], out_done[1]})
            if (e) cudaEventDestroy(e);
    }
};

}  // namespace

extern "C" {

rs_status rs_sort_host_batches(rs_key_type key_type, int batches, const void* const* h_keys_in,
                               void* const* h_keys_out, const uint32_t* const* h_vals_in,
                               uint32_t* const* h_vals_out, size_t n, int begin_bit, int end_bit,
                               void* d_work, size_t work_bytes, void* stream)
{
    rs_status st = check_shape(key_type, n, begin_bit, end_bit);
    if (st != RS_OK) return st;
    if (batches < 0 || (batches > 0 && (!h_keys_in || !h_keys_out))) return RS_ERR_INVALID_ARG;
    const bool vals = h_vals_in || h_vals_out;
    if (vals && (!h_vals_in || !h_vals_out)) return RS_ERR_INVALID_ARG;
    for (int i = 0; i < batches; ++i)
        if (!h_keys_in[i] || !h_keys_out[i] || (vals && (!h_vals_in[i] || !h_vals_out[i])))
            return RS_ERR_INVALID_ARG;
    if (n == 0 || batches == 0) return RS_OK;
    if (!d_work) return RS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return RS_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return RS_ERR_UNSUPPORTED;

    size_t kin, kout, vin, vout;
    const rs::TempLayout t = host_work_layout(key_type, vals, n, begin_bit, end_bit, &kin, &kout, &vin, &vout);
    const size_t slot_bytes = rs::align_up(t.total, 256);
    if (work_bytes < 2 * slot_bytes) return RS_ERR_TEMP_TOO_SMALL;
    const size_t kb = n * key_bytes(key_type), vbytes = n * 4;
    const size_t sort_temp = rs::temp_layout(key_bytes(key_type), vals ? 4 : 0, n, begin_bit, end_bit).total;

    BatchPipe bp;
    if (!bp.create()) return RS_ERR_CUDA;
    if (cudaEventRecord(bp.fork, s) != cudaSuccess) return RS_ERR_CUDA;
    for (cudaStream_t x : {bp.sh, bp.sc, bp.sd})
        if (cudaStreamWaitEvent(x, bp.fork, 0) != cudaSuccess) return RS_ERR_CUDA;

    // Batch i uses slot i % 2.  Its copy in waits for the sort of batch i-2
    // (the slot's input buffer), its sort for its copy in and for the copy
    // out of batch i-2 (the slot's output buffer and temp), its copy out for
    // its sort.  Each wait is enqueued after the record it refers to and
    // before that event is recorded again.
    st = RS_OK;
    for (int i = 0; i < batches && st == RS_OK; ++i) {
        const int k = i & 1;
        unsigned char* w = static_cast<unsigned char*>(d_work) + k * slot_bytes;
        bool ok = true;
        if (i >= 2) ok = ok && cudaStreamWaitEvent(bp.sh, bp.sort_done[k], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(w + kin, h_keys_in[i], kb, cudaMemcpyHostToDevice, bp.sh) == cudaSuccess;
        if (vals) ok = ok && cudaMemcpyAsync(w + vin, h_vals_in[i], vbytes, cudaMemcpyHostToDevice, bp.sh) == cudaSuccess;
        ok = ok && cudaEventRecord(bp.in_done[k], bp.sh) == cudaSuccess;
        ok = ok && cudaStreamWaitEvent(bp.sc, bp.in_done[k], 0) == cudaSuccess;
        if (i >= 2) ok = ok && cudaStreamWaitEvent(bp.sc, bp.out_done[k], 0) == cudaSuccess;
        if (!ok) { st = RS_ERR_CUDA; break; }
        rs_sort_desc d{};
        d.key_type = key_type;
        d.keys_in = w + kin;
        d.keys_out = w + kout;
        d.vals_in = vals ? static_cast<const void*>(w + vin) : nullptr;
        d.vals_out = vals ? static_cast<void*>(w + vout) : nullptr;
        d.n = n;
        d.begin_bit = begin_bit;
        d.end_bit = end_bit;
        d.temp = w;
        d.temp_bytes = sort_temp;
        d.stream = bp.sc;
        st = rs_sort(&d);
        if (st != RS_OK) break;
        ok = cudaEventRecord(bp.sort_done[k], bp.sc) == cudaSuccess;
        ok = ok && cudaStreamWaitEvent(bp.sd, bp.sort_done[k], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(h_keys_out[i], w + kout, kb, cudaMemcpyDeviceToHost, bp.sd) == cudaSuccess;
        if (vals) ok = ok && cudaMemcpyAsync(h_vals_out[i], w + vout, vbytes, cudaMemcpyDeviceToHost, bp.sd) == cudaSuccess;
        ok = ok && cudaEventRecord(bp.out_done[k], bp.sd) == cudaSuccess;
        if (!ok) st = RS_ERR_CUDA;
    }
    // Join everything enqueued so far back into the caller's stream, also on
    // an error, so that a sync of `stream` covers it.
    bool joined = true;
    for (cudaStream_t x : {bp.sh, bp.sc, bp.sd}) {
        joined = joined && cudaEventRecord(bp.join, x) == cudaSuccess &&
                 cudaStreamWaitEvent(s, bp.join, 0) == cudaSuccess;
    }
    if (!joined && st == RS_OK) st = RS_ERR_CUDA;
    return st;
}

}  // extern "C"
