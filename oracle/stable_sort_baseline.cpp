// stable_sort_baseline.cpp -- TEST INFRASTRUCTURE ONLY: a single-threaded
// std::stable_sort of the same problem the oracle solves, timed by the bench
// as a CPU baseline beside the oracle and used by the tests as one more
// cross-check.  Linked into the oracle's library; the CUDA library never
// loads it.
//
// The problem ("Radix sort paralelo sobre el scan", section "La idea y el
// requisito de estabilidad"): the stable permutation that orders the bits
// [begin_bit, end_bit) of each key's order-preserving unsigned image, ties in
// input order.  Here that is one comparison sort: the images come from the
// oracle's own map (oracle_ordered_keys), masked to the bit range, and
// std::stable_sort orders (image, index) records by the image alone.
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <thread>
#include <vector>

extern "C" void oracle_ordered_keys(int key_type, const void* keys, size_t n, uint64_t* out);
extern "C" size_t oracle_key_size(int key_type);

namespace {

struct Rec {
    uint64_t d;   // the bits [begin_bit, end_bit) of the ordered key, shifted down
    uint32_t i;   // input position
};

}  // namespace

// Sorts keys (and values, if both value pointers are non-NULL) stably by the
// bit range of the ordered key, ascending, descending = 0, or descending (ties
// still in input order), descending = 1.  Returns 0, or -1 on a bad argument.
extern "C" int cpu_stable_sort(int key_type, const void* keys_in, void* keys_out, const uint32_t* vals_in,
                               uint32_t* vals_out, size_t n, int begin_bit, int end_bit, int descending)
{
    if (key_type < 0 || key_type > 6) return -1;  // u32 i32 f32 u64 u16 i16 f16
    const size_t ks = oracle_key_size(key_type);
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > (int)(8 * ks) || n > 0xFFFFFFFFull)
        return -1;
    std::vector<uint64_t> ordered(n);
    oracle_ordered_keys(key_type, keys_in, n, ordered.data());
    const int width = end_bit - begin_bit;
    const uint64_t mask = width >= 64 ? ~0ull : ((1ull << width) - 1ull);
    std::vector<Rec> r(n);
    for (size_t i = 0; i < n; ++i) r[i] = Rec{begin_bit >= 64 ? 0ull : (ordered[i] >> begin_bit) & mask, (uint32_t)i};
    if (descending)
        std::stable_sort(r.begin(), r.end(), [](const Rec& a, const Rec& b) { return a.d > b.d; });
    else
        std::stable_sort(r.begin(), r.end(), [](const Rec& a, const Rec& b) { return a.d < b.d; });
    const unsigned char* src = static_cast<const unsigned char*>(keys_in);
    unsigned char* dst = static_cast<unsigned char*>(keys_out);
    for (size_t j = 0; j < n; ++j) std::memcpy(dst + j * ks, src + (size_t)r[j].i * ks, ks);
    if (vals_in && vals_out)
        for (size_t j = 0; j < n; ++j) vals_out[j] = vals_in[r[j].i];
    return 0;
}

// The host's hardware thread count as the C++ runtime reports it.
extern "C" unsigned cpu_hardware_concurrency() { return std::thread::hardware_concurrency(); }
