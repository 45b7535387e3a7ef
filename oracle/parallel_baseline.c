/* parallel_baseline.c -- TEST INFRASTRUCTURE ONLY: a multi-threaded CPU LSD
 * radix sort, timed by the bench beside the single-threaded baselines so that
 * the GPU is also compared with the whole host, and checked by the tests
 * against the oracle.  Linked into the oracle's library; the CUDA library
 * never loads it.  Built with OpenMP when the compiler has it, else it runs
 * on one thread (cpu_parallel_threads() says which).
 *
 * Each pass of 8-bit digits over [begin_bit, end_bit) of the order-preserving
 * key (the oracle's map, oracle_ordered_key) is the scheme of "Radix sort
 * paralelo sobre el scan" (section "Las tres fases de una pasada") with one
 * block per thread: every thread counts the digits of its contiguous block,
 * the counts are scanned in digit-major order (digit d of thread t starts
 * after every smaller digit of every thread and after digit d of threads
 * 0..t-1), and every thread then places its block's keys in order, so each
 * pass is stable.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

uint64_t oracle_ordered_key(int key_type, uint64_t raw);
size_t oracle_key_size(int key_type);

static uint64_t load_key(const void* a, size_t ks, size_t i)
{
    switch (ks) {
    case 8: return ((const uint64_t*)a)[i];
    case 2: return ((const uint16_t*)a)[i];
    default: return ((const uint32_t*)a)[i];
    }
}

static void store_key(void* a, size_t ks, size_t i, uint64_t v)
{
    switch (ks) {
    case 8: ((uint64_t*)a)[i] = v; break;
    case 2: ((uint16_t*)a)[i] = (uint16_t)v; break;
    default: ((uint32_t*)a)[i] = (uint32_t)v; break;
    }
}

int cpu_parallel_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Returns 0, or -1 on a bad argument or when memory runs out. */
int cpu_parallel_lsd_sort(int key_type, const void* keys_in, void* keys_out, const uint32_t* vals_in,
                          uint32_t* vals_out, size_t n, int begin_bit, int end_bit, int threads)
{
    if (key_type < 0 || key_type > 6) return -1;
    const size_t ks = oracle_key_size(key_type);
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > (int)(8 * ks)) return -1;
    const int with_vals = vals_in != NULL && vals_out != NULL;
    if (threads < 1) threads = 1;
    memcpy(keys_out, keys_in, n * ks);
    if (with_vals) memcpy(vals_out, vals_in, n * sizeof(uint32_t));
    if (n == 0 || end_bit == begin_bit) return 0;
    void* tk = malloc(n * ks);
    uint32_t* tv = with_vals ? (uint32_t*)malloc(n * sizeof(uint32_t)) : NULL;
    size_t* counts = (size_t*)malloc((size_t)threads * 256 * sizeof(size_t));
    if (!tk || (with_vals && !tv) || !counts) {
        free(tk);
        free(tv);
        free(counts);
        return -1;
    }
    void* src = keys_out;
    void* dst = tk;
    uint32_t* vsrc = with_vals ? vals_out : NULL;
    uint32_t* vdst = tv;
    for (int lo = begin_bit; lo < end_bit; lo += 8) {
        const int width = end_bit - lo < 8 ? end_bit - lo : 8;
        const uint64_t mask = ((uint64_t)1 << width) - 1;
#ifdef _OPENMP
#pragma omp parallel num_threads(threads)
#endif
        {
#ifdef _OPENMP
            const int t = omp_get_thread_num(), T = omp_get_num_threads();
#else
            const int t = 0, T = 1;
#endif
            const size_t b0 = n * (size_t)t / (size_t)T, b1 = n * (size_t)(t + 1) / (size_t)T;
            size_t* c = counts + (size_t)t * 256;
            memset(c, 0, 256 * sizeof(size_t));
            for (size_t i = b0; i < b1; ++i)
                c[(oracle_ordered_key(key_type, load_key(src, ks, i)) >> lo) & mask] += 1;
#ifdef _OPENMP
#pragma omp barrier
#pragma omp single
#endif
            {
                size_t run = 0;
                for (int d = 0; d < 256; ++d)
                    for (int u = 0; u < T; ++u) {
                        const size_t x = counts[(size_t)u * 256 + d];
                        counts[(size_t)u * 256 + d] = run;
                        run += x;
                    }
            }
            for (size_t i = b0; i < b1; ++i) {
                const uint64_t k = load_key(src, ks, i);
                const size_t pos = c[(oracle_ordered_key(key_type, k) >> lo) & mask]++;
                store_key(dst, ks, pos, k);
                if (with_vals) vdst[pos] = vsrc[i];
            }
        }
        void* sw = src;
        src = dst;
        dst = sw;
        uint32_t* vsw = vsrc;
        vsrc = vdst;
        vdst = vsw;
    }
    if (src != keys_out) {
        memcpy(keys_out, src, n * ks);
        if (with_vals) memcpy(vals_out, vsrc, n * sizeof(uint32_t));
    }
    free(tk);
    free(tv);
    free(counts);
    return 0;
}
