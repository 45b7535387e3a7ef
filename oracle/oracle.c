/*
 * oracle.c -- CPU oracle for the stable least-significant-digit radix sort.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's CPU
 * baseline call it; the CUDA library never includes, links or calls it, and
 * it shares no code with the CUDA library.  It is plain, single-threaded,
 * deliberately unoptimised C whose steps follow the pages it cites:
 *
 *   [P1] "Radix sort を実装 & 測定してみた" (Silicon Studio blog)
 *   [P2] "Radix sort paralelo sobre el scan" (wandres.dev WebGPU guide)
 *   [P3] "정렬: 라딕스와 머지소트" (PMPP chapter 13 notes)
 *   [P5] "高性能计算：GPU上的基数排序" (OnikataHoshio)
 *
 * What it computes: for key type t and bit range [begin, end) the unique
 * stable permutation that orders D(i) = bits [begin, end) of the ordered key
 * T_t(key_i) ascending (or descending), ties kept in input order.  Output keys
 * are the original bit patterns; output values follow their keys.
 *
 * Readings of the pages taken here (each pinned by the tests):
 *  - int32: the order-preserving map is the sign-bit flip of [P2] "Claves con
 *    signo y en coma flotante".  [P1]'s "flip all bits if negative" rule
 *    reverses the order of negative two's-complement ints, so it is applied
 *    to float32 only.
 *  - float32: [P1] "符号付型、浮動小数点型に対する radix sort": NaN and both
 *    infinities map to 0xFFFFFFFF (all tie, sort last, stable); otherwise a
 *    set sign bit flips every bit and a clear one sets the MSB.
 *  - A digit that would run past end_bit is cut to the remaining bits.
 *  - 16-bit keys (uint16, int16, IEEE binary16) follow "by the same
 *    procedure" ([P1] "符号付型、浮動小数点型に対する radix sort" says 16- and
 *    64-bit keys sort the same way): the int16 map flips the sign bit, the
 *    binary16 map is [P1]'s float rule at 16 bits (exponent field all ones
 *    -> 0xFFFF; negative -> all bits flipped; positive -> MSB set).
 *  - Descending order is the ascending order of the complemented ordered key
 *    restricted to [begin, end): each pass's counting sort takes its buckets
 *    in reverse (digit ^ mask), still walking the input in order, so ties
 *    keep their input order.  (The pages sort ascending only.)
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_U32 = 0, OR_I32 = 1, OR_F32 = 2, OR_U64 = 3, OR_U16 = 4, OR_I16 = 5, OR_F16 = 6 };

enum { OR_OK = 0, OR_BAD_ARG = 1, OR_NO_MEMORY = 2 };

/* [P2] "Claves con signo y en coma flotante": flipping the sign bit makes
 * two's-complement ints compare as unsigned. */
uint32_t oracle_ordered_i32(uint32_t bits)
{
    return bits ^ 0x80000000u;
}

/* [P1] "符号付型、浮動小数点型に対する radix sort", FloatToOrderedUint: NaN and
 * +-Inf (exponent field all ones) become the maximum; a negative value has
 * all its bits flipped; a positive value gets its MSB set. */
uint32_t oracle_ordered_f32(uint32_t bits)
{
    if ((bits & 0x7F800000u) == 0x7F800000u)
        return 0xFFFFFFFFu;
    if (bits & 0x80000000u)
        return ~bits;
    return bits ^ 0x80000000u;
}

/* The int16 map: the sign-bit flip of [P2] at 16 bits. */
uint32_t oracle_ordered_i16(uint32_t bits)
{
    return (bits ^ 0x8000u) & 0xFFFFu;
}

/* The binary16 map: [P1]'s FloatToOrderedUint rule at 16 bits (5-bit
 * exponent field in bits 10..14). */
uint32_t oracle_ordered_f16(uint32_t bits)
{
    bits &= 0xFFFFu;
    if ((bits & 0x7C00u) == 0x7C00u)
        return 0xFFFFu;
    if (bits & 0x8000u)
        return ~bits & 0xFFFFu;
    return bits ^ 0x8000u;
}

uint64_t oracle_ordered_key(int key_type, uint64_t raw)
{
    switch (key_type) {
    case OR_U32: return raw & 0xFFFFFFFFull;
    case OR_I32: return oracle_ordered_i32((uint32_t)raw);
    case OR_F32: return oracle_ordered_f32((uint32_t)raw);
    case OR_U16: return raw & 0xFFFFull;
    case OR_I16: return oracle_ordered_i16((uint32_t)raw);
    case OR_F16: return oracle_ordered_f16((uint32_t)raw);
    default:     return raw;
    }
}

static int valid_key_type(int key_type) { return key_type >= OR_U32 && key_type <= OR_F16; }

static int key_bits(int key_type)
{
    return key_type == OR_U64 ? 64 : key_type >= OR_U16 ? 16 : 32;
}

static size_t key_size(int key_type) { return (size_t)key_bits(key_type) / 8; }

static uint64_t load_raw(int key_type, const void* keys, size_t i)
{
    switch (key_size(key_type)) {
    case 8: return ((const uint64_t*)keys)[i];
    case 2: return ((const uint16_t*)keys)[i];
    default: return ((const uint32_t*)keys)[i];
    }
}

static void store_raw(int key_type, void* keys, size_t i, uint64_t v)
{
    switch (key_size(key_type)) {
    case 8: ((uint64_t*)keys)[i] = v; break;
    case 2: ((uint16_t*)keys)[i] = (uint16_t)v; break;
    default: ((uint32_t*)keys)[i] = (uint32_t)v; break;
    }
}

/* [P5] "CPU上的扫描", written in its exclusive form: out[i] = sum of in[0..i). */
void oracle_exclusive_scan(const uint64_t* in, uint64_t* out, size_t n)
{
    uint64_t run = 0;
    for (size_t i = 0; i < n; ++i) {
        uint64_t v = in[i];
        out[i] = run;
        run += v;
    }
}

/*
 * One stable counting-sort pass ([P1] "アルゴリズムの詳細" bucket sort; [P5]
 * "CPU上的基数排序"): count how many keys fall in each bucket, turn the counts
 * into bucket starts with an exclusive scan, then walk the input in order and
 * place every key at the next free slot of its bucket.  Walking in input
 * order is what makes the pass stable ([P2] "La idea y el requisito de
 * estabilidad").  `start` is caller scratch of nbins entries.
 */
static void counting_pass(const uint64_t* src_keys, const uint32_t* src_vals,
                          const uint32_t* digit, size_t n, uint32_t nbins,
                          uint64_t* dst_keys, uint32_t* dst_vals,
                          uint64_t* count, uint64_t* start)
{
    for (uint32_t b = 0; b < nbins; ++b) count[b] = 0;
    for (size_t i = 0; i < n; ++i) count[digit[i]] += 1;
    oracle_exclusive_scan(count, start, nbins);
    for (size_t i = 0; i < n; ++i) {
        uint64_t j = start[digit[i]]++;
        dst_keys[j] = src_keys[i];
        if (src_vals) dst_vals[j] = src_vals[i];
    }
}

/*
 * LSD radix sort by passes of counting sort over r-bit digits, lowest digit
 * first ([P1] "アルゴリズムの詳細"; [P2] "Las tres fases de una pasada"; [P3]
 * 13.2).  Pass p sorts by bits [begin + p*r, min(begin + (p+1)*r, end)) of the
 * ordered key, recomputed from the original bits in every pass as [P1]'s CPU
 * code does, so the output keeps the original bit patterns.  With descending
 * set, each pass takes its buckets in reverse order (digit ^ mask).
 * vals_in / vals_out may both be NULL (keys only).
 */
int oracle_lsd_sort_dir(int key_type, const void* keys_in, void* keys_out,
                        const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                        int begin_bit, int end_bit, int radix_bits, int descending)
{
    if (!valid_key_type(key_type)) return OR_BAD_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > key_bits(key_type)) return OR_BAD_ARG;
    if (radix_bits < 1 || radix_bits > 16) return OR_BAD_ARG;
    if ((vals_in == NULL) != (vals_out == NULL)) return OR_BAD_ARG;
    if (n == 0) return OR_OK;

    uint32_t nbins = 1u << radix_bits;
    uint64_t* a = malloc(n * sizeof(uint64_t));
    uint64_t* b = malloc(n * sizeof(uint64_t));
    uint32_t* va = vals_in ? malloc(n * sizeof(uint32_t)) : NULL;
    uint32_t* vb = vals_in ? malloc(n * sizeof(uint32_t)) : NULL;
    uint32_t* digit = malloc(n * sizeof(uint32_t));
    uint64_t* count = malloc(nbins * sizeof(uint64_t));
    uint64_t* start = malloc(nbins * sizeof(uint64_t));
    int rc = OR_OK;
    if (!a || !b || !digit || !count || !start || (vals_in && (!va || !vb))) {
        rc = OR_NO_MEMORY;
        goto done;
    }
    for (size_t i = 0; i < n; ++i) a[i] = load_raw(key_type, keys_in, i);
    if (vals_in) memcpy(va, vals_in, n * sizeof(uint32_t));

    for (int lo = begin_bit; lo < end_bit; lo += radix_bits) {
        int width = end_bit - lo < radix_bits ? end_bit - lo : radix_bits;
        uint64_t mask = (width == 64) ? ~0ull : ((1ull << width) - 1);
        const uint64_t flip = descending ? mask : 0;
        for (size_t i = 0; i < n; ++i)
            digit[i] = (uint32_t)(((oracle_ordered_key(key_type, a[i]) >> lo) & mask) ^ flip);
        counting_pass(a, va, digit, n, nbins, b, vb, count, start);
        uint64_t* t = a; a = b; b = t;
        uint32_t* tv = va; va = vb; vb = tv;
    }
    for (size_t i = 0; i < n; ++i) store_raw(key_type, keys_out, i, a[i]);
    if (vals_in) memcpy(vals_out, va, n * sizeof(uint32_t));
done:
    free(a); free(b); free(va); free(vb); free(digit); free(count); free(start);
    return rc;
}

int oracle_lsd_sort(int key_type, const void* keys_in, void* keys_out,
                    const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                    int begin_bit, int end_bit, int radix_bits)
{
    return oracle_lsd_sort_dir(key_type, keys_in, keys_out, vals_in, vals_out, n, begin_bit, end_bit,
                               radix_bits, 0);
}

/*
 * The decimal LSD example of [P2] "La idea y el requisito de estabilidad":
 * the same counting pass, with the digit of pass p being (x / 10^p) mod 10.
 * trace receives the array after each pass, row-major (passes x n).
 */
int oracle_decimal_lsd_trace(const uint64_t* keys, size_t n, int passes, uint64_t* trace)
{
    if (passes < 0 || passes > 19) return OR_BAD_ARG;
    uint64_t* a = malloc((n ? n : 1) * sizeof(uint64_t));
    uint64_t* b = malloc((n ? n : 1) * sizeof(uint64_t));
    uint32_t* digit = malloc((n ? n : 1) * sizeof(uint32_t));
    uint64_t count[10], start[10];
    if (!a || !b || !digit) { free(a); free(b); free(digit); return OR_NO_MEMORY; }
    memcpy(a, keys, n * sizeof(uint64_t));
    uint64_t place = 1;
    for (int p = 0; p < passes; ++p) {
        for (size_t i = 0; i < n; ++i) digit[i] = (uint32_t)((a[i] / place) % 10u);
        counting_pass(a, NULL, digit, n, 10, b, NULL, count, start);
        memcpy(trace + (size_t)p * n, b, n * sizeof(uint64_t));
        uint64_t* t = a; a = b; b = t;
        place *= 10;
    }
    free(a); free(b); free(digit);
    return OR_OK;
}

/*
 * A second, independent CPU path: [P1]'s one-bit split sort restated from its
 * index formula ("アルゴリズムの詳細").  For bit b, with s_i the number of
 * zero bits before position i and F the number of zero bits in all, a key
 * whose bit is 0 moves to s_i and a key whose bit is 1 moves to F + i - s_i.
 * (The display equation prints n - s_i + F for the second case; the
 * derivation beneath it and the page's code use F + i - s_i, which is the
 * one that is a permutation.)  One pass per bit of [begin, end).
 */
int oracle_one_bit_split_sort(int key_type, const void* keys_in, void* keys_out,
                              const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                              int begin_bit, int end_bit)
{
    if (!valid_key_type(key_type)) return OR_BAD_ARG;
    if (begin_bit < 0 || end_bit < begin_bit || end_bit > key_bits(key_type)) return OR_BAD_ARG;
    if ((vals_in == NULL) != (vals_out == NULL)) return OR_BAD_ARG;
    if (n == 0) return OR_OK;
    uint64_t* a = malloc(n * sizeof(uint64_t));
    uint64_t* b = malloc(n * sizeof(uint64_t));
    uint32_t* va = vals_in ? malloc(n * sizeof(uint32_t)) : NULL;
    uint32_t* vb = vals_in ? malloc(n * sizeof(uint32_t)) : NULL;
    uint64_t* s = malloc(n * sizeof(uint64_t));
    int rc = OR_OK;
    if (!a || !b || !s || (vals_in && (!va || !vb))) { rc = OR_NO_MEMORY; goto done; }
    for (size_t i = 0; i < n; ++i) a[i] = load_raw(key_type, keys_in, i);
    if (vals_in) memcpy(va, vals_in, n * sizeof(uint32_t));

    for (int bit = begin_bit; bit < end_bit; ++bit) {
        uint64_t zeros = 0;
        for (size_t i = 0; i < n; ++i) {
            s[i] = zeros;  /* zeros strictly before i */
            if (((oracle_ordered_key(key_type, a[i]) >> bit) & 1u) == 0) zeros += 1;
        }
        uint64_t F = zeros;
        for (size_t i = 0; i < n; ++i) {
            int one = (int)((oracle_ordered_key(key_type, a[i]) >> bit) & 1u);
            uint64_t dst = one ? F + (uint64_t)i - s[i] : s[i];
            b[dst] = a[i];
            if (va) vb[dst] = va[i];
        }
        uint64_t* t = a; a = b; b = t;
        uint32_t* tv = va; va = vb; vb = tv;
    }
    for (size_t i = 0; i < n; ++i) store_raw(key_type, keys_out, i, a[i]);
    if (vals_in) memcpy(vals_out, va, n * sizeof(uint32_t));
done:
    free(a); free(b); free(va); free(vb); free(s);
    return rc;
}

/* Ordered keys of a whole array, for the transform-invariant tests. */
void oracle_ordered_keys(int key_type, const void* keys, size_t n, uint64_t* out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_ordered_key(key_type, load_raw(key_type, keys, i));
}

size_t oracle_key_size(int key_type) { return key_size(key_type); }
