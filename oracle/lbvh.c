/* lbvh.c -- TEST INFRASTRUCTURE ONLY: the binary radix tree over sorted
 * Morton codes, built top-down from its definition, as the oracle for the
 * GPU's per-node build.  Plain, single-threaded C; shares nothing with the
 * CUDA library.
 *
 * The tree (the hierarchy of a linear BVH; "高性能计算：GPU上的基数排序" names
 * building it as the reason to sort on the GPU, and the node numbering is
 * that of Karras 2012): the keys are the codes made distinct by position,
 * key(i) = code[i] * 2^32 + i.  A node covering leaves [first, last] with
 * first < last splits where the highest bit in which key(first) and
 * key(last) differ turns from 0 to 1; as the keys are sorted, the split is
 * the last position in the range whose key has that bit clear.  Internal
 * node numbering: the root is 0 and covers [0, n-1]; a left child covering
 * [first, split] is internal node `split` (leaf `split` when first == split),
 * a right child covering [split+1, last] is internal node `split+1` (leaf
 * `split+1` when split+1 == last).
 *
 * Here the split is found by walking the range from its first leaf until the
 * bit turns to 1 -- no search, no prefix lengths -- and the nodes are built
 * from the root down with an explicit stack.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#define LEAF 0x80000000u
#define NONE 0xFFFFFFFFu

static uint64_t key_at(const uint32_t* codes, size_t i) { return ((uint64_t)codes[i] << 32) | (uint64_t)i; }

static int highest_set_bit(uint64_t x)
{
    int b = -1;
    while (x) {
        x >>= 1;
        ++b;
    }
    return b;
}

/* Returns 0, or -1 if n is too large or memory runs out.  Array sizes as in
 * rs_lbvh_build: left/right/first/last/node_parent n-1, leaf_parent n. */
int oracle_lbvh_build(const uint32_t* codes, size_t n, uint32_t* left, uint32_t* right, uint32_t* first,
                      uint32_t* last, uint32_t* leaf_parent, uint32_t* node_parent)
{
    if (n > ((size_t)1 << 31)) return -1;
    if (n == 0) return 0;
    if (n == 1) {
        leaf_parent[0] = NONE;
        return 0;
    }
    /* stack of internal nodes still to split: (node, first, last) */
    size_t cap = 64, top = 0;
    uint32_t* st = (uint32_t*)malloc(3 * cap * sizeof(uint32_t));
    if (!st) return -1;
    node_parent[0] = NONE;
    st[0] = 0;
    st[1] = 0;
    st[2] = (uint32_t)(n - 1);
    top = 1;
    while (top > 0) {
        --top;
        const uint32_t node = st[3 * top], f = st[3 * top + 1], l = st[3 * top + 2];
        const int bit = highest_set_bit(key_at(codes, f) ^ key_at(codes, l));
        const uint64_t mask = (uint64_t)1 << bit;
        uint32_t split = f;
        while (split + 1 < l && (key_at(codes, split + 1) & mask) == 0) ++split;
        first[node] = f;
        last[node] = l;
        uint32_t children[2][3] = {{split, f, split}, {split + 1, split + 1, l}};
        for (int c = 0; c < 2; ++c) {
            const uint32_t idx = children[c][0], cf = children[c][1], cl = children[c][2];
            const int is_leaf = cf == cl;
            if (c == 0) left[node] = is_leaf ? (idx | LEAF) : idx;
            else right[node] = is_leaf ? (idx | LEAF) : idx;
            if (is_leaf) {
                leaf_parent[idx] = node;
            } else {
                node_parent[idx] = node;
                if (top == cap) {
                    cap *= 2;
                    uint32_t* grown = (uint32_t*)realloc(st, 3 * cap * sizeof(uint32_t));
                    if (!grown) {
                        free(st);
                        return -1;
                    }
                    st = grown;
                }
                st[3 * top] = idx;
                st[3 * top + 1] = cf;
                st[3 * top + 2] = cl;
                ++top;
            }
        }
    }
    free(st);
    return 0;
}
