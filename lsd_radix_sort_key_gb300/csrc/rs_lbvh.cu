// rs_lbvh.cu -- rs_lbvh_build: the binary radix tree (the hierarchy of a
// linear BVH) over Morton codes that the sort has put in order.
//
// Building an LBVH on the GPU is the pipeline that "高性能计算：GPU上的基数排序"
// (its opening sections) names as the reason to sort on the GPU at all: the
// codes are sorted where they are made, and the tree is built from them on
// the device.  The page stops at the sort; the tree step here follows the
// published per-node construction of Karras (2012, "Maximizing parallelism in
// the construction of BVHs, octrees, and k-d trees"), restated:
//
// Keys are the sorted codes made distinct by their position: key(i) =
// (code[i] << 32) | i, so delta(i, j), the length of the common prefix of
// key(i) and key(j), is clz(code[i] ^ code[j]) when the codes differ and
// 32 + clz(i ^ j) when they are equal (-1 outside [0, n)).  The n - 1
// internal nodes are numbered so that node i covers a key range with one end
// at i: root 0 covers [0, n - 1]; a node covering [first, last] splits at
// gamma, the last position whose key has a 0 in the highest bit where
// key(first) and key(last) differ; its left child covers [first, gamma] (leaf
// gamma if that is one key, else internal node gamma), its right child
// [gamma + 1, last] (leaf gamma + 1, else internal node gamma + 1).  Each
// thread finds its node's direction, the far end of its range (exponential
// then binary search on delta) and the split (binary search), independently
// of every other node, so the build is one kernel of n - 1 threads.
#include <cuda_runtime.h>
#include <stdint.h>

#include "rs.h"

namespace {

constexpr uint32_t kLeafFlag = 0x80000000u;
constexpr uint32_t kNone = 0xFFFFFFFFu;

// Positions are 32-bit: with n <= 2^31, a probe i + l*d (l <= 2^31, the
// search never doubles past the end of [0, n)) wraps below 0 to a value
// >= 2^31 >= n, so one unsigned compare rejects both ends.
__device__ __forceinline__ uint32_t toward(uint32_t i, uint32_t l, int d) { return d > 0 ? i + l : i - l; }

// delta(i, j): the common prefix length of key(i) and key(j), given ci =
// codes[i]; -1 if j is outside [0, n).
__device__ __forceinline__ int delta(const uint32_t* __restrict__ codes, uint32_t n, uint32_t i, uint32_t ci,
                                     uint32_t j)
{
    if (j >= n) return -1;
    const uint32_t x = ci ^ __ldg(codes + j);
    return x ? __clz(x) : 32 + __clz(i ^ j);
}

// delta(i, j) > m, for m in [-1, 63], without counting the prefix: the keys
// share more than m leading bits exactly when their 64-bit XOR, (code xor)
// << 32 | (position xor), is below 2^(63 - m), i.e. has no bit set under the
// masks of Above(m) (high word: code xor; low word: position xor).
struct Above {
    uint32_t hmask, lmask;
    __device__ __forceinline__ explicit Above(int m)
    {
        const int s = 63 - m;  // 0..64
        hmask = s >= 64 ? 0u : s >= 32 ? ~0u << (s - 32) : ~0u;
        lmask = s >= 32 ? 0u : ~0u << s;
    }
};

__device__ __forceinline__ bool shares_more(const uint32_t* __restrict__ codes, uint32_t n, uint32_t i,
                                            uint32_t ci, uint32_t j, Above a)
{
    if (j >= n) return false;
    return (((ci ^ __ldg(codes + j)) & a.hmask) | ((i ^ j) & a.lmask)) == 0u;
}

__global__ void __launch_bounds__(256) k_lbvh_build(const uint32_t* __restrict__ codes, uint32_t n,
                                                    uint32_t* __restrict__ left, uint32_t* __restrict__ right,
                                                    uint32_t* __restrict__ first, uint32_t* __restrict__ last,
                                                    uint32_t* __restrict__ leaf_parent,
                                                    uint32_t* __restrict__ node_parent)
{
    const uint32_t nodes = n - 1;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nodes; i += gridDim.x * blockDim.x) {
        const uint32_t ci = __ldg(codes + i);
        // Direction of the range: towards the neighbour sharing the longer prefix.
        const int d = (delta(codes, n, i, ci, i + 1) - delta(codes, n, i, ci, i - 1)) >= 0 ? 1 : -1;
        // The far end: every key in the range shares more than delta(i, i - d) bits with key(i).
        const Above far(delta(codes, n, i, ci, toward(i, 1, -d)));
        uint32_t lmax = 2;
        while (shares_more(codes, n, i, ci, toward(i, lmax, d), far)) lmax <<= 1;
        uint32_t l = 0;
        for (uint32_t t = lmax >> 1; t >= 1; t >>= 1)
            if (shares_more(codes, n, i, ci, toward(i, l + t, d), far)) l += t;
        const uint32_t j = toward(i, l, d);
        // The split: the last key (from i towards j) sharing more than the
        // node's own prefix with key(i).
        const Above split(delta(codes, n, i, ci, j));
        uint32_t s = 0, t = l;
        do {
            t = (t + 1) >> 1;
            if (shares_more(codes, n, i, ci, toward(i, s + t, d), split)) s += t;
        } while (t > 1);
        const uint32_t g = toward(i, s, d) - (d < 0 ? 1u : 0u);
        const uint32_t lo = i < j ? i : j, hi = i < j ? j : i;
        const bool left_leaf = lo == g, right_leaf = hi == g + 1;
        left[i] = left_leaf ? (g | kLeafFlag) : g;
        right[i] = right_leaf ? ((g + 1) | kLeafFlag) : g + 1;
        first[i] = lo;
        last[i] = hi;
        if (left_leaf) leaf_parent[g] = i;
        else node_parent[g] = i;
        if (right_leaf) leaf_parent[g + 1] = i;
        else node_parent[g + 1] = i;
        if (i == 0) node_parent[0] = kNone;
    }
}

}  // namespace

extern "C" rs_status rs_lbvh_build(const uint32_t* sorted_codes, size_t n, uint32_t* left, uint32_t* right,
                                   uint32_t* first, uint32_t* last, uint32_t* leaf_parent,
                                   uint32_t* node_parent, void* stream)
{
    if (n > (size_t)RS_LBVH_MAX_N) return RS_ERR_INVALID_ARG;
    if (n == 0) return RS_OK;
    if (!sorted_codes || !leaf_parent) return RS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n == 1) {  // one leaf, no internal node: the leaf has no parent
        return cudaMemsetAsync(leaf_parent, 0xFF, sizeof(uint32_t), s) == cudaSuccess ? RS_OK : RS_ERR_CUDA;
    }
    if (!left || !right || !first || !last || !node_parent) return RS_ERR_INVALID_ARG;
    const uint32_t nodes = (uint32_t)(n - 1);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return RS_ERR_CUDA;
    const uint64_t want = ((uint64_t)nodes + 255) / 256;
    const unsigned grid = (unsigned)(want < (uint64_t)sms * 8 ? want : (uint64_t)sms * 8);
    k_lbvh_build<<<grid, 256, 0, s>>>(sorted_codes, (uint32_t)n, left, right, first, last, leaf_parent,
                                      node_parent);
    return cudaGetLastError() == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}
