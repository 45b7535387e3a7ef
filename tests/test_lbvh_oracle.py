"""The LBVH oracle (oracle.lbvh_build) pinned to the definition of the tree.

The tree is the binary radix tree over the sorted codes made distinct by
position, key(i) = code[i] * 2^32 + i, with the internal-node numbering of
Karras 2012 (building it is what "高性能计算：GPU上的基数排序" sorts for).  The
oracle builds it top-down; these tests check what the definition fixes,
independently of how it is built: a hand-derived tree, and on random and
tie-heavy inputs every structural rule (each leaf and non-root node has
exactly one parent; ranges nest and split in two contiguous halves; each
split sits where the highest differing bit of the range's end keys turns
from 0 to 1; one end of each node's range is its own index).
"""
import numpy as np
import pytest

import oracle
import synth

LEAF = oracle.LBVH_LEAF
NONE = oracle.LBVH_NONE


def keys64(codes):
    return (codes.astype(np.uint64) << np.uint64(32)) | np.arange(codes.size, dtype=np.uint64)


def check_tree(codes, t):
    """Every rule of the definition, by brute force over the ranges."""
    n = codes.size
    if n <= 1:
        if n == 1:
            assert t["leaf_parent"][0] == NONE
        return
    k = keys64(codes)
    left, right, first, last = (t[x].astype(np.int64) for x in ("left", "right", "first", "last"))
    leaf_refs = np.zeros(n, np.int64)
    node_refs = np.zeros(n - 1, np.int64)
    assert first[0] == 0 and last[0] == n - 1 and t["node_parent"][0] == NONE
    for i in range(n - 1):
        f, l = first[i], last[i]
        assert f < l and (f == i or l == i)
        b = int(k[f] ^ k[l]).bit_length() - 1
        mask = np.uint64(1 << b)
        hi = ~np.uint64((1 << (b + 1)) - 1) if b < 63 else np.uint64(0)
        seg = k[f:l + 1]
        # all keys of the range share every bit above b ...
        assert np.all((seg & hi) == (k[f] & hi))
        # ... and the range is maximal: the neighbours outside it do not
        if f > 0:
            assert (k[f - 1] & hi) != (k[f] & hi)
        if l < n - 1:
            assert (k[l + 1] & hi) != (k[l] & hi)
        split = f + int(np.count_nonzero((seg & mask) == 0)) - 1
        assert np.all((k[f:split + 1] & mask) == 0) and np.all((k[split + 1:l + 1] & mask) != 0)
        for child, cf, cl, idx in ((left[i], f, split, split), (right[i], split + 1, l, split + 1)):
            if cf == cl:
                assert child == (idx | LEAF)
                leaf_refs[idx] += 1
                assert t["leaf_parent"][idx] == i
            else:
                assert child == idx and first[idx] == cf and last[idx] == cl
                node_refs[idx] += 1
                assert t["node_parent"][idx] == i
    assert np.all(leaf_refs == 1)
    assert node_refs[0] == 0 and np.all(node_refs[1:] == 1)


def test_hand_derived_example():
    # Eight 5-bit codes; the tree below was derived by hand from the
    # definition (root splits on bit 4 after position 3, node 3 on bit 2
    # after position 1, node 4 on bit 3 after position 4, node 5 on bit 2
    # after position 6, nodes 1, 2 and 6 on their last differing bit).
    codes = np.array([0b00001, 0b00010, 0b00100, 0b00101, 0b10011, 0b11000, 0b11001, 0b11110], np.uint32)
    t = oracle.lbvh_build(codes)
    L = lambda i: i | LEAF  # noqa: E731
    assert t["left"].tolist() == [3, L(0), L(2), 1, L(4), 6, L(5)]
    assert t["right"].tolist() == [4, L(1), L(3), 2, 5, L(7), L(6)]
    assert t["first"].tolist() == [0, 0, 2, 0, 4, 5, 5]
    assert t["last"].tolist() == [7, 1, 3, 3, 7, 7, 6]
    assert t["node_parent"].tolist() == [NONE, 3, 3, 0, 0, 4, 5]
    assert t["leaf_parent"].tolist() == [1, 1, 2, 2, 4, 6, 6, 5]
    check_tree(codes, t)


def test_small_sizes():
    assert oracle.lbvh_build(np.zeros(0, np.uint32))["leaf_parent"].size == 0
    t = oracle.lbvh_build(np.array([7], np.uint32))
    assert t["leaf_parent"].tolist() == [NONE]
    t = oracle.lbvh_build(np.array([5, 9], np.uint32))
    assert t["left"].tolist() == [0 | LEAF] and t["right"].tolist() == [1 | LEAF]
    assert t["leaf_parent"].tolist() == [0, 0] and t["node_parent"].tolist() == [NONE]


@pytest.mark.parametrize("n,seed,mask", [(3, 1, 0xFFFFFFFF), (17, 2, 0xFFFFFFFF), (1000, 3, 0xFFFFFFFF),
                                         (1000, 4, 0x3), (777, 5, 0x0), (3000, 6, 0x0F0F0F0F)])
def test_definition_holds_on_random_and_tied_codes(n, seed, mask):
    codes = np.sort(synth.u32_uniform(n, seed) & np.uint32(mask))
    check_tree(codes, oracle.lbvh_build(codes))


def test_morton_codes():
    codes = np.sort(synth.u32_morton30(2000, 7))
    check_tree(codes, oracle.lbvh_build(codes))


def test_a_planted_split_error_is_caught():
    codes = np.sort(synth.u32_uniform(200, 8))
    t = oracle.lbvh_build(codes)
    bad = {k: v.copy() for k, v in t.items()}
    i = int(np.flatnonzero((bad["right"] & LEAF) == 0)[0])  # a node with an internal right child
    bad["right"][i] += 1
    with pytest.raises(AssertionError):
        check_tree(codes, bad)
