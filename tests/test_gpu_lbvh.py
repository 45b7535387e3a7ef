"""rs_lbvh_build on the GPU against the CPU oracle.

Morton codes (and tie-heavy codes) are sorted on the GPU with
rs_sort_pairs_u32 -- the pipeline "高性能计算：GPU上的基数排序" sorts for -- and
the radix tree built from them is compared with the oracle's top-down build,
array by array and bit for bit, at sizes that span many blocks of the kernel.
At the full 2^28-key Morton workload the oracle is too slow, so there the
tree is checked by properties that hold at any size (every leaf and every
non-root node has exactly one parent, computed on the GPU) and sampled nodes
against the definition, each from a few keys.
"""
import numpy as np
import pytest

import lsd_radix_sort_key_gb300 as rs
import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = "cuda:0"
FIELDS = ("left", "right", "first", "last", "leaf_parent", "node_parent")


def sorted_on_gpu(codes):
    kin = torch.from_numpy(codes.view(np.int32)).to(DEV)
    vin = torch.arange(codes.size, dtype=torch.int32, device=DEV)
    kout, vout = rs.sort(kin, vin, key_type="u32")
    return kout, vout


@pytest.mark.parametrize("n,kind", [(2, "uniform"), (3, "uniform"), (5, "ties"), (100, "morton"),
                                    (4097, "uniform"), (100_003, "morton"), (100_000, "ties"),
                                    (65_536, "equal"), (1 << 20, "morton")])
def test_tree_matches_oracle(n, kind):
    rs.build()
    if kind == "morton":
        codes = synth.u32_morton30(n, 11)
    elif kind == "ties":
        codes = synth.u32_uniform(n, 12) & np.uint32(0x00F000F1)
    elif kind == "equal":
        codes = np.full(n, 0x1234, np.uint32)
    else:
        codes = synth.u32_uniform(n, 13)
    kout, vout = sorted_on_gpu(codes)
    tree = rs.lbvh_build(kout)
    torch.cuda.synchronize()
    sorted_codes = kout.cpu().numpy().view(np.uint32)
    want_k, want_v = oracle.sort("u32", codes, np.arange(n, dtype=np.uint32))
    assert np.array_equal(sorted_codes, want_k)
    assert np.array_equal(vout.cpu().numpy().view(np.uint32), want_v)
    want = oracle.lbvh_build(want_k)
    for f in FIELDS:
        assert np.array_equal(tree[f].cpu().numpy().view(np.uint32), want[f]), f


def test_one_and_zero_codes():
    rs.build()
    one = torch.tensor([5], dtype=torch.int32, device=DEV)
    lp = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert rs.rs_lbvh_build(one, 1, None, None, None, None, lp, None) == 0
    torch.cuda.synchronize()
    assert int(lp.cpu().numpy().view(np.uint32)[0]) == oracle.LBVH_NONE
    assert rs.rs_lbvh_build(None, 0, None, None, None, None, None, None) == 0
    assert rs.rs_lbvh_build(one, 2, None, None, None, None, lp, None) == 1  # NULL outputs


def test_full_size_morton_workload_by_properties():
    rs.build()
    w = synth.WORKLOADS["morton30_index_2p28"]
    n = w.n
    codes = w.keys(n)
    kin = torch.from_numpy(codes.view(np.int32)).to(DEV)
    del codes
    vin = torch.arange(n, dtype=torch.int32, device=DEV)
    kout, _ = rs.sort(kin, vin, key_type="u32", begin_bit=w.begin_bit, end_bit=w.end_bit)
    del kin, vin
    tree = rs.lbvh_build(kout)
    torch.cuda.synchronize()
    leaf_mask = torch.tensor(rs.LBVH_LEAF - (1 << 32), dtype=torch.int32, device=DEV)  # bit 31 as int32
    # every leaf exactly once as a child, every internal node but the root exactly once
    kids = torch.cat([tree["left"], tree["right"]])
    is_leaf = (kids & leaf_mask) != 0
    leaf_count = torch.bincount((kids[is_leaf] & 0x7FFFFFFF).long(), minlength=n)
    node_count = torch.bincount(kids[~is_leaf].long(), minlength=n - 1)
    assert int(leaf_count.min()) == 1 and int(leaf_count.max()) == 1
    assert int(node_count[0]) == 0 and int(node_count[1:].min()) == 1 and int(node_count[1:].max()) == 1
    del kids, is_leaf, leaf_count, node_count
    # sampled nodes against the definition (a few keys each)
    rng = np.random.default_rng(2028)
    idx = np.unique(np.concatenate([[0, 1, n - 2], rng.integers(0, n - 1, 4000)]))
    ti = torch.from_numpy(idx).to(DEV)
    f = tree["first"][ti].cpu().numpy().view(np.uint32).astype(np.int64)
    l = tree["last"][ti].cpu().numpy().view(np.uint32).astype(np.int64)
    left = tree["left"][ti].cpu().numpy().view(np.uint32).astype(np.int64)
    right = tree["right"][ti].cpu().numpy().view(np.uint32).astype(np.int64)

    def key(pos):
        pos = np.asarray(pos, dtype=np.int64)
        c = kout[torch.from_numpy(np.clip(pos, 0, n - 1)).to(DEV)].cpu().numpy().view(np.uint32)
        return (c.astype(np.uint64) << np.uint64(32)) | pos.astype(np.uint64)

    kf, kl = key(f), key(l)
    kprev, knext = key(f - 1), key(l + 1)
    split = left & 0x7FFFFFFF
    ks, ks1 = key(split), key(split + 1)
    assert np.all((f == idx) | (l == idx)) and np.all(f < l)
    assert f[0] == 0 and l[0] == n - 1
    assert np.all((right & 0x7FFFFFFF) == split + 1)
    for j in range(idx.size):
        b = int(kf[j] ^ kl[j]).bit_length() - 1
        hi = ((1 << 64) - 1) ^ ((1 << (b + 1)) - 1)
        assert (int(ks[j]) >> b) & 1 == 0 and (int(ks1[j]) >> b) & 1 == 1
        assert f[j] <= split[j] < l[j]
        if f[j] > 0:
            assert int(kprev[j]) & hi != int(kf[j]) & hi
        if l[j] < n - 1:
            assert int(knext[j]) & hi != int(kl[j]) & hi
