"""The block-aligned ZeRO split (bwd_zero_shard, host only): over all ranks
the pieces cover every element of every tensor exactly once, cut only on
2048-element block boundaries, and give every rank a contiguous run of the
same number of blocks (the last ranks fewer or none)."""

import ctypes

import numpy as np
import pytest

B = 2048


@pytest.fixture(scope="module")
def lib():
    from block_wise_dynamic_gb300 import build as b

    b.build()
    from block_wise_dynamic_gb300 import _abi

    return _abi.load()


def shard(lib, sizes, world, rank):
    T = len(sizes)
    n = (ctypes.c_int64 * max(T, 1))(*sizes)
    k = ctypes.c_int64(-1)
    cnt = ctypes.c_int32(-1)
    ti = (ctypes.c_int32 * max(T, 1))()
    off = (ctypes.c_int64 * max(T, 1))()
    c = (ctypes.c_int64 * max(T, 1))()
    st = lib.bwd_zero_shard(T, n, world, rank, ctypes.byref(k), ctypes.byref(cnt), ti, off, c)
    return st, k.value, [(ti[j], off[j], c[j]) for j in range(cnt.value)]


def size_lists():
    rng = np.random.default_rng(7)
    yield [2048 * 5]
    yield [1, 2047, 2048, 2049, 0, 4096 * 3 + 17]
    yield [0, 0, 0]
    yield [3000] * 11
    yield [int(x) for x in np.floor(np.exp(rng.uniform(np.log(1), np.log(50_000), 300)))]
    yield [6_738_415_616 // 291] * 7 + [5]


@pytest.mark.parametrize("world", [1, 2, 3, 5, 8, 64])
def test_pieces_cover_each_element_once_on_block_boundaries(lib, world):
    for sizes in size_lists():
        nb = [-(-n // B) for n in sizes]
        NB = sum(nb)
        covered = [[] for _ in sizes]
        ks, next_block = set(), 0
        for r in range(world):
            st, k, pieces = shard(lib, sizes, world, r)
            assert st == 0
            ks.add(k)
            assert k * world >= NB and (k == 0 if NB == 0 else (k - 1) * world < NB)  # equal, minimal shares
            blocks = 0
            prev = (-1, -1)
            for ti, off, cnt in pieces:
                assert (ti, off) > prev
                prev = (ti, off)
                assert off % B == 0 and 0 < cnt and off + cnt <= sizes[ti]
                assert cnt % B == 0 or off + cnt == sizes[ti]  # a piece ends on a block edge or the tensor's end
                covered[ti].append((off, off + cnt))
                blocks += -(-cnt // B)
            assert blocks <= k
            if blocks:  # rank r's blocks are the run starting at r * k
                assert next_block == r * k
                next_block += blocks
        assert next_block == NB and len(ks) == 1
        for n, iv in zip(sizes, covered):
            iv.sort()
            pos = 0
            for a, b in iv:
                assert a == pos
                pos = b
            assert pos == n


def test_world_larger_than_blocks_leaves_ranks_empty(lib):
    sizes = [100, 2048 + 1]
    for r in range(8):
        st, k, pieces = shard(lib, sizes, 8, r)
        assert st == 0 and k == 1
        assert len(pieces) == (1 if r < 3 else 0)


def test_bad_arguments(lib):
    for world, rank in [(0, 0), (2, 2), (2, -1)]:
        assert shard(lib, [10], world, rank)[0] == 1
    assert shard(lib, [10, -1], 2, 0)[0] == 1
    n = (ctypes.c_int64 * 1)(10)
    assert lib.bwd_zero_shard(1, n, 1, 0, None, None, None, None, None) == 1  # num_pieces is required
    cnt = ctypes.c_int32(-1)
    assert lib.bwd_zero_shard(1, n, 1, 0, None, ctypes.byref(cnt), None, None, None) == 0 and cnt.value == 1
    big = (ctypes.c_int64 * 2)(2 ** 62, 2 ** 62)
    assert lib.bwd_zero_shard(2, big, 2, 0, None, ctypes.byref(cnt), None, None, None) == 1  # overflow


def test_layout_positions_fall_inside_the_rank_slice():
    from block_wise_dynamic_gb300.zero import ShardLayout

    sizes = [5000, 2048, 17, 0, 40_000]
    for world in (1, 2, 3, 4):
        L = ShardLayout(sizes, world)
        assert L.flat_numel == world * L.shard_numel >= sum(-(-n // B) * B for n in sizes)
        for r in range(world):
            for pc in L.pieces[r]:
                s = L.flat_start(r, pc)
                assert s % B == 0 and 0 <= s and s + pc[2] <= L.shard_numel
