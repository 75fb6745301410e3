"""The KV block allocator with one block bitmap per (layer, KV head)
("国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析", §2.4 KDA):
the plain model in oracle/kda.py pinned to its stated policy, then the
library's allocator (C ABI) against the model on random operation sequences."""
import ctypes as C

import numpy as np
import pytest

from oracle.kda import BitmapKDA

DSA_OK, INVALID, UNSUPPORTED, OOM = 0, 1, 2, 3


# ---------------------------------------------------------------- model pins
def test_model_fresh_pool_gives_the_lowest_ids_in_order():
    a = BitmapKDA(1, 1, 10)
    assert a.alloc(0, 0, 3) == [0, 1, 2]
    assert a.alloc(0, 0, 4) == [3, 4, 5, 6]
    assert a.num_free(0, 0) == 3
    assert a.alloc(0, 0, 4) is None and a.num_free(0, 0) == 3  # too few: nothing taken
    assert a.alloc(0, 0, 3) == [7, 8, 9] and a.num_free(0, 0) == 0


def test_model_freed_blocks_are_reused_lowest_first():
    a = BitmapKDA(1, 1, 8)
    a.alloc(0, 0, 8)
    assert a.free(0, 0, [5, 2])
    assert a.alloc(0, 0, 1) == [2]
    assert a.alloc(0, 0, 1) == [5]


def test_model_heads_and_layers_are_independent():
    """Every (layer, head) has its own bitmap: the same ids are handed to
    different heads, and a release in one leaves the others unchanged."""
    a = BitmapKDA(2, 3, 5)
    got = {(l, h): a.alloc(l, h, 2) for l in range(2) for h in range(3)}
    assert all(v == [0, 1] for v in got.values())
    assert a.free(1, 2, [0])
    assert a.num_free(1, 2) == 4 and all(a.num_free(l, h) == 3 for l in range(2) for h in range(3) if (l, h) != (1, 2))
    assert a.alloc(0, 0, 1) == [2] and a.alloc(1, 2, 1) == [0]


def test_model_bad_release_changes_nothing():
    a = BitmapKDA(1, 2, 6)
    a.alloc(0, 0, 3)
    before = a.bitmap(0, 0)
    assert not a.free(0, 0, [1, 1])   # twice
    assert not a.free(0, 0, [4])      # not held
    assert not a.free(0, 1, [0])      # held by the other head
    assert a.bitmap(0, 0) == before


def test_model_bitmap_words():
    a = BitmapKDA(1, 1, 130)
    a.alloc(0, 0, 66)
    w = a.bitmap(0, 0)
    assert w == [(1 << 64) - 1, 0b11, 0]


# --------------------------------------------------- the library allocator
@pytest.fixture(scope="module")
def bm(lib):
    return lib


def _create(lib, layers, heads, blocks):
    h = C.c_void_p()
    assert lib.dsa_kv_bitmap_create(layers, heads, blocks, C.byref(h)) == DSA_OK
    return h


def test_library_matches_the_model_on_random_operations(bm):
    lib = bm
    rng = np.random.default_rng(11)
    for layers, heads, blocks in ((1, 1, 1), (2, 3, 70), (3, 8, 257)):
        a = _create(lib, layers, heads, blocks)
        m = BitmapKDA(layers, heads, blocks)
        held = {(l, g): [] for l in range(layers) for g in range(heads)}
        try:
            for _ in range(400):
                l, g = int(rng.integers(layers)), int(rng.integers(heads))
                if rng.random() < 0.55:
                    n = int(rng.integers(0, max(2, blocks // 3)))
                    out = (C.c_int32 * max(n, 1))()
                    st = lib.dsa_kv_bitmap_alloc(a, l, g, n, out)
                    want = m.alloc(l, g, n)
                    if want is None:
                        assert st == OOM
                    else:
                        assert st == DSA_OK and list(out)[:n] == want
                        held[(l, g)] += want
                else:
                    ids = list(held[(l, g)])
                    rng.shuffle(ids)
                    ids = ids[:int(rng.integers(0, len(ids) + 1))]
                    if rng.random() < 0.15:  # a bad id somewhere in the call
                        ids = ids + [int(rng.integers(blocks))] if rng.random() < 0.5 else ids + ids[:1]
                    arr = (C.c_int32 * max(len(ids), 1))(*ids)
                    st = lib.dsa_kv_bitmap_free(a, l, g, arr, len(ids))
                    ok = m.free(l, g, ids)
                    assert (st == DSA_OK) == ok
                    if ok:
                        for i in ids:
                            held[(l, g)].remove(i)
                assert lib.dsa_kv_bitmap_num_free(a, l, g) == m.num_free(l, g)
                words = m.bitmap(l, g)
                got = (C.c_uint64 * len(words))()
                assert lib.dsa_kv_bitmap_words(a, l, g, got, len(words)) == DSA_OK
                assert list(got) == words
        finally:
            lib.dsa_kv_bitmap_destroy(a)


def test_library_argument_checks(bm):
    lib = bm
    h = C.c_void_p()
    assert lib.dsa_kv_bitmap_create(0, 1, 8, C.byref(h)) == INVALID
    assert lib.dsa_kv_bitmap_create(1, 0, 8, C.byref(h)) == INVALID
    assert lib.dsa_kv_bitmap_create(1, 1, 0, C.byref(h)) == INVALID
    assert lib.dsa_kv_bitmap_create(1, 1, 8, None) == INVALID
    a = _create(lib, 2, 2, 8)
    try:
        out = (C.c_int32 * 8)()
        assert lib.dsa_kv_bitmap_alloc(a, 2, 0, 1, out) == INVALID   # layer out of range
        assert lib.dsa_kv_bitmap_alloc(a, 0, -1, 1, out) == INVALID  # head out of range
        assert lib.dsa_kv_bitmap_alloc(a, 0, 0, -1, out) == INVALID
        assert lib.dsa_kv_bitmap_alloc(a, 0, 0, 1, None) == INVALID
        assert lib.dsa_kv_bitmap_alloc(a, 0, 0, 9, out) == OOM
        assert lib.dsa_kv_bitmap_num_free(a, 0, 0) == 8
        assert lib.dsa_kv_bitmap_num_free(a, 5, 0) == -1
        w = (C.c_uint64 * 1)()
        assert lib.dsa_kv_bitmap_words(a, 0, 0, w, 0) == INVALID     # too few words
    finally:
        lib.dsa_kv_bitmap_destroy(a)
