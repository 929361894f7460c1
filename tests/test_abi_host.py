"""CPU tests of the library: it loads, exports every symbol the header declares,
and its host-side parts (slot mapping, block manager) behave as specified."""
import os
import re

import numpy as np
import pytest

import oracle
import pagedattention_paged_kv_gb300 as pkv
from pagedattention_paged_kv_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build_library()
    return pkv.lib()


def header_symbols():
    with open(os.path.join(ROOT, "include", "pagedkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = header_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pagedkv.h but not exported"


def test_status_strings(lib):
    import ctypes
    lib.pkv_status_string.restype = ctypes.c_char_p
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(-5) == b"out of blocks"


def test_slot_mapping_matches_oracle(lib):
    rng = np.random.Generator(np.random.PCG64(1))
    S, MB, bs = 9, 12, 16
    tables = rng.permutation(S * MB).astype(np.int32).reshape(S, MB)
    seq = rng.integers(-1, S, size=500).astype(np.int32)
    pos = rng.integers(0, MB * bs, size=500).astype(np.int32)
    got = pkv.slot_mapping(tables, seq, pos, bs)
    ref = oracle.load().slot_mapping(tables, seq, pos, bs)
    assert np.array_equal(got, ref)


def test_slot_mapping_rejects_position_past_table(lib):
    with pytest.raises(pkv.PagedKVError):
        pkv.slot_mapping(np.zeros((1, 2), np.int32), np.array([0], np.int32), np.array([32], np.int32))


def test_block_manager_fifo_and_oom(lib):
    bm = pkv.BlockManager(10)
    a = bm.allocate(4)
    assert a == [0, 1, 2, 3]
    b = bm.allocate(6)
    assert b == [4, 5, 6, 7, 8, 9] and bm.num_free() == 0
    with pytest.raises(pkv.OutOfBlocks):
        bm.allocate(1)
    bm.free([2, 0])
    assert bm.num_free() == 2
    with pytest.raises(pkv.OutOfBlocks):
        bm.allocate(3)            # fails without taking anything
    assert bm.num_free() == 2
    assert bm.allocate(2) == [2, 0]   # freed ids come back in the order they were freed


def test_block_manager_rejects_bad_free(lib):
    bm = pkv.BlockManager(4)
    ids = bm.allocate(2)
    with pytest.raises(pkv.PagedKVError):
        bm.free([ids[0], ids[0]])  # the same id twice
    with pytest.raises(pkv.PagedKVError):
        bm.free([3])               # not allocated
    with pytest.raises(pkv.PagedKVError):
        bm.free([7])               # outside the pool
    assert bm.num_free() == 2
    bm.free(ids)
    assert bm.num_free() == 4
