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


# ---- argument checks the C ABI makes on the host, before any device work ----------------

def _c():
    import ctypes
    return ctypes


def test_decode_rejects_bad_shapes_before_touching_the_device(lib):
    c = _c()
    vp = c.c_void_p
    f = lib.pkv_paged_attention_decode
    args = lambda Hq, Hkv, d, bs, dtype: [vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), 4, 2, Hq, Hkv, d, bs, 64,
                                          c.c_float(0.1), dtype, vp(0), c.c_size_t(0), vp(0)]
    assert f(*args(8, 3, 128, 16, 0)) == -1          # num_heads not a multiple of num_kv_heads
    assert f(*args(8, 2, 96, 16, 0)) == -2           # head_dim 96
    assert f(*args(8, 2, 128, 12, 0)) == -2          # block size 12
    assert f(*args(8, 2, 128, 16, 7)) == -2          # dtype other than bf16
    zero = [vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), 0, 2, 8, 2, 128, 16, 64, c.c_float(0.1), 0, vp(0),
            c.c_size_t(0), vp(0)]
    assert f(*zero) == 0                             # no sequences: nothing to do


def test_fp8_calls_reject_bad_scales_and_head_dim_on_the_host(lib):
    c = _c()
    vp = c.c_void_p
    def varlen_fp8(d, ks, vs):
        return lib.pkv_paged_attention_varlen_fp8(vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), 2, 3, 2, 1, 8, 2,
                                                  d, 16, 64, c.c_float(0.1), 1, c.c_float(ks), c.c_float(vs),
                                                  vp(0), c.c_size_t(0), vp(0))
    assert varlen_fp8(128, 0.0, 1.0) == -1
    assert varlen_fp8(128, 1.0, float("nan")) == -1
    assert varlen_fp8(128, float("inf"), 1.0) == -1
    assert varlen_fp8(64, 1.0, 1.0) == -2
    def decode_fp8(d, ks, vs):
        return lib.pkv_paged_attention_decode_fp8(vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), 2, 1, 8, 2, d, 16, 64,
                                                  c.c_float(0.1), c.c_float(ks), c.c_float(vs), vp(0),
                                                  c.c_size_t(0), vp(0))
    assert decode_fp8(128, -1.0, 1.0) == -1
    assert decode_fp8(64, 1.0, 1.0) == -2
    f = lib.pkv_reshape_and_cache_fp8
    assert f(vp(0), vp(0), vp(0), vp(0), vp(0), 0, 4, 16, 2, 128, c.c_float(0.0), c.c_float(1.0), vp(0)) == -1
    assert f(vp(0), vp(0), vp(0), vp(0), vp(0), 0, 4, 16, 2, 128, c.c_float(1.0), c.c_float(1.0), vp(0)) == 0
    assert f(vp(0), vp(0), vp(0), vp(0), vp(0), 3, 4, 16, 2, 128, c.c_float(1.0), c.c_float(1.0), vp(0)) == -1


def test_step_copies_check_arguments_on_the_host(lib):
    c = _c()
    vp = c.c_void_p
    assert lib.pkv_copy_to_device(vp(0), vp(0), c.c_size_t(0), vp(0)) == 0     # nothing to copy
    assert lib.pkv_copy_to_device(vp(0), vp(16), c.c_size_t(64), vp(0)) == -1  # no destination
    assert lib.pkv_copy_to_host(vp(16), vp(0), c.c_size_t(64), vp(0)) == -1    # no source
