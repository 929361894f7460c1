"""pagedattention_paged_kv_gb300 -- attention over a block-paged KV cache on GB300.

A thin Python binding of ``libpagedkv.so`` (C ABI in ``include/pagedkv.h``).  The
functions take torch tensors only for their device pointers, sizes and the current
CUDA stream; every step of the computation runs in the library's sm_103a kernels.
There is no fallback: if the library is missing or fails to load, every call raises.

Calls (names as in the C ABI, without the ``pkv_`` prefix):
  reshape_and_cache         KV write through a slot mapping
  paged_attention_decode    one query row per sequence
  paged_attention_varlen    ragged batch: prefill chunks and decodes in one call
  workspace_size            device scratch the attention calls need
  get_device_error          flags the kernels raised on bad device metadata
  slot_mapping              host: slot of each new token from the block tables
  BlockManager              host: free-list allocator of physical block ids
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

BLOCK_SIZE = 16
OP_DECODE = 0
OP_VARLEN = 1
DTYPE_BF16 = 0
DTYPE_FP8_E4M3 = 1

_STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported configuration",
           -3: "workspace too small", -4: "CUDA error", -5: "out of blocks",
           -6: "invalid device data"}

DEVERR_SLOT = 0x1
DEVERR_BLOCK_ID = 0x2
DEVERR_CONTEXT_LEN = 0x4
DEVERR_QUERY_LEN = 0x8
DEVERR_TIMEOUT = 0x10

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")
_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, 'status %d' % status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built (see _build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "pagedattention_paged_kv_gb300._build.build_library()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                 ctypes.c_float)
        L.pkv_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, i32, vp]
        L.pkv_paged_attention_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                 i32, i64, f32, i32, vp, sz, vp]
        L.pkv_paged_attention_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                 i32, i32, i32, i32, i64, f32, i32, i32, vp, sz, vp]
        L.pkv_paged_attention_varlen_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                     i32, i32, i32, i32, i64, f32, i32, f32, f32, vp, sz, vp]
        L.pkv_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, f32, f32, vp]
        L.pkv_paged_attention_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                     i32, i64, f32, f32, f32, vp, sz, vp]
        L.pkv_copy_blocks.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, i32, vp]
        L.pkv_paged_attention_decode_kvwrite.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                         i32, i32, i64, f32, i32, vp, sz, vp]
        L.pkv_paged_attention_decode_kvwrite_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                             i32, i32, i32, i64, f32, f32, f32, vp, sz, vp]
        L.pkv_block_manager_share.argtypes = [vp, vp, i64]
        L.pkv_block_manager_ref_count.argtypes = [vp, ctypes.c_int32]
        L.pkv_block_manager_copy_on_write.argtypes = [vp, ctypes.c_int32, vp]
        L.pkv_copy_to_device.argtypes = [vp, vp, sz, vp]
        L.pkv_copy_to_host.argtypes = [vp, vp, sz, vp]
        L.pkv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.pkv_set_wait_limit_ns.restype = None
        L.pkv_set_decode_split.argtypes = [ctypes.c_int]
        L.pkv_set_decode_split.restype = None
        L.pkv_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        L.pkv_workspace_size.restype = sz
        L.pkv_status_string.argtypes = [i32]
        L.pkv_status_string.restype = ctypes.c_char_p
        L.pkv_get_device_error.argtypes = [vp]
        L.pkv_slot_mapping.argtypes = [vp, vp, i32, vp, vp, i64, i32]
        L.pkv_block_manager_create.argtypes = [i64, i32]
        L.pkv_block_manager_create.restype = vp
        L.pkv_block_manager_destroy.argtypes = [vp]
        L.pkv_block_manager_allocate.argtypes = [vp, i64, vp]
        L.pkv_block_manager_free.argtypes = [vp, vp, i64]
        L.pkv_block_manager_num_free.argtypes = [vp]
        L.pkv_block_manager_num_free.restype = i64
        for name in ("pkv_reshape_and_cache", "pkv_paged_attention_decode", "pkv_reshape_and_cache_fp8",
                     "pkv_paged_attention_decode_fp8",
                     "pkv_paged_attention_varlen", "pkv_paged_attention_varlen_fp8", "pkv_get_device_error", "pkv_slot_mapping",
                     "pkv_block_manager_allocate", "pkv_block_manager_free", "pkv_copy_blocks",
                     "pkv_block_manager_share", "pkv_block_manager_ref_count",
                     "pkv_block_manager_copy_on_write", "pkv_paged_attention_decode_kvwrite",
                     "pkv_paged_attention_decode_kvwrite_fp8", "pkv_copy_to_device", "pkv_copy_to_host"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise PagedKVError(status, what)


# ---------------------------------------------------------------------------
# device calls (torch tensors)
# ---------------------------------------------------------------------------

def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _require(t, dtype, name, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def reshape_and_cache(k_cache, v_cache, k, v, slot_mapping, stream=None) -> None:
    """k_cache/v_cache [NB, bs, Hkv, d] bf16 <- k/v [T, Hkv, d] bf16 at int64 slot_mapping [T]."""
    import torch
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, torch.bfloat16, n, 4)
    for t, n in ((k, "k"), (v, "v")):
        _require(t, torch.bfloat16, n, 3)
    _require(slot_mapping, torch.int64, "slot_mapping", 1)
    NB, bs, Hkv, d = k_cache.shape
    T = k.shape[0]
    if v_cache.shape != k_cache.shape or v.shape != k.shape or tuple(k.shape[1:]) != (Hkv, d) \
            or slot_mapping.shape[0] != T:
        raise ValueError("shape mismatch")
    _check(lib().pkv_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v),
                                       _ptr(slot_mapping), T, NB, bs, Hkv, d, DTYPE_BF16,
                                       _stream_ptr(stream)), "reshape_and_cache")


def workspace_size(op: int, num_seqs: int, total_q_tokens: int, num_heads: int, num_kv_heads: int,
                   head_dim: int, block_size: int = BLOCK_SIZE) -> int:
    n = lib().pkv_workspace_size(op, num_seqs, total_q_tokens, num_heads, num_kv_heads, head_dim,
                                 block_size)
    if n == 0:
        raise PagedKVError(-2, "workspace_size")
    return int(n)


def _workspace(workspace, nbytes, device):
    import torch
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise PagedKVError(-3, "workspace")
    return workspace


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           workspace=None, stream=None) -> None:
    """out/q [S, Hq, d] bf16; k_cache/v_cache [NB, bs, Hkv, d] bf16; block_tables [S, MB]
    int32; context_lens [S] int32."""
    import torch
    _require(out, torch.bfloat16, "out", 3)
    _require(q, torch.bfloat16, "q", 3)
    _require(k_cache, torch.bfloat16, "k_cache", 4)
    _require(v_cache, torch.bfloat16, "v_cache", 4)
    _require(block_tables, torch.int32, "block_tables", 2)
    _require(context_lens, torch.int32, "context_lens", 1)
    S, Hq, d = q.shape
    NB, bs, Hkv, d2 = k_cache.shape
    if out.shape != q.shape or d2 != d or v_cache.shape != k_cache.shape \
            or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("shape mismatch")
    nbytes = workspace_size(OP_DECODE, S, S, Hq, Hkv, d, bs)
    ws = _workspace(workspace, nbytes, q.device)
    _check(lib().pkv_paged_attention_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        S, block_tables.shape[1], Hq, Hkv, d, bs, NB, float(scale), DTYPE_BF16, _ptr(ws),
        ws.numel() * ws.element_size(), _stream_ptr(stream)), "paged_attention_decode")


def reshape_and_cache_fp8(k_cache, v_cache, k, v, slot_mapping, k_scale: float, v_scale: float,
                          stream=None) -> None:
    """FP8 cache: k_cache/v_cache [NB, bs, Hkv, d] uint8 (e4m3 codes) <- k/v [T, Hkv, d] bf16,
    each element stored as e4m3(fp32(x) / scale) (k_scale for K, v_scale for V)."""
    import torch
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, torch.uint8, n, 4)
    for t, n in ((k, "k"), (v, "v")):
        _require(t, torch.bfloat16, n, 3)
    _require(slot_mapping, torch.int64, "slot_mapping", 1)
    NB, bs, Hkv, d = k_cache.shape
    T = k.shape[0]
    if v_cache.shape != k_cache.shape or v.shape != k.shape or tuple(k.shape[1:]) != (Hkv, d) \
            or slot_mapping.shape[0] != T:
        raise ValueError("shape mismatch")
    _check(lib().pkv_reshape_and_cache_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v),
                                           _ptr(slot_mapping), T, NB, bs, Hkv, d, float(k_scale),
                                           float(v_scale), _stream_ptr(stream)), "reshape_and_cache_fp8")


def paged_attention_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                               k_scale: float, v_scale: float, workspace=None, stream=None) -> None:
    """Decode over an FP8 cache: out/q [S, Hq, d] bf16; k_cache/v_cache [NB, bs, Hkv, d] uint8
    e4m3 codes (element = code value x k_scale / v_scale); block_tables [S, MB] int32;
    context_lens [S] int32."""
    import torch
    _require(out, torch.bfloat16, "out", 3)
    _require(q, torch.bfloat16, "q", 3)
    _require(k_cache, torch.uint8, "k_cache", 4)
    _require(v_cache, torch.uint8, "v_cache", 4)
    _require(block_tables, torch.int32, "block_tables", 2)
    _require(context_lens, torch.int32, "context_lens", 1)
    S, Hq, d = q.shape
    NB, bs, Hkv, d2 = k_cache.shape
    if out.shape != q.shape or d2 != d or v_cache.shape != k_cache.shape \
            or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("shape mismatch")
    nbytes = workspace_size(OP_DECODE, S, S, Hq, Hkv, d, bs)
    ws = _workspace(workspace, nbytes, q.device)
    _check(lib().pkv_paged_attention_decode_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        S, block_tables.shape[1], Hq, Hkv, d, bs, NB, float(scale), float(k_scale), float(v_scale),
        _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream)), "paged_attention_decode_fp8")


def paged_attention_varlen(out, q, query_start_loc, k_cache, v_cache, block_tables, context_lens,
                           scale: float, causal: bool = True, max_q_len: int | None = None,
                           workspace=None, stream=None, k_scale: float | None = None,
                           v_scale: float | None = None) -> None:
    """out/q [total_q, Hq, d] bf16; query_start_loc [S+1] int32 (on the device);
    max_q_len is the longest q_len (read back from the device if not given).  A uint8
    (e4m3) cache needs k_scale and v_scale; a bf16 cache takes none."""
    import torch
    fp8 = k_cache.dtype == torch.uint8
    _require(out, torch.bfloat16, "out", 3)
    _require(q, torch.bfloat16, "q", 3)
    _require(query_start_loc, torch.int32, "query_start_loc", 1)
    _require(k_cache, torch.uint8 if fp8 else torch.bfloat16, "k_cache", 4)
    _require(v_cache, k_cache.dtype, "v_cache", 4)
    _require(block_tables, torch.int32, "block_tables", 2)
    _require(context_lens, torch.int32, "context_lens", 1)
    total_q, Hq, d = q.shape
    NB, bs, Hkv, d2 = k_cache.shape
    S = context_lens.shape[0]
    if out.shape != q.shape or d2 != d or v_cache.shape != k_cache.shape \
            or block_tables.shape[0] != S or query_start_loc.shape[0] != S + 1:
        raise ValueError("shape mismatch")
    if fp8 and (k_scale is None or v_scale is None):
        raise ValueError("an FP8 cache needs k_scale and v_scale")
    if max_q_len is None:
        max_q_len = int((query_start_loc[1:] - query_start_loc[:-1]).max().item()) if S else 0
    nbytes = workspace_size(OP_VARLEN, S, total_q, Hq, Hkv, d, bs)
    ws = _workspace(workspace, nbytes, q.device)
    args = [_ptr(out), _ptr(q), _ptr(query_start_loc), _ptr(k_cache), _ptr(v_cache),
            _ptr(block_tables), _ptr(context_lens), S, total_q, int(max_q_len), block_tables.shape[1],
            Hq, Hkv, d, bs, NB, float(scale), int(bool(causal))]
    tail = [_ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream)]
    if fp8:
        _check(lib().pkv_paged_attention_varlen_fp8(*args, float(k_scale), float(v_scale), *tail),
               "paged_attention_varlen_fp8")
    else:
        _check(lib().pkv_paged_attention_varlen(*args, DTYPE_BF16, *tail), "paged_attention_varlen")


def paged_attention_decode_kvwrite(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                                   scale: float, k_scale: float | None = None, v_scale: float | None = None,
                                   workspace=None, stream=None) -> None:
    """Decode step with the KV write fused in: k_new/v_new [S, Hkv, d] bf16 rows go to position
    context_lens[s] - 1, then out = decode attention.  A uint8 (e4m3) cache needs k_scale and
    v_scale; a bf16 cache takes none."""
    import torch
    fp8 = k_cache.dtype == torch.uint8
    _require(out, torch.bfloat16, "out", 3)
    _require(q, torch.bfloat16, "q", 3)
    _require(k_new, torch.bfloat16, "k_new", 3)
    _require(v_new, torch.bfloat16, "v_new", 3)
    _require(k_cache, torch.uint8 if fp8 else torch.bfloat16, "k_cache", 4)
    _require(v_cache, k_cache.dtype, "v_cache", 4)
    _require(block_tables, torch.int32, "block_tables", 2)
    _require(context_lens, torch.int32, "context_lens", 1)
    S, Hq, d = q.shape
    NB, bs, Hkv, d2 = k_cache.shape
    if out.shape != q.shape or d2 != d or v_cache.shape != k_cache.shape or block_tables.shape[0] != S \
            or context_lens.shape[0] != S or tuple(k_new.shape) != (S, Hkv, d) or v_new.shape != k_new.shape:
        raise ValueError("shape mismatch")
    if fp8 and (k_scale is None or v_scale is None):
        raise ValueError("an FP8 cache needs k_scale and v_scale")
    nbytes = workspace_size(OP_DECODE, S, S, Hq, Hkv, d, bs)
    ws = _workspace(workspace, nbytes, q.device)
    args = [_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(context_lens), S, block_tables.shape[1], Hq, Hkv, d, bs, NB, float(scale)]
    tail = [_ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream)]
    if fp8:
        _check(lib().pkv_paged_attention_decode_kvwrite_fp8(*args, float(k_scale), float(v_scale), *tail),
               "paged_attention_decode_kvwrite_fp8")
    else:
        _check(lib().pkv_paged_attention_decode_kvwrite(*args, DTYPE_BF16, *tail), "paged_attention_decode_kvwrite")


def copy_blocks(k_cache, v_cache, block_pairs, stream=None) -> None:
    """k_cache[dst] = k_cache[src], v_cache[dst] = v_cache[src] for each row (src, dst) of
    block_pairs (int32 [n, 2] on the device); caches bf16 or uint8 (FP8 codes)."""
    import torch
    if k_cache.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif k_cache.dtype == torch.uint8:
        dt = DTYPE_FP8_E4M3
    else:
        raise ValueError("k_cache must be bf16 or uint8")
    _require(k_cache, k_cache.dtype, "k_cache", 4)
    _require(v_cache, k_cache.dtype, "v_cache", 4)
    _require(block_pairs, torch.int32, "block_pairs", 2)
    if v_cache.shape != k_cache.shape or block_pairs.shape[1] != 2:
        raise ValueError("shape mismatch")
    NB, bs, Hkv, d = k_cache.shape
    _check(lib().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), block_pairs.shape[0], NB,
                                 bs, Hkv, d, dt, _stream_ptr(stream)), "copy_blocks")


def attention_launches(max_q_len: int) -> int:
    """Kernels one paged_attention_varlen call launches for a batch whose longest q_len is
    max_q_len: the decode kernel and its merge; or, when some sequence has q_len >= 2, the
    one varlen kernel (decode and prefill CTAs) and the two merges."""
    return 2 if max_q_len < 2 else 3


def set_wait_limit_ns(limit_ns: int) -> None:
    """Limit of the kernels' pipeline waits for launches from now on (0: the default,
    2 s).  A wait that runs out flags DEVERR_TIMEOUT and the kernel returns; short limits
    exist to test that failure path."""
    lib().pkv_set_wait_limit_ns(int(limit_ns))


def set_decode_split(enabled: bool) -> None:
    """Split-K of the decode rows for launches from now on (default on).  Off, every
    (sequence, KV-head tile) item is computed whole by one CTA: the split's ablation."""
    lib().pkv_set_decode_split(1 if enabled else 0)


def get_device_error(stream=None) -> int:
    """Synchronizes the stream and returns (and clears) the device error flags."""
    r = lib().pkv_get_device_error(_stream_ptr(stream))
    if r < 0:
        raise PagedKVError(r, "get_device_error")
    return r


# ---------------------------------------------------------------------------
# host calls (numpy)
# ---------------------------------------------------------------------------

def slot_mapping(block_tables: np.ndarray, token_seq: np.ndarray, token_pos: np.ndarray,
                 block_size: int = BLOCK_SIZE) -> np.ndarray:
    """int64 slot of each new token (host)."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ts = np.ascontiguousarray(token_seq, dtype=np.int32)
    tp = np.ascontiguousarray(token_pos, dtype=np.int32)
    out = np.empty(ts.shape[0], dtype=np.int64)
    _check(lib().pkv_slot_mapping(out.ctypes.data, bt.ctypes.data, bt.shape[1] if bt.ndim == 2 else 0,
                                  ts.ctypes.data, tp.ctypes.data, ts.shape[0], block_size),
           "slot_mapping")
    return out


class OutOfBlocks(PagedKVError):
    pass


class BlockManager:
    """Free list of physical block ids over a pool of num_blocks blocks (host, C++)."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE):
        self._h = lib().pkv_block_manager_create(int(num_blocks), int(block_size))
        if not self._h:
            raise PagedKVError(-1, "BlockManager")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.pkv_block_manager_destroy(h)

    def allocate(self, n: int) -> list[int]:
        ids = np.empty(max(int(n), 1), dtype=np.int32)
        st = lib().pkv_block_manager_allocate(self._h, int(n), ids.ctypes.data)
        if st == -5:
            raise OutOfBlocks(st, f"allocate({n}) with {self.num_free()} free")
        _check(st, "allocate")
        return ids[:n].tolist()

    def free(self, ids) -> None:
        arr = np.ascontiguousarray(list(ids), dtype=np.int32)
        _check(lib().pkv_block_manager_free(self._h, arr.ctypes.data, arr.shape[0]), "free")

    def num_free(self) -> int:
        return int(lib().pkv_block_manager_num_free(self._h))

    def share(self, ids) -> None:
        """One more holder for each listed (held) block: read-only sharing."""
        arr = np.ascontiguousarray(list(ids), dtype=np.int32)
        _check(lib().pkv_block_manager_share(self._h, arr.ctypes.data, arr.shape[0]), "share")

    def ref_count(self, block_id: int) -> int:
        r = int(lib().pkv_block_manager_ref_count(self._h, int(block_id)))
        if r < 0:
            raise PagedKVError(r, "ref_count")
        return r

    def copy_on_write(self, block_id: int) -> tuple[int, bool]:
        """(id to write into, whether the block must be copied there first)."""
        new = ctypes.c_int32(-1)
        st = int(lib().pkv_block_manager_copy_on_write(self._h, int(block_id), ctypes.byref(new)))
        if st == -5:
            raise OutOfBlocks(st, "copy_on_write")
        if st < 0:
            raise PagedKVError(st, "copy_on_write")
        return int(new.value), st == 1


def copy_to_device(dst, src, stream=None) -> None:
    """dst (CUDA tensor) <- src (CPU tensor, ideally pinned), same byte size, both
    contiguous; asynchronous on the stream.  Pinned host memory is read by the SMs."""
    if not (dst.is_cuda and not src.is_cuda and dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy_to_device needs a contiguous CUDA dst and a contiguous CPU src")
    n = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != n:
        raise ValueError("size mismatch")
    _check(lib().pkv_copy_to_device(_ptr(dst), _ptr(src), n, _stream_ptr(stream)), "copy_to_device")


def copy_to_host(dst, src, stream=None) -> None:
    """dst (CPU tensor, ideally pinned) <- src (CUDA tensor), same byte size, both
    contiguous; asynchronous on the stream.  Pinned host memory is written by the SMs."""
    if not (src.is_cuda and not dst.is_cuda and dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy_to_host needs a contiguous CPU dst and a contiguous CUDA src")
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("size mismatch")
    _check(lib().pkv_copy_to_host(_ptr(dst), _ptr(src), n, _stream_ptr(stream)), "copy_to_host")
