"""rotated_bit_kv_gb300: rotation-quantised packed KV cache and compressed-domain
decode attention for one NVIDIA GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/tq.h``: every function here
has the name of the C entry point it marshals arguments for; all work runs in
the library (host C++ for setup, CUDA kernels for the hot path).  PyTorch is
used only for device memory and streams.  Importing works without a GPU; the
first call loads ``_lib/libtq.so`` and raises if it has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from ._build import LIB as _LIB_PATH, build  # noqa: F401

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_NO_CONVERGENCE, TQ_ERR_WORKSPACE = range(6)
TQ_DEV_SEQ_OVER_CAPACITY, TQ_DEV_SEQ_OVER_MAX, TQ_DEV_BAD_POSITION, TQ_DEV_INTERNAL = 1, 2, 4, 8
TQ_DEV_BAD_METADATA = 16
TQ_F32, TQ_F16, TQ_BF16 = 0, 1, 2
TQ_ROT_WHT128, TQ_ROT_WHT32, TQ_ROT_SO4_WHT128 = 0, 1, 2
TQ_PART_K_CODES, TQ_PART_K_NORMS, TQ_PART_V_CODES, TQ_PART_V_NORMS, TQ_PART_PARAMS = range(5)
TQ_VMODE_AUTO, TQ_VMODE_TOKEN_PARALLEL, TQ_VMODE_DIM_PARALLEL, TQ_VMODE_TENSOR, TQ_VMODE_TENSOR_STREAMK = -1, 0, 1, 2, 3
TQ_LAYOUT_NATURAL, TQ_LAYOUT_TILE16 = 0, 1
TQ_HEAD_DIM, TQ_MAX_GROUP, TQ_MAX_SPLITS = 128, 16, 1024


class TQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {tq_status_string(status)} ({status})")


class tq_cache_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "head_dim", "n_q_heads", "n_kv_heads", "batch", "t_capacity", "rot", "k_bits", "v_bits",
        "norm_dtype", "k_mixed", "group", "k_code_bytes", "v_code_bytes", "k_norm_slots",
        "v_norm_slots", "norm_bytes", "layout", "t_alloc")] + [("params_bytes", ctypes.c_int64)]


class tq_cache_ptrs(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_norms", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_norms", ctypes.c_void_p), ("params", ctypes.c_void_p)]


_lib_handle = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGS = {
    "tq_status_string": (ctypes.c_char_p, [_I]),
    "tq_codebook": (_I, [_I, _I, _P, _P]),
    "tq_block_energy": (_I, [_P, _P, _I, _I, _I, _P]),
    "tq_block_bit_alloc": (_I, [_P, _I, _I, _I, _I, _P]),
    "tq_cache_desc_init": (_I, [ctypes.POINTER(tq_cache_desc), _I, _I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "tq_cache_bytes": (ctypes.c_size_t, [ctypes.POINTER(tq_cache_desc), _I]),
    "tq_params_build": (_I, [ctypes.POINTER(tq_cache_desc), _P, _P, _P, _P, _P]),
    "tq_quantize_append": (_I, [ctypes.POINTER(tq_cache_desc), ctypes.POINTER(tq_cache_ptrs), _P, _P, _I, _P,
                                _I, _P, _P]),
    "tq_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tq_cache_desc), _I]),
    "tq_decode_attention": (_I, [ctypes.POINTER(tq_cache_desc), ctypes.POINTER(tq_cache_ptrs), _P, _I, _P, _I,
                                 _P, _P, ctypes.c_size_t, _P, _P]),
    "tq_decode_attention_ex": (_I, [ctypes.POINTER(tq_cache_desc), ctypes.POINTER(tq_cache_ptrs), _P, _I, _P,
                                    _I, _P, _P, ctypes.c_size_t, _P, _P, _I, _I]),
    "tq_decode_plan": (_I, [ctypes.POINTER(tq_cache_desc), _I, _I, _I, _P, _P]),
    "tq_decode_attention_noalloc": (_I, [ctypes.POINTER(tq_cache_desc), ctypes.POINTER(tq_cache_ptrs), _P, _I,
                                         _P, _I, _P, _P, _P]),
    "tq_decode_noalloc_max_scratch_bytes": (ctypes.c_size_t, []),
    "tq_decode_attention_prefix": (_I, [ctypes.POINTER(tq_cache_desc), ctypes.POINTER(tq_cache_ptrs), _P, _I, _P,
                                        _I, _P, _P, _I, _I, _P, _I, _P, _P, ctypes.c_size_t, _P, _P]),
    "tq_decode_prefix_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tq_cache_desc), _I]),
    "tq_zip_pool_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "tq_zip_meta_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "tq_zip_store": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "tq_zip_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "tq_zip_decode_attention": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, ctypes.c_size_t, _P,
                                     _P]),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was never built: there is no fallback)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {_LIB_PATH} is missing; call rotated_bit_kv_gb300.build()")
        h = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = h
    return _lib_handle


def _check(st: int, what: str):
    if st != TQ_OK:
        raise TQError(st, what)


def tq_status_string(s: int) -> str:
    return lib().tq_status_string(int(s)).decode()


# ---------------------------------------------------------------- host API
def tq_codebook(block_dim: int, bits: int):
    """(centroids fp32 [2^bits], boundaries fp32 [2^bits - 1])."""
    c = np.zeros(1 << bits, dtype=np.float32)
    b = np.zeros(max(1, (1 << bits) - 1), dtype=np.float32)
    _check(lib().tq_codebook(block_dim, bits, c.ctypes.data, b.ctypes.data), "tq_codebook")
    return c, b[: (1 << bits) - 1]


def tq_block_energy(q_cal: np.ndarray, k_cal: np.ndarray) -> np.ndarray:
    """q_cal fp32 [T][G][d], k_cal fp32 [T][d] -> s fp64 [d/2]."""
    q = np.ascontiguousarray(q_cal, dtype=np.float32)
    k = np.ascontiguousarray(k_cal, dtype=np.float32)
    T, G, d = q.shape
    if k.shape != (T, d):
        raise ValueError(f"k_cal must be [T][d] = [{T}][{d}] like q_cal's tokens, got {list(k.shape)}")
    s = np.zeros(d // 2, dtype=np.float64)
    _check(lib().tq_block_energy(q.ctypes.data, k.ctypes.data, T, G, d, s.ctypes.data), "tq_block_energy")
    return s


def tq_block_bit_alloc(s, b_min: int, b_max: int, B_total: int) -> np.ndarray:
    s = np.ascontiguousarray(s, dtype=np.float64)
    out = np.zeros(s.size, dtype=np.int32)
    _check(lib().tq_block_bit_alloc(s.ctypes.data, s.size, b_min, b_max, B_total, out.ctypes.data),
           "tq_block_bit_alloc")
    return out


def tq_cache_desc_init(head_dim, n_q_heads, n_kv_heads, batch, t_capacity, rot, k_bits, v_bits, norm_dtype,
                       k_mixed=0) -> tq_cache_desc:
    d = tq_cache_desc()
    _check(lib().tq_cache_desc_init(ctypes.byref(d), head_dim, n_q_heads, n_kv_heads, batch, t_capacity, rot,
                                    k_bits, v_bits, norm_dtype, int(k_mixed)), "tq_cache_desc_init")
    return d


def tq_cache_bytes(desc: tq_cache_desc, part: int) -> int:
    return int(lib().tq_cache_bytes(ctypes.byref(desc), part))


def _params_sizes(desc: tq_cache_desc, signs, quats, k_block_bits, k_group_mats):
    """Check the host arrays against what tq_params_build reads (include/tq.h), so
    that a short array is an error here rather than a read past its end."""
    nkv = int(desc.n_kv_heads)

    def size(x):
        return None if x is None else int(np.asarray(x).size)

    if signs is not None and size(signs) != nkv * 128:
        raise ValueError(f"signs: {size(signs)} values, want n_kv * 128 = {nkv * 128}")
    if quats is not None and size(quats) != nkv * 32 * 8:
        raise ValueError(f"quats: {size(quats)} values, want n_kv * 256 = {nkv * 256}")
    if int(desc.k_mixed):
        if k_block_bits is None or k_group_mats is None:
            raise ValueError("mixed-rate keys need k_block_bits and k_group_mats")
        bb = np.asarray(k_block_bits)
        if bb.size != nkv * 64:
            raise ValueError(f"k_block_bits: {bb.size} values, want n_kv * 64 = {nkv * 64}")
        bb = bb.reshape(nkv, 64)
        need = int(sum((2 * int(np.sum(bb[h] == b))) ** 2 for h in range(nkv) for b in range(1, 5)))
        if size(k_group_mats) != need:
            raise ValueError(f"k_group_mats: {size(k_group_mats)} values, the allocation needs {need}")
    elif int(desc.k_bits) in (1, 2):
        if size(k_group_mats) != nkv * 128 * 128:
            raise ValueError(f"two-stage keys need k_group_mats = the projections, n_kv * 128 * 128 values")


def tq_params_build(desc: tq_cache_desc, signs=None, quats=None, k_block_bits=None, k_group_mats=None) -> np.ndarray:
    """Host parameter blob (uint8); copy it to a 16-byte aligned device buffer.
    k_group_mats: the group matrices of mixed-rate keys, or the projections S
    [n_kv][128][128] of two-stage keys (k_bits 1 or 2)."""
    _params_sizes(desc, signs, quats, k_block_bits, k_group_mats)
    blob = np.zeros(int(desc.params_bytes), dtype=np.uint8)
    keep = []

    def ptr(x, dt):
        if x is None:
            return None
        a = np.ascontiguousarray(x, dtype=dt)
        keep.append(a)
        return a.ctypes.data

    _check(lib().tq_params_build(ctypes.byref(desc), ptr(signs, np.float32), ptr(quats, np.float32),
                                 ptr(k_block_bits, np.int32), ptr(k_group_mats, np.float32), blob.ctypes.data),
           "tq_params_build")
    return blob


# ---------------------------------------------------------------- device API
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    m = {torch.float32: TQ_F32, torch.float16: TQ_F16, torch.bfloat16: TQ_BF16}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("device API arguments must be CUDA tensors")
        if t is not None and not t.is_contiguous():
            raise ValueError("device API arguments must be contiguous")


def tq_quantize_append(desc: tq_cache_desc, cache: tq_cache_ptrs, K, V, start_pos, n_new: int,
                       status=None, stream=None):
    """K, V: CUDA [batch][n_new][n_kv][128] fp32/fp16/bf16; start_pos CUDA int32 [batch]."""
    _require_cuda(K, V, start_pos, status)
    if K.dtype != V.dtype:
        raise TypeError("K and V must share a dtype")
    _check(lib().tq_quantize_append(ctypes.byref(desc), ctypes.byref(cache), _ptr(K), _ptr(V), _dtype_code(K),
                                    _ptr(start_pos), int(n_new), _ptr(status), _stream(stream)),
           "tq_quantize_append")


def tq_decode_workspace_bytes(desc: tq_cache_desc, max_splits: int) -> int:
    return int(lib().tq_decode_workspace_bytes(ctypes.byref(desc), int(max_splits)))


def tq_decode_plan(desc: tq_cache_desc, max_seq_len: int, v_mode: int = TQ_VMODE_AUTO, n_splits: int = 0):
    sp = ctypes.c_int32(0)
    vm = ctypes.c_int32(0)
    _check(lib().tq_decode_plan(ctypes.byref(desc), int(max_seq_len), int(v_mode), int(n_splits),
                                ctypes.addressof(sp), ctypes.addressof(vm)), "tq_decode_plan")
    return sp.value, vm.value


def tq_decode_attention(desc: tq_cache_desc, cache: tq_cache_ptrs, q, seq_lens, max_seq_len: int, out,
                        workspace, status=None, stream=None):
    """q CUDA [batch][n_q][128]; seq_lens CUDA int32 [batch]; out CUDA fp32 [batch][n_q][128]."""
    _require_cuda(q, seq_lens, out, workspace, status)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tq_decode_attention(ctypes.byref(desc), ctypes.byref(cache), _ptr(q), _dtype_code(q),
                                     _ptr(seq_lens), int(max_seq_len), _ptr(out), _ptr(workspace), nbytes,
                                     _ptr(status), _stream(stream)), "tq_decode_attention")


def tq_decode_attention_ex(desc: tq_cache_desc, cache: tq_cache_ptrs, q, seq_lens, max_seq_len: int, out,
                           workspace, status=None, stream=None, v_mode: int = TQ_VMODE_AUTO, n_splits: int = 0):
    _require_cuda(q, seq_lens, out, workspace, status)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tq_decode_attention_ex(ctypes.byref(desc), ctypes.byref(cache), _ptr(q), _dtype_code(q),
                                        _ptr(seq_lens), int(max_seq_len), _ptr(out), _ptr(workspace), nbytes,
                                        _ptr(status), _stream(stream), int(v_mode), int(n_splits)),
           "tq_decode_attention_ex")


def tq_decode_noalloc_max_scratch_bytes() -> int:
    return int(lib().tq_decode_noalloc_max_scratch_bytes())


def tq_decode_attention_noalloc(desc: tq_cache_desc, cache: tq_cache_ptrs, q, seq_lens, max_seq_len: int, out,
                                status=None, stream=None):
    """Decode attention without a workspace: the split-K scratch is the
    library's fixed device array (for callers that cannot allocate)."""
    _require_cuda(q, seq_lens, out, status)
    _check(lib().tq_decode_attention_noalloc(ctypes.byref(desc), ctypes.byref(cache), _ptr(q), _dtype_code(q),
                                             _ptr(seq_lens), int(max_seq_len), _ptr(out), _ptr(status),
                                             _stream(stream)), "tq_decode_attention_noalloc")


def tq_decode_prefix_workspace_bytes(desc: tq_cache_desc, max_prefix_len: int) -> int:
    return int(lib().tq_decode_prefix_workspace_bytes(ctypes.byref(desc), int(max_prefix_len)))


def tq_decode_attention_prefix(desc: tq_cache_desc, cache: tq_cache_ptrs, q, seq_lens, max_seq_len: int,
                               k_prefix, v_prefix, prefix_lens, max_prefix_len: int, out, workspace, status=None,
                               stream=None):
    """Attention over the unquantised tokens k_prefix / v_prefix (CUDA
    [batch][capacity][n_kv][128] fp32/fp16/bf16, the first prefix_lens[b] of
    batch b) plus the packed cache (the first seq_lens[b] tokens); out CUDA fp32
    [batch][n_q][128]; workspace zero-filled before its first use."""
    _require_cuda(q, seq_lens, k_prefix, v_prefix, prefix_lens, out, workspace, status)
    if k_prefix is not None and (v_prefix is None or k_prefix.dtype != v_prefix.dtype or
                                 k_prefix.shape != v_prefix.shape):
        raise TypeError("k_prefix and v_prefix must share a dtype and a shape")
    cap = 0 if k_prefix is None else int(k_prefix.shape[1])
    pdt = TQ_F16 if k_prefix is None else _dtype_code(k_prefix)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tq_decode_attention_prefix(ctypes.byref(desc), ctypes.byref(cache), _ptr(q), _dtype_code(q),
                                            _ptr(seq_lens), int(max_seq_len), _ptr(k_prefix), _ptr(v_prefix), pdt,
                                            cap, _ptr(prefix_lens), int(max_prefix_len), _ptr(out), _ptr(workspace),
                                            nbytes, _ptr(status), _stream(stream)), "tq_decode_attention_prefix")


def tq_zip_pool_bytes(batch: int, n_kv_heads: int, t_capacity: int) -> int:
    return int(lib().tq_zip_pool_bytes(int(batch), int(n_kv_heads), int(t_capacity)))


def tq_zip_meta_bytes(batch: int, n_kv_heads: int, t_capacity: int) -> int:
    return int(lib().tq_zip_meta_bytes(int(batch), int(n_kv_heads), int(t_capacity)))


def tq_zip_workspace_bytes(batch: int, n_q_heads: int, n_kv_heads: int, max_seq_len: int) -> int:
    return int(lib().tq_zip_workspace_bytes(int(batch), int(n_q_heads), int(n_kv_heads), int(max_seq_len)))


def tq_zip_store(K, V, lens, t_capacity: int, k_pool, v_pool, k_meta, v_meta, status=None, stream=None):
    """K, V: CUDA bf16 [batch][n_tokens][n_kv][128]; lens CUDA int32 [batch]."""
    _require_cuda(K, V, lens, k_pool, v_pool, k_meta, v_meta, status)
    torch = _torch()
    if K.dtype != torch.bfloat16 or V.dtype != torch.bfloat16 or K.shape != V.shape:
        raise TypeError("K and V must be bf16 tensors of one shape")
    B, T, Hkv, d = K.shape
    _check(lib().tq_zip_store(_ptr(K), _ptr(V), B, Hkv, T, int(t_capacity), _ptr(lens), _ptr(k_pool), _ptr(v_pool),
                              _ptr(k_meta), _ptr(v_meta), _ptr(status), _stream(stream)), "tq_zip_store")


def tq_zip_decode_attention(q, n_kv_heads: int, t_capacity: int, k_pool, v_pool, k_meta, v_meta, seq_lens,
                            max_seq_len: int, out, workspace, status=None, stream=None):
    _require_cuda(q, k_pool, v_pool, k_meta, v_meta, seq_lens, out, workspace, status)
    B, Hq, d = q.shape
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tq_zip_decode_attention(_ptr(q), _dtype_code(q), B, Hq, int(n_kv_heads), int(t_capacity),
                                         _ptr(k_pool), _ptr(v_pool), _ptr(k_meta), _ptr(v_meta), _ptr(seq_lens),
                                         int(max_seq_len), _ptr(out), _ptr(workspace), nbytes, _ptr(status),
                                         _stream(stream)), "tq_zip_decode_attention")


class ZipKVCache:
    """Device buffers of a ZipFusion store (pools, metadata, workspace, status),
    allocated through PyTorch."""

    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, t_capacity: int, device="cuda"):
        torch = _torch()
        self.batch, self.n_q_heads, self.n_kv_heads, self.t_capacity = batch, n_q_heads, n_kv_heads, t_capacity
        self.device = torch.device(device)

        def buf(n):
            return torch.zeros(max(int(n), 16), dtype=torch.uint8, device=self.device)

        self.k_pool = buf(tq_zip_pool_bytes(batch, n_kv_heads, t_capacity))
        self.v_pool = buf(tq_zip_pool_bytes(batch, n_kv_heads, t_capacity))
        self.k_meta = buf(tq_zip_meta_bytes(batch, n_kv_heads, t_capacity))
        self.v_meta = buf(tq_zip_meta_bytes(batch, n_kv_heads, t_capacity))
        self.workspace = buf(tq_zip_workspace_bytes(batch, n_q_heads, n_kv_heads, t_capacity))
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def store(self, K, V, lens, stream=None):
        tq_zip_store(K, V, lens, self.t_capacity, self.k_pool, self.v_pool, self.k_meta, self.v_meta, self.status,
                     stream)

    def decode(self, q, seq_lens, max_seq_len, out=None, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        tq_zip_decode_attention(q, self.n_kv_heads, self.t_capacity, self.k_pool, self.v_pool, self.k_meta,
                                self.v_meta, seq_lens, max_seq_len, out, self.workspace, self.status, stream)
        return out


# ---------------------------------------------------------------- allocation helper
class PackedKVCache:
    """Device buffers of one packed cache, allocated through PyTorch (the
    library itself never allocates).  Holds the descriptor, the cache parts,
    the parameter blob, a zeroed decode workspace and a status word."""

    def __init__(self, desc: tq_cache_desc, params_blob: np.ndarray, device="cuda", max_splits: int = TQ_MAX_SPLITS):
        torch = _torch()
        self.desc = desc
        self.device = torch.device(device)

        def buf(n):
            # 256-byte aligned allocations (PyTorch's caching allocator aligns to 512)
            return torch.zeros(max(int(n), 16), dtype=torch.uint8, device=self.device)

        self.k_codes = buf(tq_cache_bytes(desc, TQ_PART_K_CODES))
        self.k_norms = buf(tq_cache_bytes(desc, TQ_PART_K_NORMS))
        self.v_codes = buf(tq_cache_bytes(desc, TQ_PART_V_CODES))
        self.v_norms = buf(tq_cache_bytes(desc, TQ_PART_V_NORMS))
        self.params = torch.from_numpy(np.ascontiguousarray(params_blob)).to(self.device)
        self.workspace = buf(tq_decode_workspace_bytes(desc, max_splits))
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.ptrs = tq_cache_ptrs(self.k_codes.data_ptr(), self.k_norms.data_ptr(), self.v_codes.data_ptr(),
                                  self.v_norms.data_ptr(), self.params.data_ptr())

    def append(self, K, V, start_pos, stream=None):
        tq_quantize_append(self.desc, self.ptrs, K, V, start_pos, K.shape[1], self.status, stream)

    def decode(self, q, seq_lens, max_seq_len, out=None, v_mode=TQ_VMODE_AUTO, n_splits=0, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        tq_decode_attention_ex(self.desc, self.ptrs, q, seq_lens, max_seq_len, out, self.workspace, self.status,
                               stream, v_mode, n_splits)
        return out

    def decode_prefix(self, q, seq_lens, max_seq_len, k_prefix, v_prefix, prefix_lens, max_prefix_len, out=None,
                      stream=None):
        """Attention over the unquantised tokens k_prefix / v_prefix plus the
        packed cache (tq_decode_attention_prefix); the workspace grows as needed."""
        torch = _torch()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        need = tq_decode_prefix_workspace_bytes(self.desc, max_prefix_len)
        if getattr(self, "prefix_workspace", None) is None or self.prefix_workspace.numel() < need:
            self.prefix_workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=self.device)
        tq_decode_attention_prefix(self.desc, self.ptrs, q, seq_lens, max_seq_len, k_prefix, v_prefix, prefix_lens,
                                   max_prefix_len, out, self.prefix_workspace, self.status, stream)
        return out

    def norms_view(self, which: str):
        """The norms array as stored: [batch][n_kv][t_alloc * slots] (norm dtype);
        in the tile layout the positions within each 16-token tile are permuted
        as include/tq.h documents."""
        torch = _torch()
        d = self.desc
        slots = d.k_norm_slots if which == "k" else d.v_norm_slots
        raw = self.k_norms if which == "k" else self.v_norms
        dt = torch.float16 if d.norm_dtype == TQ_F16 else torch.float32
        n = d.batch * d.n_kv_heads * d.t_alloc * slots
        return raw[: n * d.norm_bytes].view(dt).view(d.batch, d.n_kv_heads, d.t_alloc * slots)

    def codes_view(self, which: str):
        """The code array as stored: [batch][n_kv][t_alloc * code_bytes] uint8."""
        d = self.desc
        nb = d.k_code_bytes if which == "k" else d.v_code_bytes
        raw = self.k_codes if which == "k" else self.v_codes
        return raw[: d.batch * d.n_kv_heads * d.t_alloc * nb].view(d.batch, d.n_kv_heads, d.t_alloc * nb)
