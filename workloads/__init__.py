"""Seeded synthetic workloads for the rotation-quantised KV cache.

This module is shared by the fp64 oracle's tests, the GPU parity tests and the
benchmark.  It holds shapes, value distributions and random draws only: none of
the method's arithmetic (no norm, rotation, codebook, packing or attention).
Random quantities that the method itself draws (the +-1 sign vector of the
sign-flipped Walsh-Hadamard transform, the unit quaternions of the SO(4)
rotation, the random orthogonal matrix of each mixed-rate key group) are drawn
here and handed to both the oracle and the CUDA library as inputs.

Every array is produced from ``np.random.default_rng(seed)`` in a fixed draw
order (outlier/scale channels -> K -> V -> calibration q -> decode q ->
rotation parameters), so the oracle and the GPU see the same bytes.  The
matrices drawn per head (mixed-rate key groups, two-stage key projections)
come from streams of their own.

bf16 tensors are represented as ``uint16`` bit patterns, obtained by
round-to-nearest-even from the fp32 samples.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

HEAD_DIM = 128

# Rotation kinds (same integer values as the C header).
ROT_WHT128 = 0        # y = H_128 . diag(signs) . x
ROT_WHT32 = 1         # four independent 32-point sign-flipped WHTs
ROT_SO4_WHT128 = 2    # y = S . H_128 . x with 32 quaternion-pair 4x4 blocks
ROT_GROUP_DENSE = 3   # mixed-rate keys: one random orthogonal matrix per bit group

F32, F16, BF16 = 0, 1, 2


# ----------------------------------------------------------------------------
# dtype helpers (input preparation, not method arithmetic)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 samples to bf16 (round-to-nearest-even); return uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_float64(x: np.ndarray, dtype: int) -> np.ndarray:
    """Exact value of an input tensor stored as `dtype` (uint16 bits for bf16)."""
    if dtype == BF16:
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x).astype(np.float64)


# ----------------------------------------------------------------------------
# workload descriptions
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    n_q_heads: int
    n_kv_heads: int
    batch: int
    seq_len: int
    rot: int
    k_bits: int
    v_bits: int
    in_dtype: int          # dtype of K, V and q
    norm_dtype: int        # F32 or F16
    k_recipe: str          # "outlier4x20", "lognormal_outlier", "rope_decay"
    v_recipe: str          # "outlier4x20", "normal"
    q_recipe: str          # "normal", "rope_decay"
    mixed_k: bool = False  # mixed-rate keys (greedy RoPE-block bit allocation)
    tight_k: bool = False  # mixed-rate keys packed at their own widths (avg_bits * 16 B records)
    b_min: int = 1
    b_max: int = 4
    avg_bits: int = 3
    calib_tokens: int = 512
    seed: int = 0
    head_dim: int = HEAD_DIM

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def tiny_single_head(seed: int = 0) -> Workload:
    """1 query head, 1 KV head, d=128, T=256, batch 1; fp32 N(0,1) K/V with four
    fixed channels scaled x20; 128-point WHT with a seeded sign vector; 3-bit
    codes; one fp32 norm per vector."""
    return Workload("tiny_single_head", 1, 1, 1, 256, ROT_WHT128, 3, 3, F32, F32,
                    "outlier4x20", "outlier4x20", "normal", seed=seed)


def llama8b_decode(seq_len: int = 8192, batch: int = 32, seed: int = 0) -> Workload:
    """Llama-3.1-8B-shaped decode: 32 query heads, 8 KV heads, d=128, bf16 q/K/V,
    3-bit K and V, one 128-wide sign-flipped WHT block per vector, fp16 norm.
    K channel scales lognormal(0, 0.5) with 2% of channels x15; V ~ N(0,1)."""
    return Workload("llama8b_decode", 32, 8, batch, seq_len, ROT_WHT128, 3, 3, BF16, F16,
                    "lognormal_outlier", "normal", "normal", seed=seed)


def block32(bits: int = 3, seq_len: int = 8192, batch: int = 8, seed: int = 0) -> Workload:
    """head_dim split into four 32-dim blocks, each with its own fp16 norm and its
    own 5-stage sign-flipped WHT; TQ3 or TQ4 for both K and V."""
    return Workload(f"block32_tq{bits}", 32, 8, batch, seq_len, ROT_WHT32, bits, bits, BF16, F16,
                    "lognormal_outlier", "normal", "normal", seed=seed)


def so4_wht(seq_len: int = 8192, seed: int = 0) -> Workload:
    """128-point WHT followed by 32 quaternion-pair 4x4 rotations; 3-bit codes;
    32 query heads, 4 KV heads, batch 1."""
    return Workload("so4_wht", 32, 4, 1, seq_len, ROT_SO4_WHT128, 3, 3, BF16, F16,
                    "lognormal_outlier", "normal", "normal", seed=seed)


def mixed_rate_long(seq_len: int = 131072, seed: int = 0) -> Workload:
    """Long-context split-K with mixed-rate keys: 16 query heads, 2 KV heads,
    d=128 (64 two-dim RoPE blocks), batch 1.  q/k block i scaled by 10^(-2i/64);
    greedy bit allocation (b_min=1, b_max=4, 3 bits/coordinate on average) from
    the first 512 tokens; uniform 3-bit V with a sign-flipped 128-point WHT."""
    return Workload("mixed_rate_long", 16, 2, 1, seq_len, ROT_WHT128, 3, 3, BF16, F16,
                    "rope_decay", "normal", "rope_decay", mixed_k=True, seed=seed)


def two_stage_keys(k_bits: int = 2, seq_len: int = 8192, batch: int = 8, seed: int = 0) -> Workload:
    """Keys at 1 or 2 bits with the two-stage code ((k_bits - 1)-bit MSE code plus
    a 1-bit QJL code of the residual, its projection drawn by two_stage_projection);
    Llama-3.1-8B-shaped heads (32 query / 8 KV, d = 128), bf16 q/K/V, 3-bit V, one
    128-wide sign-flipped WHT, fp16 norms; K channel scales lognormal(0, 0.5) with
    2% of channels x15; V ~ N(0,1)."""
    return Workload(f"two_stage_k{k_bits}", 32, 8, batch, seq_len, ROT_WHT128, k_bits, 3, BF16, F16,
                    "lognormal_outlier", "normal", "normal", seed=seed)


def two_stage_projection(d: int, seed: int, head: int) -> np.ndarray:
    """The QJL projection S of one KV head: d x d, i.i.d. N(0, 1) entries, from
    its own seeded stream (depends only on (seed, head))."""
    rng = np.random.default_rng([seed, 0x514A, head])
    return rng.standard_normal((d, d)).astype(np.float32)


# T sweeps named by the workload descriptions.
LLAMA8B_T_SWEEP = (512, 2048, 8192)
SO4_T_SWEEP = (128, 256, 511, 512, 2048, 8192, 32768)
MIXED_T_SWEEP = (131072, 524288)


# ----------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Inputs:
    wl: Workload
    K: np.ndarray            # [B][T][Hkv][d] (fp32, or uint16 bf16 bits)
    V: np.ndarray            # [B][T][Hkv][d]
    q: np.ndarray            # [B][Hq][d]
    q_calib: Optional[np.ndarray]  # [T_cal][Hq][d] (same dtype) for mixed-rate keys
    signs: np.ndarray        # [Hkv][d] float32 +-1
    quats: np.ndarray        # [Hkv][d/4][2][4] float32 unit quaternions (q_L, q_R)
    seq_lens: np.ndarray     # [B] int32


def _channel_scales(rng, wl: Workload) -> np.ndarray:
    """Per-(kv-head, channel) multiplicative scale for K (and for V when it uses
    the same recipe)."""
    d = wl.head_dim
    if wl.k_recipe == "outlier4x20":
        s = np.ones((wl.n_kv_heads, d))
        ch = rng.choice(d, size=4, replace=False)
        s[:, ch] = 20.0
        return s
    if wl.k_recipe == "lognormal_outlier":
        s = rng.lognormal(mean=0.0, sigma=0.5, size=(wl.n_kv_heads, d))
        n_out = int(round(0.02 * d))
        for h in range(wl.n_kv_heads):
            ch = rng.choice(d, size=n_out, replace=False)
            s[h, ch] *= 15.0
        return s
    if wl.k_recipe == "rope_decay":
        return np.broadcast_to(rope_block_scale(d), (wl.n_kv_heads, d)).copy()
    raise ValueError(wl.k_recipe)


def rope_block_scale(d: int = HEAD_DIM) -> np.ndarray:
    """Scale 10^(-2i/64) on RoPE block i = coordinates (2i, 2i+1)."""
    i = np.arange(d) // 2
    return 10.0 ** (-2.0 * i / (d // 2))


def _normal(rng, shape, chunk=1 << 24) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    flat = out.reshape(-1)
    for s in range(0, flat.size, chunk):
        n = min(chunk, flat.size - s)
        flat[s:s + n] = rng.standard_normal(n, dtype=np.float32)
    return out


def _store(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == BF16:
        return f32_to_bf16_bits(x)
    if dtype == F16:
        return x.astype(np.float16)
    return x.astype(np.float32)


def make_inputs(wl: Workload, seq_len: Optional[int] = None, seq_lens=None) -> Inputs:
    """Draw every input of one workload.  `seq_len` overrides wl.seq_len (the
    number of cached tokens drawn); `seq_lens` optionally gives ragged per-batch
    lengths (each <= seq_len)."""
    T = wl.seq_len if seq_len is None else seq_len
    d, B, Hkv, Hq = wl.head_dim, wl.batch, wl.n_kv_heads, wl.n_q_heads
    rng = np.random.default_rng(wl.seed)
    scale = _channel_scales(rng, wl)                      # [Hkv][d]
    K = _normal(rng, (B, T, Hkv, d))
    K *= scale[None, None].astype(np.float32)
    V = _normal(rng, (B, T, Hkv, d))
    if wl.v_recipe == "outlier4x20":
        V *= scale[None, None].astype(np.float32)
    q_calib = None
    if wl.mixed_k:
        q_calib = _normal(rng, (wl.calib_tokens, Hq, d))
        q_calib *= rope_block_scale(d)[None, None].astype(np.float32)
    q = _normal(rng, (B, Hq, d))
    if wl.q_recipe == "rope_decay":
        q *= rope_block_scale(d)[None, None].astype(np.float32)
    signs = np.where(rng.random((Hkv, d)) < 0.5, -1.0, 1.0).astype(np.float32)
    g = rng.standard_normal((Hkv, d // 4, 2, 4))
    quats = (g / np.linalg.norm(g, axis=-1, keepdims=True)).astype(np.float32)
    if seq_lens is None:
        seq_lens = np.full(B, T, dtype=np.int32)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (B,) and seq_lens.max() <= T
    return Inputs(wl, _store(K, wl.in_dtype), _store(V, wl.in_dtype), _store(q, wl.in_dtype),
                  None if q_calib is None else _store(q_calib, wl.in_dtype),
                  signs, quats, seq_lens)


def haar_orthogonal(n: int, seed: int, head: int, bits: int) -> np.ndarray:
    """A Haar-distributed random orthogonal n x n matrix (QR of a Gaussian with
    the sign of R's diagonal moved into Q), drawn from its own seeded stream so
    that it depends only on (seed, head, bits)."""
    rng = np.random.default_rng([seed, 0x4841, head, bits])
    a = rng.standard_normal((n, n))
    qm, r = np.linalg.qr(a)
    qm = qm * np.sign(np.diag(r))[None, :]
    return qm.astype(np.float32)


def ragged_lengths(batch: int, t_max: int, seed: int) -> np.ndarray:
    """Seeded ragged sequence lengths in [1, t_max], including 1 and t_max."""
    rng = np.random.default_rng([seed, 0x5241])
    L = rng.integers(1, t_max + 1, size=batch).astype(np.int32)
    L[0] = t_max
    if batch > 1:
        L[1] = 1
    return L
