"""fp64 CPU oracle for the rotation-quantised KV cache and compressed-domain
decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library (``rotated_bit_kv_gb300``), and the library never imports it.

The oracle is deliberately plain and slow: dense matrices instead of butterflies,
closed-form Beta-density integrals instead of tables, one function per step of
the method, in the order the pages give them.  Sources, by page title:

* [TQ-MNN]  "TurboQuant: ... MNN runs it on the phone" (zhaode.wang):
  §2.1 the three-step encoder (norm, rotate, per-coordinate codebook search);
  §2.2 the coordinate density after a random rotation, f(t) ~ (1-t^2)^((d-3)/2);
  §2.3 the Lloyd-Max codebook (centroid / midpoint conditions) and the
       MSE <= 2.7/4^b bound;
  §2.4 the two-stage key code for 1-2 bits: a (b-1)-bit MSE code plus a 1-bit
       QJL code (signs of a random projection) of its residual, for an
       unbiased inner product;
  §3.1 Hadamard with a +-1 sign flip in place of a random orthogonal matrix,
       32-wide blocks with their own norm;
  §3.3 8 three-bit indices in 3 bytes, two four-bit indices per byte,
       rotated-domain K dot and V accumulation, in-place quantisation on write;
  §3.4 codebook search as a count of boundary comparisons (strict greater-than).
* [RotaryQuant] "RotaryQuant: Fitting 120B MoE Models on Consumer Hardware via
  Fused Compressed-Space Attention" (papernotes.org):
  Key design 2: R = R_SO(4) o H_d with v -> q_L v conj(q_R) per 4-dim block;
  Key design 3: <Rq, Rk> = q^T k, o~ = sum_j a_j v~_j = R o, one inverse rotation.
* [Block-GTQ] "RoPE-Aware Bit Allocation for KV-Cache Quantization" (aitrends.kr):
  block energy s_i, objective J(b) = sum_i s_i 4^(-b_i), greedy allocation by
  Delta_i = (3/4) s_i 4^(-b_i), same-width grouping, key-axis split with
  log-sum-exp merge.
* [ZipFusion] "ZipFusion: Fusing Lossless KV Decompression with Attention for
  Efficient LLM Decoding" (paper-daily.com): the lossless bf16 block codec
  (compression format; register restore) and attention on the restored values.

Readings where the pages are silent or ambiguous:
* density exponent (d-3)/2 (the §2.2 formula; the intuition paragraph's
  (d-2)/2 omits the Jacobian of the slice);
* the codebook dimension d is the width of the normalised block (128, 32, or a
  mixed-rate group's width);
* y = H . D . x (sign flip first); SO(4) variant y = S . H . x with no sign flip;
* search ties go to the lower cell (strict >, as the NEON compare-count does);
  the decision is taken in fp32: fp32(y) against fp32 boundaries;
* 3-bit packing is LSB first: index i of a vector occupies bits [3i, 3i+3) of
  the little-endian byte stream, so each 3-byte group holds 8 whole indices;
* the stored norm is ||x|| as is (no re-normalisation by ||Q(y)||), rounded to
  the norm dtype; a zero vector stores norm 0 and index 2^(b-1)-1 everywhere;
* mixed-rate keys: RoPE block i is coordinates (2i, 2i+1); each same-width group
  is encoded by one TQ-MSE encoder with its own random orthogonal matrix, its
  own norm and the codebook for its own width; groups are laid out in ascending
  bit width, one index per nibble, or (tight packing) each index at its
  group's width, concatenated LSB first, the record rounded up to whole
  16-byte units;
* attention scale 1/sqrt(head_dim); greedy ties go to the lowest block index;
* two-stage keys: the residual is taken in the rotated, normalised domain of the
  MSE stage (r = y - C[idx]); the projection S (d x d, i.i.d. N(0, 1)) is an
  input; sign(0) counts as +1; the stored norms are n and n * ||r||; the
  estimator is the sign projection's unbiased one, ||r|| sqrt(pi/2)/d <S q~, sign>.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Sequence, Tuple

import numpy as np
from scipy.special import betainc, beta as beta_fn

# ============================================================================
# 1. Coordinate density and the Lloyd-Max codebook  [TQ-MNN §2.2, §2.3]
# ============================================================================


def density_exponent(d: int) -> float:
    """a in f(t) = (1 - t^2)^a / Z on [-1, 1] for one coordinate of a uniformly
    random point on the unit sphere in R^d  [TQ-MNN §2.2]."""
    return (d - 3) / 2.0


def _Z(d: int) -> float:
    a = density_exponent(d)
    return beta_fn(0.5, a + 1.0)


def coord_cdf(t, d: int):
    """P(T <= t).  T^2 ~ Beta(1/2, a+1), so P(|T| <= x) = I_{x^2}(1/2, a+1)."""
    t = np.asarray(t, dtype=np.float64)
    a = density_exponent(d)
    return 0.5 + 0.5 * np.sign(t) * betainc(0.5, a + 1.0, np.minimum(t * t, 1.0))


def coord_tail(t, d: int):
    """P(T > t) for t >= 0, computed without cancellation: 1/2 I_{1-t^2}(a+1, 1/2)."""
    t = np.asarray(t, dtype=np.float64)
    a = density_exponent(d)
    return 0.5 * betainc(a + 1.0, 0.5, np.maximum(1.0 - t * t, 0.0))


def cell_probability(lo, hi, d: int):
    """P(lo < T <= hi), using the tail form on the positive side."""
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    pos = lo >= 0
    neg = hi <= 0
    out = coord_cdf(hi, d) - coord_cdf(lo, d)
    out = np.where(pos, coord_tail(np.abs(lo), d) - coord_tail(np.abs(hi), d), out)
    out = np.where(neg, coord_tail(np.abs(hi), d) - coord_tail(np.abs(lo), d), out)
    return out


def first_moment_antiderivative(t, d: int):
    """F1(t) with F1' = t f(t):  F1(t) = -(1 - t^2)^(a+1) / (2 (a+1) Z)."""
    t = np.asarray(t, dtype=np.float64)
    a = density_exponent(d)
    return -np.power(np.maximum(1.0 - t * t, 0.0), a + 1.0) / (2.0 * (a + 1.0) * _Z(d))


def cell_first_moment(lo, hi, d: int):
    """integral over (lo, hi] of t f(t) dt."""
    return first_moment_antiderivative(hi, d) - first_moment_antiderivative(lo, d)


def cell_second_moment(lo, hi, d: int):
    """integral over (lo, hi] of t^2 f(t) dt.  With u = t^2, the integral over
    [0, x] is 1/2 B(3/2, a+1) I_{x^2}(3/2, a+1) / Z; odd extension by sign."""
    a = density_exponent(d)
    Z = _Z(d)

    def G(t):
        t = np.asarray(t, dtype=np.float64)
        return np.sign(t) * 0.5 * beta_fn(1.5, a + 1.0) * betainc(1.5, a + 1.0, np.minimum(t * t, 1.0)) / Z

    return G(hi) - G(lo)


@dataclass
class Codebook:
    d: int
    bits: int
    centroids: np.ndarray    # ascending, 2^bits entries (fp64)
    boundaries: np.ndarray   # 2^bits - 1 midpoints (fp64)
    iterations: int


def lloyd_max_codebook(d: int, bits: int, tol: float = 1e-15, max_iter: int = 2_000_000) -> Codebook:
    """1-D continuous k-means on f(t) with 2^bits cells  [TQ-MNN §2.3]:
    boundaries are midpoints of neighbouring centroids; each centroid is the
    conditional mean of its cell; iterate until the centroids stop moving."""
    if d < 2:
        raise ValueError("codebook dimension must be >= 2")
    K = 1 << bits
    # initial centroids: the density's own quantiles at (k + 1/2) / K
    from scipy.special import betaincinv
    a = density_exponent(d)
    p = (np.arange(K) + 0.5) / K
    mag = np.sqrt(betaincinv(0.5, a + 1.0, np.abs(2.0 * p - 1.0)))
    c = np.sign(p - 0.5) * mag
    for it in range(1, max_iter + 1):
        b = 0.5 * (c[:-1] + c[1:])
        lo = np.concatenate(([-1.0], b))
        hi = np.concatenate((b, [1.0]))
        c_new = cell_first_moment(lo, hi, d) / cell_probability(lo, hi, d)
        if np.max(np.abs(c_new - c)) < tol:
            c = c_new
            break
        c = c_new
    else:
        raise RuntimeError(f"Lloyd-Max did not converge for d={d}, bits={bits}")
    return Codebook(d, bits, c, 0.5 * (c[:-1] + c[1:]), it)


def codebook_mse(cb: Codebook) -> float:
    """E[(T - Q(T))^2] per coordinate (closed form from cell moments)."""
    lo = np.concatenate(([-1.0], cb.boundaries))
    hi = np.concatenate((cb.boundaries, [1.0]))
    P = cell_probability(lo, hi, cb.d)
    M1 = cell_first_moment(lo, hi, cb.d)
    M2 = cell_second_moment(lo, hi, cb.d)
    return float(np.sum(M2 - 2.0 * cb.centroids * M1 + cb.centroids ** 2 * P))


_CB_CACHE = {}


def codebook(d: int, bits: int) -> Codebook:
    key = (d, bits)
    if key not in _CB_CACHE:
        _CB_CACHE[key] = lloyd_max_codebook(d, bits)
    return _CB_CACHE[key]


# ============================================================================
# 2. Rotations  [TQ-MNN §3.1; RotaryQuant Key design 2; Block-GTQ grouping]
# ============================================================================


def hadamard(n: int) -> np.ndarray:
    """Normalised Walsh-Hadamard matrix in natural (Sylvester) order, built by
    the doubling recursion H_2n = [[H, H], [H, -H]] / sqrt(2)."""
    if n < 1 or n & (n - 1):
        raise ValueError("n must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]]) / math.sqrt(2.0)
    return H


def quat_mul(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Hamilton product of quaternions (w, x, y, z)."""
    pw, px, py, pz = p
    qw, qx, qy, qz = q
    return np.array([
        pw * qw - px * qx - py * qy - pz * qz,
        pw * qx + px * qw + py * qz - pz * qy,
        pw * qy - px * qz + py * qw + pz * qx,
        pw * qz + px * qy - py * qx + pz * qw,
    ])


def quat_conj(q: np.ndarray) -> np.ndarray:
    return np.array([q[0], -q[1], -q[2], -q[3]])


def so4_block_matrix(qL: np.ndarray, qR: np.ndarray) -> np.ndarray:
    """4x4 matrix of v -> q_L v conj(q_R), v = (w, x, y, z) read as w + xi + yj + zk
    [RotaryQuant, Key design 2].  Built column by column from the Hamilton
    product of the basis quaternions."""
    qRc = quat_conj(np.asarray(qR, dtype=np.float64))
    qL = np.asarray(qL, dtype=np.float64)
    M = np.zeros((4, 4))
    for j in range(4):
        e = np.zeros(4)
        e[j] = 1.0
        M[:, j] = quat_mul(quat_mul(qL, e), qRc)
    return M


def block_diag(blocks: Sequence[np.ndarray]) -> np.ndarray:
    n = sum(b.shape[0] for b in blocks)
    out = np.zeros((n, n))
    o = 0
    for b in blocks:
        k = b.shape[0]
        out[o:o + k, o:o + k] = b
        o += k
    return out


@dataclass
class Segment:
    """A contiguous run of rotated coordinates that shares one norm and one
    codebook: positions [start, start+length) of the code record."""
    start: int
    length: int
    cb_dim: int
    bits: int
    norm_slot: int


@dataclass
class HeadSpec:
    """Everything the encoder needs for one KV head: the dense rotation R
    (rotated = R @ x, in code-record order), its segments, and the coordinate
    sets whose norms each segment stores (norm over x restricted to them)."""
    R: np.ndarray
    segments: List[Segment]
    seg_coords: List[np.ndarray]
    n_norm_slots: int
    nibble_codes: bool        # codes stored one per nibble (4-bit or mixed)
    tight: bool = False       # mixed-rate keys packed at their own widths (pack_tight)


def spec_wht128(signs: np.ndarray, bits: int) -> HeadSpec:
    """y = H_128 D x, one norm  [TQ-MNN §3.1]."""
    d = signs.shape[0]
    R = hadamard(d) @ np.diag(signs.astype(np.float64))
    return HeadSpec(R, [Segment(0, d, d, bits, 0)], [np.arange(d)], 1, bits == 4)


def spec_wht32(signs: np.ndarray, bits: int) -> HeadSpec:
    """Four independent 32-point sign-flipped WHTs, one norm per block
    [TQ-MNN §3.1 block_size = 32]; block k uses signs[32k:32k+32]."""
    d = signs.shape[0]
    H = hadamard(32)
    blocks = [H @ np.diag(signs[32 * k:32 * k + 32].astype(np.float64)) for k in range(d // 32)]
    segs = [Segment(32 * k, 32, 32, bits, k) for k in range(d // 32)]
    coords = [np.arange(32 * k, 32 * k + 32) for k in range(d // 32)]
    return HeadSpec(block_diag(blocks), segs, coords, d // 32, bits == 4)


def spec_so4_wht128(quats: np.ndarray, bits: int) -> HeadSpec:
    """R = R_SO(4) o H_d  [RotaryQuant, Key design 2]: y = S H x, S block
    diagonal with one q_L v conj(q_R) map per 4-dim block, no sign flip."""
    d = quats.shape[0] * 4
    S = block_diag([so4_block_matrix(quats[i, 0], quats[i, 1]) for i in range(d // 4)])
    return HeadSpec(S @ hadamard(d), [Segment(0, d, d, bits, 0)], [np.arange(d)], 1, bits == 4)


def group_layout(block_bits: Sequence[int], b_min: int = 1, b_max: int = 4):
    """Same-width grouping of RoPE blocks  [Block-GTQ, physical encoding]:
    for each width b (ascending) with at least one block, the coordinates
    (2i, 2i+1) of its blocks in ascending i.  Returns [(b, coords)]."""
    block_bits = np.asarray(block_bits)
    out = []
    for b in range(b_min, b_max + 1):
        blocks = np.nonzero(block_bits == b)[0]
        if blocks.size:
            coords = np.stack([2 * blocks, 2 * blocks + 1], axis=1).reshape(-1)
            out.append((b, coords))
    return out


def spec_group_dense(block_bits: Sequence[int], mats: dict, tight: bool = False) -> HeadSpec:
    """Mixed-rate keys: each same-width group is one TQ-MSE encoder with a
    random orthogonal matrix Pi_b of its own width, its own norm and the
    codebook for (n_b, b)  [Block-GTQ; TQ-MNN §2.1].  `mats[b]` is Pi_b.
    tight: the record packs each code at its group's width (pack_tight) instead
    of one per nibble."""
    layout = group_layout(block_bits)
    d = 2 * len(block_bits)
    R = np.zeros((d, d))
    segs, coords = [], []
    o = 0
    for b, cs in layout:
        n = cs.size
        P = np.asarray(mats[b], dtype=np.float64)
        assert P.shape == (n, n)
        R[o:o + n, cs] = P
        segs.append(Segment(o, n, n, b, b - 1))
        coords.append(cs)
        o += n
    return HeadSpec(R, segs, coords, 4, not tight, tight)


# ============================================================================
# 3. Quantise and pack  [TQ-MNN §2.1, §3.3, §3.4]
# ============================================================================


def round_norm(n: np.ndarray, norm_dtype: str) -> np.ndarray:
    if norm_dtype == "f16":
        return n.astype(np.float16)
    return n.astype(np.float32)


def codebook_search(y: np.ndarray, cb: Codebook) -> np.ndarray:
    """idx = #{k : y > beta_k}: the count of boundaries strictly below y
    [TQ-MNN §3.4], so a coordinate on a boundary takes the lower cell.  The
    comparison is made in fp32 (fp32(y) against fp32 boundaries)."""
    b32 = cb.boundaries.astype(np.float32)
    y32 = np.asarray(y).astype(np.float32)
    return np.sum(y32[..., None] > b32, axis=-1).astype(np.int64)


def quantize(x: np.ndarray, spec: HeadSpec, norm_dtype: str):
    """Encode vectors x [N][d] (exact fp64 values of the inputs).

    Per segment: n = ||x_seg||; y = (R x)_seg / n; idx = #{k : y > beta_k}
    with the decision in fp32.  Returns (idx [N][d] int, stored norms
    [N][slots], y [N][d] fp64)."""
    x = np.asarray(x, dtype=np.float64)
    N, d = x.shape
    rot = x @ spec.R.T
    idx = np.zeros((N, d), dtype=np.int64)
    y = np.zeros((N, d))
    norms = np.zeros((N, spec.n_norm_slots))
    for seg, cs in zip(spec.segments, spec.seg_coords):
        n = np.sqrt(np.sum(x[:, cs] ** 2, axis=1))
        sl = slice(seg.start, seg.start + seg.length)
        with np.errstate(invalid="ignore", divide="ignore"):
            ys = np.where(n[:, None] > 0, rot[:, sl] / n[:, None], 0.0)
        y[:, sl] = ys
        idx[:, sl] = codebook_search(ys, codebook(seg.cb_dim, seg.bits))
        norms[:, seg.norm_slot] = n
    return idx, round_norm(norms, norm_dtype), y


def pack_3bit(idx: np.ndarray) -> np.ndarray:
    """8 three-bit indices per 3 bytes: for group g, w = sum_i idx[8g+i] << 3i,
    stored little-endian as w & 255, (w >> 8) & 255, (w >> 16) & 255."""
    idx = np.asarray(idx, dtype=np.int64)
    N, d = idx.shape
    assert d % 8 == 0 and idx.min() >= 0 and idx.max() < 8
    g = idx.reshape(N, d // 8, 8)
    w = np.zeros((N, d // 8), dtype=np.int64)
    for i in range(8):
        w |= g[:, :, i] << (3 * i)
    out = np.stack([w & 255, (w >> 8) & 255, (w >> 16) & 255], axis=2)
    return out.reshape(N, 3 * d // 8).astype(np.uint8)


def unpack_3bit(b: np.ndarray, d: int) -> np.ndarray:
    b = np.asarray(b, dtype=np.int64).reshape(b.shape[0], d // 8, 3)
    w = b[:, :, 0] | (b[:, :, 1] << 8) | (b[:, :, 2] << 16)
    return np.stack([(w >> (3 * i)) & 7 for i in range(8)], axis=2).reshape(b.shape[0], d)


def pack_4bit(idx: np.ndarray) -> np.ndarray:
    """Two indices per byte: byte j = idx[2j] | idx[2j+1] << 4."""
    idx = np.asarray(idx, dtype=np.int64)
    assert idx.min() >= 0 and idx.max() < 16
    return (idx[:, 0::2] | (idx[:, 1::2] << 4)).astype(np.uint8)


def unpack_4bit(b: np.ndarray, d: int) -> np.ndarray:
    b = np.asarray(b, dtype=np.int64)
    out = np.zeros((b.shape[0], d), dtype=np.int64)
    out[:, 0::2] = b & 15
    out[:, 1::2] = b >> 4
    return out


def code_widths(spec: HeadSpec) -> np.ndarray:
    """[d] bits of the code at each record position (its segment's width)."""
    w = np.zeros(sum(sg.length for sg in spec.segments), dtype=np.int64)
    for sg in spec.segments:
        w[sg.start:sg.start + sg.length] = sg.bits
    return w


def pack_tight(idx: np.ndarray, spec: HeadSpec) -> np.ndarray:
    """Mixed-rate keys at their own widths  [Block-GTQ, packed cache: the groups'
    codes concatenated]: the code at record position p takes w_p bits at bit
    offset sum_{p' < p} w_p' of the little-endian byte stream, LSB first (the
    positions are the groups in ascending width, as for the nibble record).
    The record is the total width rounded up to whole 16-byte units."""
    idx = np.asarray(idx, dtype=np.int64)
    N, d = idx.shape
    w = code_widths(spec)
    assert w.size == d and np.all(idx < (1 << w)[None, :]) and idx.min() >= 0
    total = int(w.sum())
    nbits = -(-total // 128) * 128
    bits = np.zeros((N, nbits), dtype=np.uint8)
    off = 0
    for p in range(d):
        for k in range(int(w[p])):
            bits[:, off + k] = (idx[:, p] >> k) & 1
        off += int(w[p])
    return np.packbits(bits, axis=1, bitorder="little")


def unpack_tight(codes: np.ndarray, spec: HeadSpec, d: int) -> np.ndarray:
    bits = np.unpackbits(np.asarray(codes, dtype=np.uint8), axis=1, bitorder="little").astype(np.int64)
    w = code_widths(spec)
    out = np.zeros((bits.shape[0], d), dtype=np.int64)
    off = 0
    for p in range(d):
        for k in range(int(w[p])):
            out[:, p] |= bits[:, off + k] << k
        off += int(w[p])
    return out


def pack(idx: np.ndarray, spec: HeadSpec) -> np.ndarray:
    if spec.tight:
        return pack_tight(idx, spec)
    return pack_4bit(idx) if spec.nibble_codes else pack_3bit(idx)


def unpack(codes: np.ndarray, spec: HeadSpec, d: int) -> np.ndarray:
    if spec.tight:
        return unpack_tight(codes, spec, d)
    return unpack_4bit(codes, d) if spec.nibble_codes else unpack_3bit(codes, d)


def dequantize_rotated(idx: np.ndarray, norms: np.ndarray, spec: HeadSpec) -> np.ndarray:
    """v~ = n_seg * C_seg[idx] in the rotated domain (no inverse rotation)."""
    N, d = idx.shape
    out = np.zeros((N, d))
    nrm = np.asarray(norms, dtype=np.float64)
    for seg in spec.segments:
        sl = slice(seg.start, seg.start + seg.length)
        C = codebook(seg.cb_dim, seg.bits).centroids
        out[:, sl] = nrm[:, seg.norm_slot][:, None] * C[idx[:, sl]]
    return out


def dequantize(idx: np.ndarray, norms: np.ndarray, spec: HeadSpec) -> np.ndarray:
    """Reverse of the encoder [TQ-MNN §2.1]: codebook lookup -> inverse
    rotation -> times the norm."""
    return dequantize_rotated(idx, norms, spec) @ spec.R


# ============================================================================
# 4. Block energy and greedy bit allocation  [Block-GTQ]
# ============================================================================


def block_energy(q_cal: np.ndarray, k_cal: np.ndarray) -> np.ndarray:
    """s_i = 1/2 (E_{t, g in G(h)} ||q^(i)||^2 + E_t ||k^(i)||^2), block i =
    coordinates (2i, 2i+1).  q_cal [T][G][d] holds the query heads that read
    this KV head; k_cal [T][d]."""
    q = np.asarray(q_cal, dtype=np.float64)
    k = np.asarray(k_cal, dtype=np.float64)
    d = k.shape[-1]
    qb = (q.reshape(q.shape[0], q.shape[1], d // 2, 2) ** 2).sum(-1)   # [T][G][L]
    kb = (k.reshape(k.shape[0], d // 2, 2) ** 2).sum(-1)                # [T][L]
    return 0.5 * (qb.mean(axis=(0, 1)) + kb.mean(axis=0))


def greedy_bit_alloc(s: Sequence[float], b_min: int, b_max: int, B_total: int) -> np.ndarray:
    """Minimise J(b) = sum_i s_i 4^(-b_i) s.t. b_min <= b_i <= b_max,
    sum_i b_i = B_total: start at b_min, then repeatedly add one bit to the
    block with the largest marginal gain Delta_i = (3/4) s_i 4^(-b_i) among
    blocks below b_max (ties -> lowest index)."""
    s = np.asarray(s, dtype=np.float64)
    L = s.size
    if B_total < L * b_min or B_total > L * b_max or b_min > b_max:
        raise ValueError("infeasible bit budget")
    b = np.full(L, b_min, dtype=np.int64)
    for _ in range(B_total - L * b_min):
        best, best_gain = -1, -np.inf
        for i in range(L):
            if b[i] < b_max:
                gain = 0.75 * s[i] * 4.0 ** (-b[i])
                if gain > best_gain:
                    best, best_gain = i, gain
        b[best] += 1
    return b


def allocation_objective(s, b) -> float:
    return float(np.sum(np.asarray(s, dtype=np.float64) * 4.0 ** (-np.asarray(b, dtype=np.float64))))


# ============================================================================
# 5. Decode attention on the packed cache  [RotaryQuant Key design 3;
#    TQ-MNN §3.3; Block-GTQ key-axis split]
# ============================================================================


def attend_rotated(q: np.ndarray, k_idx, k_norm, k_spec: HeadSpec, v_idx, v_norm, v_spec: HeadSpec,
                   seq_len: int) -> np.ndarray:
    """One (batch, KV head): q [G][d] (exact fp64 of the stored query).

    q~ = R_K q; s_j = <q~, k~_j> / sqrt(d) with k~_j = n_j C[idx_j] per segment;
    a = softmax over j < seq_len; o~ = sum_j a_j v~_j; o = R_V^T o~."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    L = int(seq_len)
    if L <= 0:
        return np.zeros_like(q)
    qt = q @ k_spec.R.T                                   # [G][d]
    Kt = dequantize_rotated(k_idx[:L], k_norm[:L], k_spec)
    Vt = dequantize_rotated(v_idx[:L], v_norm[:L], v_spec)
    s = qt @ Kt.T / math.sqrt(d)                          # [G][L]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    a = p / p.sum(axis=1, keepdims=True)
    ot = a @ Vt                                           # rotated-domain output
    return ot @ v_spec.R                                  # R^T applied: o = R^T o~


def attend_dequantized(q, k_idx, k_norm, k_spec, v_idx, v_norm, v_spec, seq_len) -> np.ndarray:
    """The same attention computed the conventional way: dequantise every key
    and value back to the original domain, then attend with the raw q."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    L = int(seq_len)
    if L <= 0:
        return np.zeros_like(q)
    K = dequantize(k_idx[:L], k_norm[:L], k_spec)
    V = dequantize(v_idx[:L], v_norm[:L], v_spec)
    s = q @ K.T / math.sqrt(d)
    a = np.exp(s - s.max(axis=1, keepdims=True))
    a /= a.sum(axis=1, keepdims=True)
    return a @ V


def attend_exact(q, K, V, seq_len) -> np.ndarray:
    """Unquantised fp64 attention (for the reported quantisation-error statistic)."""
    q = np.asarray(q, dtype=np.float64)
    L = int(seq_len)
    s = q @ np.asarray(K[:L], dtype=np.float64).T / math.sqrt(q.shape[-1])
    a = np.exp(s - s.max(axis=1, keepdims=True))
    a /= a.sum(axis=1, keepdims=True)
    return a @ np.asarray(V[:L], dtype=np.float64)


def split_partials(q, k_idx, k_norm, k_spec, v_idx, v_norm, v_spec, bounds: Sequence[Tuple[int, int]]):
    """Per key-axis section [lo, hi): (m, l, o~_unnormalised) with
    m = max_j s_j, l = sum_j exp(s_j - m), o~ = sum_j exp(s_j - m) v~_j.
    An empty section yields (-inf, 0, 0)."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    qt = q @ k_spec.R.T
    out = []
    for lo, hi in bounds:
        if hi <= lo:
            out.append((np.full(q.shape[0], -np.inf), np.zeros(q.shape[0]), np.zeros_like(q)))
            continue
        Kt = dequantize_rotated(k_idx[lo:hi], k_norm[lo:hi], k_spec)
        Vt = dequantize_rotated(v_idx[lo:hi], v_norm[lo:hi], v_spec)
        s = qt @ Kt.T / math.sqrt(d)
        m = s.max(axis=1)
        p = np.exp(s - m[:, None])
        out.append((m, p.sum(axis=1), p @ Vt))
    return out


def lse_merge(partials, v_spec: HeadSpec) -> np.ndarray:
    """Log-sum-exp merge of key-axis sections, then the single inverse rotation:
    M = max m_s; l = sum_s e^(m_s - M) l_s; o~ = sum_s e^(m_s - M) o~_s / l;
    o = R_V^T o~.  Sections with m = -inf contribute nothing."""
    ms = np.stack([p[0] for p in partials])            # [S][G]
    M = ms.max(axis=0)
    w = np.where(np.isfinite(ms), np.exp(ms - M[None]), 0.0)
    l = sum(w[i] * partials[i][1] for i in range(len(partials)))
    ot = sum(w[i][:, None] * partials[i][2] for i in range(len(partials)))
    return (ot / l[:, None]) @ v_spec.R


def part_state(q, K, V) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(m, l, o) of one part of the keys in the original domain: s_j = <q, k_j> / sqrt(d),
    m = max_j s_j, l = sum_j e^(s_j - m), o = sum_j e^(s_j - m) v_j (not normalised).
    An empty part yields (-inf, 0, 0)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.full(q.shape[0], -np.inf), np.zeros(q.shape[0]), np.zeros_like(q)
    s = q @ K.T / math.sqrt(q.shape[-1])
    m = s.max(axis=1)
    p = np.exp(s - m[:, None])
    return m, p.sum(axis=1), p @ V


def attend_prefix_packed(q, K_pre, V_pre, k_idx, k_norm, k_spec: HeadSpec, v_idx, v_norm, v_spec: HeadSpec,
                         seq_len: int) -> np.ndarray:
    """Attention of one (batch, KV head) over two parts of its keys: a block of
    unquantised tokens (K_pre, V_pre [n][d]: the exact values of the stored
    fp16 / bf16 / fp32 inputs) and the first seq_len tokens of the packed cache.
    The unquantised block is the prefill kept in fp16 [RotaryQuant, deferred
    prefill] or the recent-token buffer [Block-GTQ]; the set of keys is the
    union of the two parts whatever their order in the sequence.

    Each part is attended on its own: the unquantised part in the original
    domain; the packed part in the rotated domain (q~ = R_K q, n C[idx]) and
    brought back with its one inverse rotation, o_p = R_V^T o~_p (linear, so it
    applies to the unnormalised sum).  The parts are merged by log-sum-exp
    [Block-GTQ, key-axis split]: M = max_u m_u,
      o = sum_u e^(m_u - M) o_u / sum_u e^(m_u - M) l_u."""
    q = np.asarray(q, dtype=np.float64)
    parts = [part_state(q, K_pre, V_pre)]
    L = int(seq_len)
    if L > 0:
        m, l, ot = split_partials(q, k_idx, k_norm, k_spec, v_idx, v_norm, v_spec, [(0, L)])[0]
        parts.append((m, l, ot @ v_spec.R))
    ms = np.stack([p[0] for p in parts])
    M = ms.max(axis=0)
    if not np.all(np.isfinite(M)):
        return np.zeros_like(q)
    w = np.where(np.isfinite(ms), np.exp(ms - M[None]), 0.0)
    l = sum(w[i] * parts[i][1] for i in range(len(parts)))
    o = sum(w[i][:, None] * parts[i][2] for i in range(len(parts)))
    return o / l[:, None]


# ============================================================================
# 6. Whole-cache helpers (loops over (batch, KV head); no reordering)
# ============================================================================


def head_specs(wl, inputs, block_bits=None, mats=None):
    """(k_spec, v_spec) per KV head for a workload description."""
    from workloads import ROT_WHT128, ROT_WHT32, ROT_SO4_WHT128
    specs = []
    for h in range(wl.n_kv_heads):
        if wl.rot == ROT_WHT128:
            v = spec_wht128(inputs.signs[h], wl.v_bits)
            k = spec_wht128(inputs.signs[h], wl.k_bits)
        elif wl.rot == ROT_WHT32:
            v = spec_wht32(inputs.signs[h], wl.v_bits)
            k = spec_wht32(inputs.signs[h], wl.k_bits)
        elif wl.rot == ROT_SO4_WHT128:
            v = spec_so4_wht128(inputs.quats[h], wl.v_bits)
            k = spec_so4_wht128(inputs.quats[h], wl.k_bits)
        else:
            raise ValueError(wl.rot)
        if wl.mixed_k:
            k = spec_group_dense(block_bits[h], mats[h], tight=getattr(wl, "tight_k", False))
        specs.append((k, v))
    return specs


def norm_dtype_name(wl) -> str:
    from workloads import F16
    return "f16" if wl.norm_dtype == F16 else "f32"


# ============================================================================
# 8. ZipFusion lossless bf16 block codec  [ZipFusion, compression format and
#    register restore]
# ============================================================================
#
# A block is 512 bf16 values (their 16-bit patterns).  Its base b is the smallest
# exponent field rounded down to even; the block compresses iff every exponent
# lies in [b, b + 15].  A compressed value keeps its low byte (7 mantissa bits
# and the exponent's lowest bit) and a 4-bit code: the sign and d = (e - b) >> 1.
# Restore: high byte = 128 sign + b/2 + d.  Codes of a group of 8 consecutive
# values go two per byte: byte k (k = 0..3) holds value k's sign in bit 7 and d
# in bits 0-2, value k + 4's sign in bit 6 and d in bits 3-5.
ZF_BLOCK = 512


def zf_exponent(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.int64) >> 7) & 0xFF


def zf_base(bits: np.ndarray) -> int:
    """b: the smallest exponent field of the block, rounded down to even."""
    return int(zf_exponent(bits).min()) // 2 * 2


def zf_compressible(bits: np.ndarray) -> bool:
    e = zf_exponent(bits)
    return int(e.max()) <= zf_base(bits) + 15


def zf_encode_block(bits: np.ndarray):
    """(half_base, low[512] uint8, codes[256] uint8) of a compressible block."""
    bits = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    assert bits.size == ZF_BLOCK and zf_compressible(bits)
    b = zf_base(bits)
    e = (bits >> 7) & 0xFF
    sign = bits >> 15
    d = (e - b) >> 1
    low = (bits & 0xFF).astype(np.uint8)
    codes = np.zeros(ZF_BLOCK // 2, dtype=np.uint8)
    for g in range(ZF_BLOCK // 8):
        for k in range(4):
            i, j = 8 * g + k, 8 * g + k + 4
            codes[4 * g + k] = (sign[i] << 7) | d[i] | (sign[j] << 6) | (d[j] << 3)
    return b // 2, low, codes


def zf_decode_block(half_base: int, low: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """The 512 bf16 bit patterns of a compressed block."""
    out = np.zeros(ZF_BLOCK, dtype=np.uint16)
    for i in range(ZF_BLOCK):
        g, k = divmod(i, 8)
        byte = int(codes[4 * g + (k % 4)])
        if k < 4:
            sign, d = byte >> 7, byte & 7
        else:
            sign, d = (byte >> 6) & 1, (byte >> 3) & 7
        hi = 128 * sign + half_base + d
        out[i] = (hi << 8) | int(low[i])
    return out


def zf_high_bytes(code_byte: int, half_base: int):
    """High bytes of the two values whose codes share one code byte (the first
    value of the pair and the one four places later)."""
    hi1 = 128 * (code_byte >> 7) + half_base + (code_byte & 7)
    hi5 = 128 * ((code_byte >> 6) & 1) + half_base + ((code_byte >> 3) & 7)
    return hi1, hi5


def zf_block_groups(which: str):
    """The page's four blocks as lists of 64 groups of 8 values, in the order a
    block stores them: [4][64] of (token, first coordinate).  The pages keep each
    MMA thread's 8 values together and lay K and V out for their own products
    ([ZipFusion], register restore); here the groups a lane (r, c) reads at one
    step of the attention form one block, so that a block's mode is the same for
    the whole warp:
      K block q (q = 0..3): group 2L + u, L = 4r + c, is token r + 8u, coordinates
        32c + 8q .. +7 (the lane's keys of tokens r and r + 8);
      V block 2e + q (e, q = 0, 1): group 2L + u is token 8e + 2c + u, coordinates
        16r + 8q .. +7 (the lane's values of tokens 2c + 8e and 2c + 8e + 1)."""
    out = []
    for j in range(4):
        grp = []
        for L in range(32):
            r, c = L >> 2, L & 3
            for u in range(2):
                if which == "k":
                    grp.append((r + 8 * u, 32 * c + 8 * j))
                else:
                    e, q = j >> 1, j & 1
                    grp.append((8 * e + 2 * c + u, 16 * r + 8 * q))
        out.append(grp)
    return out


def zf_page_blocks(page: np.ndarray, which: str) -> np.ndarray:
    """The four 512-value blocks of one 16-token page of one (batch, KV head):
    page [16][128] bf16 bits -> [4][512] in block order (zf_block_groups)."""
    page = np.asarray(page, dtype=np.uint16)
    return np.stack([np.concatenate([page[t, d0:d0 + 8] for t, d0 in grp]) for grp in zf_block_groups(which)])


def zf_page_unblocks(blocks: np.ndarray, which: str) -> np.ndarray:
    """Inverse of zf_page_blocks."""
    page = np.zeros((16, 128), dtype=np.uint16)
    for j, grp in enumerate(zf_block_groups(which)):
        for g, (t, d0) in enumerate(grp):
            page[t, d0:d0 + 8] = blocks[j][8 * g:8 * g + 8]
    return page


def zf_page_roundtrip(page: np.ndarray, which: str) -> np.ndarray:
    """Encode and restore every block of a page (raw blocks as they are)."""
    out = []
    for blk in zf_page_blocks(page, which):
        if zf_compressible(blk):
            out.append(zf_decode_block(*zf_encode_block(blk)))
        else:
            out.append(blk.copy())
    return zf_page_unblocks(np.stack(out), which)


# ============================================================================
# 9. Two-stage key code: a (b-1)-bit MSE code and a 1-bit QJL code of its
#    residual  [TQ-MNN §2.4]
# ============================================================================
#
# An MSE-optimal code shrinks inner products.  For keys at 1-2 bits the page
# spends b - 1 bits on the MSE code and the last bit on a quantised
# Johnson-Lindenstrauss code of what the MSE code leaves over: the signs of a
# random Gaussian projection, which give an unbiased estimate of <q, k>.
# The estimator written out here is the standard one for a sign projection:
# for s ~ N(0, I_d), E[<s, a> sign(<s, r>)] = sqrt(2/pi) <a, r> / ||r||, so with
# the d rows of S and rho = ||r||,
#   <a, r>  ~=  rho * sqrt(pi/2) / d * <S a, sign(S r)>    (unbiased).
# Everything stays in the rotated, normalised domain of the MSE stage: y = R x /
# ||x||, r = y - C[idx], and q~ = R q as in the one-stage path.


@dataclass
class QjlSpec:
    """One KV head's two-stage key code: rotation R (as the one-stage spec),
    MSE bits b - 1 (0: no MSE code, the whole normalised vector goes to the QJL
    stage) and the d x d projection S with i.i.d. N(0, 1) entries."""
    R: np.ndarray
    mse_bits: int
    S: np.ndarray


def qjl_scale(d: int) -> float:
    """sqrt(pi/2) / d, the factor that makes the sign estimate unbiased."""
    return math.sqrt(math.pi / 2.0) / d


def qjl_quantize(x: np.ndarray, qs: QjlSpec, norm_dtype: str):
    """Encode keys x [N][d]: n = ||x||; y = R x / n; idx = #{k : y > beta_k} on
    the (b-1)-bit codebook (all 0 and no reconstruction when b = 1); r = y -
    C[idx]; rho = ||r||; z = S r; sign bit = 1 where z >= 0 (the reading of
    sign(0) is +1).  Stored norms: slot 0 n, slot 1 n * rho (rounded to the norm
    dtype).  Returns (idx [N][d], sign bits [N][d] 0/1, norms [N][2], y, z)."""
    x = np.asarray(x, dtype=np.float64)
    N, d = x.shape
    n = np.sqrt(np.sum(x * x, axis=1))
    with np.errstate(invalid="ignore", divide="ignore"):
        y = np.where(n[:, None] > 0, (x @ qs.R.T) / n[:, None], 0.0)
    if qs.mse_bits > 0:
        cb = codebook(d, qs.mse_bits)
        idx = codebook_search(y, cb)
        yhat = cb.centroids[idx]
    else:
        idx = np.zeros((N, d), dtype=np.int64)
        yhat = np.zeros((N, d))
    r = y - yhat
    rho = np.sqrt(np.sum(r * r, axis=1))
    z = r @ np.asarray(qs.S, dtype=np.float64).T
    sbits = (z >= 0).astype(np.int64)
    norms = np.stack([n, n * rho], axis=1)
    return idx, sbits, round_norm(norms, norm_dtype), y, z


def qjl_record_bytes(mse_bits: int, d: int = 128) -> int:
    """(b - 1) * d / 8 bytes of MSE codes, then d / 8 bytes of signs."""
    return (mse_bits + 1) * d // 8


def pack_bits(v: np.ndarray, width: int) -> np.ndarray:
    """Fields of `width` bits, LSB first: field i at bits [width i, width (i+1))
    of the little-endian byte stream."""
    v = np.asarray(v, dtype=np.int64)
    N, d = v.shape
    bits = np.zeros((N, d * width), dtype=np.uint8)
    for k in range(width):
        bits[:, k::width] = (v >> k) & 1
    return np.packbits(bits, axis=1, bitorder="little")


def unpack_bits(b: np.ndarray, width: int, d: int) -> np.ndarray:
    bits = np.unpackbits(np.asarray(b, dtype=np.uint8), axis=1, bitorder="little").astype(np.int64)
    v = np.zeros((bits.shape[0], d), dtype=np.int64)
    for k in range(width):
        v |= bits[:, k:d * width:width] << k
    return v


def qjl_pack(idx: np.ndarray, sbits: np.ndarray, mse_bits: int) -> np.ndarray:
    """One record per key: the MSE codes (mse_bits each, LSB first), then the d
    sign bits (bit j of the sign bytes = sign of z_j)."""
    parts = [pack_bits(idx, mse_bits)] if mse_bits > 0 else []
    parts.append(pack_bits(sbits, 1))
    return np.concatenate(parts, axis=1)


def qjl_unpack(codes: np.ndarray, mse_bits: int, d: int = 128):
    codes = np.asarray(codes, dtype=np.uint8)
    nb = mse_bits * d // 8
    idx = unpack_bits(codes[:, :nb], mse_bits, d) if mse_bits > 0 else np.zeros((codes.shape[0], d), np.int64)
    return idx, unpack_bits(codes[:, nb:nb + d // 8], 1, d)


def qjl_scores(q: np.ndarray, idx, sbits, norms, qs: QjlSpec) -> np.ndarray:
    """Estimated <q_g, k_j> [G][N]:
      n_j <q~, C[idx_j]> + (n_j rho_j) sqrt(pi/2)/d <S q~, 2 sbits_j - 1>,
    q~ = R q; the first term is absent when b = 1."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    nrm = np.asarray(norms, dtype=np.float64)
    qt = q @ qs.R.T
    if qs.mse_bits > 0:
        C = codebook(d, qs.mse_bits).centroids
        mse = (qt @ C[idx].T) * nrm[:, 0][None, :]
    else:
        mse = np.zeros((q.shape[0], idx.shape[0]))
    u = qt @ np.asarray(qs.S, dtype=np.float64).T               # S q~
    sg = 2.0 * np.asarray(sbits, dtype=np.float64) - 1.0
    return mse + qjl_scale(d) * (u @ sg.T) * nrm[:, 1][None, :]


def attend_qjl(q, k_idx, k_sbits, k_norm, qs: QjlSpec, v_idx, v_norm, v_spec: HeadSpec, seq_len: int):
    """Decode attention of one (batch, KV head) with two-stage keys: scores are
    the estimates of qjl_scores over sqrt(d); values as in attend_rotated
    (rotated domain, one inverse rotation)."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    L = int(seq_len)
    if L <= 0:
        return np.zeros_like(q)
    s = qjl_scores(q, k_idx[:L], k_sbits[:L], k_norm[:L], qs) / math.sqrt(d)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    a = p / p.sum(axis=1, keepdims=True)
    Vt = dequantize_rotated(v_idx[:L], v_norm[:L], v_spec)
    return (a @ Vt) @ v_spec.R
