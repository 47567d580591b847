"""Helpers shared by the GPU parity tests, smoke() and the benchmark's CPU leg:
build the library-side parameters and the oracle-side specs for one workload,
encode with the oracle per (batch, KV head), move records between numpy and
the device cache, and compare under the stated tolerances.

Everything on the "expected" side comes from ``oracle/``; everything on the
"actual" side comes from the CUDA library.  The two meet only here, in the
comparison."""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

import workloads as W
from oracle import tq_oracle as O

NEAR_WINDOW = 1e-5          # |y - boundary| below which a code may differ
MAX_MISMATCH_FRAC = 1e-4    # gate on the fraction of differing codes
ATT_TOL = 2e-3              # max-abs error <= ATT_TOL * max|o|


@dataclass
class Setup:
    wl: W.Workload
    inp: W.Inputs
    block_bits: np.ndarray      # [Hkv][64] (mixed-rate keys) or None
    mats: list                  # per head {b: Pi_b} (mixed) or None
    specs: list                 # per head (k_spec, v_spec)
    blob: np.ndarray            # library parameter blob
    desc: object


def calib_keys(wl, inp):
    """fp32 calibration prefix of the keys, [T_cal][Hkv][d], from batch 0."""
    return W.as_float64(inp.K[0, :wl.calib_tokens], wl.in_dtype).astype(np.float32)


def make_setup(tq, wl: W.Workload, inp: W.Inputs, t_capacity: int) -> Setup:
    """Library descriptor + blob and oracle specs for the same inputs.  For
    mixed-rate keys both sides compute block energies and the greedy
    allocation independently; they must agree."""
    block_bits = mats = None
    G = wl.group
    if wl.mixed_k:
        kc = calib_keys(wl, inp)
        qc = W.as_float64(inp.q_calib, wl.in_dtype).astype(np.float32)
        bbs = []
        for h in range(wl.n_kv_heads):
            qh = qc[:, h * G:(h + 1) * G]
            s_lib = tq.tq_block_energy(qh, kc[:, h])
            s_or = O.block_energy(qh, kc[:, h])
            np.testing.assert_allclose(s_lib, s_or, rtol=1e-12)
            B_total = wl.avg_bits * (wl.head_dim // 2)
            b_lib = tq.tq_block_bit_alloc(s_lib, wl.b_min, wl.b_max, B_total)
            b_or = O.greedy_bit_alloc(s_or, wl.b_min, wl.b_max, B_total)
            np.testing.assert_array_equal(b_lib, b_or)
            bbs.append(b_or)
        block_bits = np.stack(bbs).astype(np.int32)
        mats = []
        flat = []
        for h in range(wl.n_kv_heads):
            m = {}
            for b, cs in O.group_layout(block_bits[h], wl.b_min, wl.b_max):
                m[b] = W.haar_orthogonal(cs.size, wl.seed, h, b)
                flat.append(m[b].ravel())
            mats.append(m)
        flat = np.concatenate(flat)
    # mixed-rate keys: nibble records (k_mixed 1), or tight records (k_mixed 2, k_bits
    # the average width)
    k_mixed = (2 if wl.tight_k else 1) if wl.mixed_k else 0
    k_bits = (wl.avg_bits if wl.tight_k else 0) if wl.mixed_k else wl.k_bits
    desc = tq.tq_cache_desc_init(wl.head_dim, wl.n_q_heads, wl.n_kv_heads, wl.batch, t_capacity, wl.rot,
                                 k_bits, wl.v_bits, wl.norm_dtype, k_mixed)
    blob = tq.tq_params_build(desc, signs=inp.signs, quats=inp.quats,
                              k_block_bits=block_bits, k_group_mats=flat if wl.mixed_k else None)
    specs = O.head_specs(wl, inp, block_bits, mats)
    return Setup(wl, inp, block_bits, mats, specs, blob, desc)


@dataclass
class OracleEnc:
    codes: np.ndarray   # [T][bytes] uint8
    idx: np.ndarray     # [T][d]
    norms: np.ndarray   # [T][slots] stored dtype
    y: np.ndarray       # [T][d] fp64 normalised rotated coordinate


def oracle_encode(st: Setup, which: str, b: int, h: int, t0: int = 0, t1=None) -> OracleEnc:
    src = st.inp.K if which == "k" else st.inp.V
    x = W.as_float64(src[b, t0:t1, h], st.wl.in_dtype)
    spec = st.specs[h][0 if which == "k" else 1]
    idx, nrm, y = O.quantize(x, spec, O.norm_dtype_name(st.wl))
    return OracleEnc(O.pack(idx, spec), idx, nrm, y)


# ---------------------------------------------------------------- cache layouts
# The two layouts of include/tq.h restated in numpy from that header's text (no
# code of the library is used): TQ_LAYOUT_NATURAL keeps one record per position;
# TQ_LAYOUT_TILE16 permutes the bits of every 16-token tile as documented there.

_BIT_MAPS = {}


def tile_bit_map(which: str, bits: int) -> np.ndarray:
    """[16 tokens][64 fields][field bits] -> bit index within a code tile."""
    key = (which, bits)
    if key in _BIT_MAPS:
        return _BIT_MAPS[key]
    W = 3 if bits == 3 else 4
    fb = 6 if bits == 3 else 8
    X, Y = np.arange(6), np.array([0, 1, 4, 5, 6, 7])

    def word_byte(L, i):
        return 16 * L + 4 * i if i < 4 else 512 + 8 * (W - 2) * L + 4 * (i - 4)

    M = np.full((16, 64, fb), -1, dtype=np.int64)
    for t in range(16):
        if which == "k":
            r, first = t % 8, W * (t // 8)
            for c in range(4):
                L = 4 * r + c
                for s in range(16):
                    i = 8 * (s >> 1) + c + 4 * (s & 1)
                    if bits == 4 or s < 12:
                        base = 8 * (word_byte(L, first + (s >> 2)) + (s & 3))
                        M[t, i] = base + (np.arange(8) if bits == 4 else (Y if (s >> 2) == 1 else X))
                    else:
                        g = s - 12
                        b0, b1, b2 = (8 * (word_byte(L, first + w) + g) for w in range(3))
                        M[t, i] = [b0 + 6, b0 + 7, b1 + 2, b1 + 3, b2 + 6, b2 + 7]
        else:
            c, first, hh = (t % 8) // 2, W * (t // 8), t % 2
            for r in range(8):
                L = 4 * r + c
                for q in range(8):
                    i = 16 * (q >> 1) + r + 8 * (q & 1)
                    if bits == 4 or q < 6:
                        base = 8 * (word_byte(L, first + (q >> 1)) + 2 * hh + (q & 1))
                        M[t, i] = base + (np.arange(8) if bits == 4 else (Y if (q >> 1) == 1 else X))
                    else:
                        g = q - 6
                        b0, b1, b2 = (8 * (word_byte(L, first + w) + 2 * hh + g) for w in range(3))
                        M[t, i] = [b0 + 6, b0 + 7, b1 + 2, b1 + 3, b2 + 6, b2 + 7]
    _BIT_MAPS[key] = M
    return M


def norm_positions(which: str, slots: int) -> np.ndarray:
    """[16 tokens][slots] -> element index within a tile's norms."""
    P = np.zeros((16, slots), dtype=np.int64)
    for t in range(16):
        for b in range(slots):
            if slots == 1:
                P[t, b] = 2 * (t & 7) + (t >> 3)
            elif which == "k":
                P[t, b] = (2 * (t & 7) + (t >> 3)) * 4 + b
            else:
                P[t, b] = ((((t & 7) >> 1) * 2 + (t >> 3)) * 4 + b) * 2 + (t & 1)
    return P


def key_code_offsets(spec) -> np.ndarray:
    """[d] offset added to each key code in the tile layout of a cache with
    mixed-rate keys: 2^b for a coordinate of a b-bit group, b < 4; 0 for the
    4-bit group (include/tq.h)."""
    off = np.zeros(128, dtype=np.uint8)
    for sg in spec.segments:
        if sg.bits < 4:
            off[sg.start:sg.start + sg.length] = 1 << sg.bits
    return off


class CacheLayout:
    """Conversions between one (batch, KV head) row of a device array, as stored,
    and per-position records / norms."""

    def __init__(self, desc):
        self.tiled = int(desc.layout) == 1
        self.mixed = int(desc.k_mixed) == 1
        self.t_alloc = int(desc.t_alloc)
        self.nb = {"k": int(desc.k_code_bytes), "v": int(desc.v_code_bytes)}
        self.slots = {"k": int(desc.k_norm_slots), "v": int(desc.v_norm_slots)}

    def _offsets(self, which, kspec):
        if not (self.tiled and self.mixed and which == "k"):
            return None
        if kspec is None:
            raise ValueError("mixed-rate keys in the tile layout: the head's key spec is needed")
        return key_code_offsets(kspec)

    @staticmethod
    def _shift_nibbles(records, off, sign):
        """Add (sign = 1) or remove (sign = -1) per-coordinate offsets of nibble
        codes.  On removal a zero nibble (a position never written: a stored code
        of a 1..3-bit group is at least 2) reads back as zero."""
        out = []
        for nib, o in ((records & 15, off[0::2]), (records >> 4, off[1::2])):
            x = nib.astype(np.int16)
            y = (x + sign * o.astype(np.int16)) & 15
            if sign < 0:
                y = np.where(x == 0, 0, y)
            out.append(y)
        return (out[0] | (out[1] << 4)).astype(np.uint8)

    def records(self, raw: np.ndarray, which: str, kspec=None) -> np.ndarray:
        nb = self.nb[which]
        if not self.tiled:
            return raw.reshape(self.t_alloc, nb)
        bits = 3 if nb == 48 else 4
        M = tile_bit_map(which, bits)
        fb = M.shape[2]
        tb = np.unpackbits(raw.reshape(-1, 16 * nb), axis=1, bitorder="little")   # [tiles][tile bits]
        nat = np.zeros((tb.shape[0], 16, nb * 8), dtype=np.uint8)
        cols = (np.arange(64)[:, None] * fb + np.arange(fb)[None, :])              # record bit of (field, bit)
        for t in range(16):
            nat[:, t, cols.ravel()] = tb[:, M[t].ravel()]
        rec = np.packbits(nat, axis=2, bitorder="little").reshape(self.t_alloc, nb)
        off = self._offsets(which, kspec)
        return rec if off is None else self._shift_nibbles(rec, off, -1)

    def raw(self, records: np.ndarray, which: str, kspec=None) -> np.ndarray:
        nb = self.nb[which]
        if not self.tiled:
            return np.ascontiguousarray(records, dtype=np.uint8).reshape(-1)
        off = self._offsets(which, kspec)
        if off is not None:
            records = self._shift_nibbles(np.asarray(records, dtype=np.uint8), off, 1)
        bits = 3 if nb == 48 else 4
        M = tile_bit_map(which, bits)
        fb = M.shape[2]
        nat = np.unpackbits(records.reshape(-1, 16, nb), axis=2, bitorder="little")   # [tiles][16][bits]
        tb = np.zeros((nat.shape[0], 16 * nb * 8), dtype=np.uint8)
        cols = (np.arange(64)[:, None] * fb + np.arange(fb)[None, :])
        for t in range(16):
            tb[:, M[t].ravel()] = nat[:, t, cols.ravel()]
        return np.packbits(tb, axis=1, bitorder="little").reshape(-1)

    def norms(self, raw: np.ndarray, which: str) -> np.ndarray:
        sl = self.slots[which]
        if not self.tiled:
            return raw.reshape(self.t_alloc, sl)
        P = norm_positions(which, sl)
        tiles = raw.reshape(-1, 16 * sl)
        return tiles[:, P].reshape(self.t_alloc, sl)

    def raw_norms(self, norms: np.ndarray, which: str) -> np.ndarray:
        sl = self.slots[which]
        if not self.tiled:
            return np.ascontiguousarray(norms).reshape(-1)
        P = norm_positions(which, sl)
        out = np.zeros((self.t_alloc // 16, 16 * sl), dtype=norms.dtype)
        out[:, P] = norms.reshape(-1, 16, sl)
        return out.reshape(-1)


def _kspec(st, h):
    return None if st is None else st.specs[h][0]


def cache_records(cache, which: str, st=None) -> np.ndarray:
    """[batch][n_kv][t_alloc][code_bytes] records of a device cache (st: the
    Setup, needed for mixed-rate keys in the tile layout)."""
    lay = CacheLayout(cache.desc)
    raw = cache.codes_view(which).cpu().numpy()
    return np.stack([np.stack([lay.records(raw[b, h], which, _kspec(st, h)) for h in range(raw.shape[1])])
                     for b in range(raw.shape[0])])


def cache_norms(cache, which: str) -> np.ndarray:
    """[batch][n_kv][t_alloc][slots] norms of a device cache."""
    lay = CacheLayout(cache.desc)
    raw = cache.norms_view(which).cpu().numpy()
    return np.stack([np.stack([lay.norms(raw[b, h], which) for h in range(raw.shape[1])])
                     for b in range(raw.shape[0])])


def pair_records(cache, which: str, b: int, h: int, st=None) -> np.ndarray:
    lay = CacheLayout(cache.desc)
    return lay.records(cache.codes_view(which)[b, h].cpu().numpy(), which, _kspec(st, h))


def pair_norms(cache, which: str, b: int, h: int) -> np.ndarray:
    lay = CacheLayout(cache.desc)
    return lay.norms(cache.norms_view(which)[b, h].cpu().numpy(), which)


def put_pair(torch, cache, which: str, b: int, h: int, records: np.ndarray, norms: np.ndarray, t0: int = 0, st=None):
    """Write records / norms of positions t0 .. t0 + len - 1 of one pair into the
    device cache (the rest of the pair's row is kept)."""
    lay = CacheLayout(cache.desc)
    rec = pair_records(cache, which, b, h, st)
    nrm = pair_norms(cache, which, b, h)
    rec[t0:t0 + records.shape[0]] = records
    nrm[t0:t0 + norms.shape[0]] = norms.reshape(norms.shape[0], -1)
    cache.codes_view(which)[b, h] = torch.from_numpy(lay.raw(rec, which, _kspec(st, h)))
    cache.norms_view(which)[b, h] = torch.from_numpy(lay.raw_norms(nrm, which))


def to_torch_input(torch, x: np.ndarray, dtype: int, device="cuda"):
    if dtype == W.BF16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def segment_boundaries(spec):
    """[d][nb] fp64 boundaries per rotated coordinate (nan padded)."""
    out = np.full((128, 15), np.nan)
    for s in spec.segments:
        bd = O.codebook(s.cb_dim, s.bits).boundaries
        out[s.start:s.start + s.length, :bd.size] = bd
    return out


def compare_codes(gpu_codes: np.ndarray, enc: OracleEnc, spec, d=128):
    """Returns (n_mismatch, n_total, frac_window_normalised, frac_window_scaled,
    all_mismatches_in_window)."""
    gi = O.unpack(gpu_codes, spec, d)
    bd = segment_boundaries(spec)
    dist = np.nanmin(np.abs(enc.y[:, :, None] - bd[None]), axis=2)
    near = dist <= NEAR_WINDOW
    nseg = np.zeros((1, d))
    nrm = np.zeros(enc.y.shape)
    for s in spec.segments:
        nrm[:, s.start:s.start + s.length] = enc.norms[:, s.norm_slot].astype(np.float64)[:, None]
    near_scaled = dist * nrm <= NEAR_WINDOW
    bad = gi != enc.idx
    return (int(bad.sum()), bad.size, float(near.mean()), float(near_scaled.mean()),
            bool(np.all(near[bad])))


def compare_norms(gpu_norms: np.ndarray, enc: OracleEnc):
    a = gpu_norms.astype(np.float64)
    b = enc.norms.astype(np.float64)
    if enc.norms.dtype == np.float16:
        # equal or adjacent fp16 values
        ulp = np.spacing(np.maximum(np.abs(enc.norms), np.float16(6.1e-5)).astype(np.float16)).astype(np.float64)
        return bool(np.all(np.abs(a - b) <= ulp * 1.0001))
    return bool(np.all(np.abs(a - b) <= 4e-7 * np.maximum(np.abs(b), 1e-30)))


def oracle_attention(st: Setup, encK: OracleEnc, encV: OracleEnc, b: int, h: int, seq_len: int) -> np.ndarray:
    """[G][d] fp64 output of the oracle for one (batch, KV head)."""
    G = st.wl.group
    q = W.as_float64(st.inp.q[b, h * G:(h + 1) * G], st.wl.in_dtype)
    ks, vs = st.specs[h]
    return O.attend_rotated(q, encK.idx, encK.norms.astype(np.float64), ks, encV.idx,
                            encV.norms.astype(np.float64), vs, seq_len)


def att_error(gpu: np.ndarray, ref: np.ndarray):
    err = float(np.max(np.abs(gpu.astype(np.float64) - ref)))
    scale = float(np.max(np.abs(ref)))
    return err, scale
