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
    desc = tq.tq_cache_desc_init(wl.head_dim, wl.n_q_heads, wl.n_kv_heads, wl.batch, t_capacity, wl.rot,
                                 0 if wl.mixed_k else wl.k_bits, wl.v_bits, wl.norm_dtype, int(wl.mixed_k))
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
