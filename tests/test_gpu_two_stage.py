"""GPU parity of two-stage keys (a (k_bits - 1)-bit MSE code plus a 1-bit QJL code
of its residual, k_bits = 1 or 2)  [TQ-MNN §2.4], through the C ABI.

Write side: the kernel's MSE codes must equal the oracle's except where the
normalised rotated value lies within 1e-5 of the decision boundary; its sign bits
must equal the oracle's except where |z_j| = |(S r)_j| <= 1e-4 (the kernel forms z
in fp32, the oracle in fp64), compared on the vectors whose MSE codes all agree
(a different code moves the residual and with it every sign); both mismatch
fractions at most 1e-4.  Norms: equal or adjacent fp16 values; fp32: 4e-7
relative for ||x||, 1e-5 for ||x|| ||r||.  Values are checked as for any cache.

Read side: the oracle's records are uploaded into the device cache and the
kernel's attention must be within max-abs 2e-3 * max|o| of the oracle's
attention with the same estimated scores."""
from dataclasses import dataclass

import numpy as np
import pytest

import workloads as W
from oracle import tq_oracle as O
from gpu_harness import (ATT_TOL, MAX_MISMATCH_FRAC, NEAR_WINDOW, OracleEnc, att_error, cache_norms,
                         cache_records, compare_codes, compare_norms, put_pair, to_torch_input)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

Z_WINDOW = 1e-4


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rotated_bit_kv_gb300 as m
    m.build()
    m.lib()
    return m


@dataclass
class TwoStage:
    wl: W.Workload
    inp: W.Inputs
    qspecs: list        # per KV head: O.QjlSpec
    vspecs: list        # per KV head: the value spec
    desc: object
    blob: np.ndarray


def _setup(tq, wl, T, cap_extra=5, seq_lens=None) -> TwoStage:
    inp = W.make_inputs(wl, seq_len=T, seq_lens=seq_lens)
    desc = tq.tq_cache_desc_init(128, wl.n_q_heads, wl.n_kv_heads, wl.batch, T + cap_extra, wl.rot, wl.k_bits,
                                 wl.v_bits, wl.norm_dtype)
    S = np.stack([W.two_stage_projection(128, wl.seed, h) for h in range(wl.n_kv_heads)])
    blob = tq.tq_params_build(desc, signs=inp.signs, quats=inp.quats, k_group_mats=S)
    qspecs, vspecs = [], []
    for h in range(wl.n_kv_heads):
        if wl.rot == W.ROT_WHT128:
            base = O.spec_wht128(inp.signs[h], wl.v_bits)
        else:
            base = O.spec_so4_wht128(inp.quats[h], wl.v_bits)
        qspecs.append(O.QjlSpec(base.R, wl.k_bits - 1, S[h].astype(np.float64)))
        vspecs.append(base)
    return TwoStage(wl, inp, qspecs, vspecs, desc, blob)


def _norm_name(wl):
    return "f16" if wl.norm_dtype == W.F16 else "f32"


def _encode_k(st, b, h, t0=0, t1=None):
    x = W.as_float64(st.inp.K[b, t0:t1, h], st.wl.in_dtype)
    qs = st.qspecs[h]
    idx, sb, nr, y, z = O.qjl_quantize(x, qs, _norm_name(st.wl))
    return O.qjl_pack(idx, sb, qs.mse_bits), idx, sb, nr, y, z


def _encode_v(st, b, h, t0=0, t1=None):
    x = W.as_float64(st.inp.V[b, t0:t1, h], st.wl.in_dtype)
    spec = st.vspecs[h]
    idx, nr, y = O.quantize(x, spec, _norm_name(st.wl))
    return OracleEnc(O.pack(idx, spec), idx, nr, y)


def _workload(k_bits, variant="f16", **kw):
    wl = W.two_stage_keys(k_bits)
    if variant == "f32":
        wl = wl.with_(norm_dtype=W.F32)
    elif variant == "so4":
        wl = wl.with_(rot=W.ROT_SO4_WHT128)
    elif variant == "v4":
        wl = wl.with_(v_bits=4)
    return wl.with_(**kw)


def _append(tq, st):
    cache = tq.PackedKVCache(st.desc, st.blob)
    K = to_torch_input(torch, st.inp.K, st.wl.in_dtype)
    V = to_torch_input(torch, st.inp.V, st.wl.in_dtype)
    cache.append(K, V, torch.zeros(st.wl.batch, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    return cache


@pytest.mark.parametrize("variant", ["f16", "f32", "so4"])
@pytest.mark.parametrize("k_bits", [1, 2])
def test_append_matches_oracle(tq, k_bits, variant):
    B, T = 2, 333
    st = _setup(tq, _workload(k_bits, variant, batch=B), T)
    cache = _append(tq, st)
    assert int(cache.status.item()) == 0
    assert st.desc.layout == tq.TQ_LAYOUT_NATURAL
    kc, vc = cache_records(cache, "k"), cache_records(cache, "v")
    kn, vn = cache_norms(cache, "k"), cache_norms(cache, "v")
    mb = k_bits - 1
    code_bad = code_tot = sign_bad = sign_tot = 0
    for b in range(B):
        for h in range(st.wl.n_kv_heads):
            _, idx, sb, nr, y, z = _encode_k(st, b, h)
            gi, gs = O.qjl_unpack(kc[b, h, :T], mb)
            bad = gi != idx
            assert np.all(np.abs(y[bad]) <= NEAR_WINDOW), "an MSE code differs away from its boundary"
            code_bad += int(bad.sum())
            code_tot += bad.size
            same = ~bad.any(axis=1)                       # vectors whose MSE codes all agree
            sbad = (gs != sb) & same[:, None]
            assert np.all(np.abs(z[sbad]) <= Z_WINDOW), np.abs(z[sbad]).max()
            sign_bad += int(sbad.sum())
            sign_tot += int(same.sum()) * 128
            g = kn[b, h, :T]
            assert compare_norms(g[:, 0:1], OracleEnc(None, None, nr[:, 0:1], None)), "||x||"
            if st.wl.norm_dtype == W.F16:
                assert compare_norms(g[same, 1:2], OracleEnc(None, None, nr[same, 1:2], None)), "||x|| ||r||"
            else:
                a, e = g[same, 1].astype(np.float64), nr[same, 1].astype(np.float64)
                assert np.all(np.abs(a - e) <= 1e-5 * np.maximum(e, 1e-30)), "||x|| ||r||"
            assert not kc[b, h, T:].any()
            ev = _encode_v(st, b, h)
            nbad, n, fw, fws, ok = compare_codes(vc[b, h, :T], ev, st.vspecs[h])
            assert ok and nbad / n <= MAX_MISMATCH_FRAC
            assert compare_norms(vn[b, h, :T], ev)
    assert code_bad / code_tot <= MAX_MISMATCH_FRAC, (code_bad, code_tot)
    assert sign_bad / sign_tot <= MAX_MISMATCH_FRAC, (sign_bad, sign_tot)


def _upload(tq, st, cache, T):
    encs = {}
    for b in range(st.wl.batch):
        for h in range(st.wl.n_kv_heads):
            codes, idx, sb, nr, y, z = _encode_k(st, b, h, 0, T)
            ev = _encode_v(st, b, h, 0, T)
            put_pair(torch, cache, "k", b, h, codes, nr)
            put_pair(torch, cache, "v", b, h, ev.codes, ev.norms)
            encs[(b, h)] = (idx, sb, nr, ev)
    torch.cuda.synchronize()
    return encs


def _check(tq, st, cache, encs, seq_lens, max_seq, v_mode=-1, n_splits=0):
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.from_numpy(np.asarray(seq_lens, dtype=np.int32)).cuda()
    out = cache.decode(q, sl, max_seq, v_mode=v_mode, n_splits=n_splits)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    G = st.wl.group
    errs, scales = [], []
    for (b, h), (idx, sb, nr, ev) in encs.items():
        qb = W.as_float64(st.inp.q[b, h * G:(h + 1) * G], st.wl.in_dtype)
        L = int(min(seq_lens[b], max_seq))
        ref = O.attend_qjl(qb, idx, sb, nr.astype(np.float64), st.qspecs[h], ev.idx, ev.norms.astype(np.float64),
                           st.vspecs[h], L)
        e, s = att_error(o[b, h * G:(h + 1) * G], ref)
        errs.append(e)
        scales.append(s)
    err, scale = max(errs), max(scales)
    assert err <= ATT_TOL * max(scale, 1e-30), (err, scale)
    return err, scale


@pytest.mark.parametrize("n_splits", [1, 3, 0])
@pytest.mark.parametrize("v_mode", [0, 1])
@pytest.mark.parametrize("k_bits,variant", [(1, "f16"), (2, "f16"), (2, "v4"), (1, "so4"), (2, "f32")])
def test_decode_matches_oracle(tq, k_bits, variant, v_mode, n_splits):
    B, T = 2, 333
    seq_lens = W.ragged_lengths(B, T, 5)
    st = _setup(tq, _workload(k_bits, variant, batch=B), T, seq_lens=seq_lens)
    cache = tq.PackedKVCache(st.desc, st.blob)
    encs = _upload(tq, st, cache, T)
    _check(tq, st, cache, encs, st.inp.seq_lens, T, v_mode, n_splits)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("G", [1, 16])
@pytest.mark.parametrize("k_bits", [1, 2])
def test_decode_query_groups(tq, k_bits, G):
    """One and sixteen query heads per KV head (padded groups 1 and 16)."""
    B, T = 2, 300
    wl = _workload(k_bits, batch=B, n_kv_heads=2, n_q_heads=2 * G)
    st = _setup(tq, wl, T)
    cache = tq.PackedKVCache(st.desc, st.blob)
    encs = _upload(tq, st, cache, T)
    _check(tq, st, cache, encs, st.inp.seq_lens, T)


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129])
def test_decode_short(tq, T):
    st = _setup(tq, _workload(2, batch=1, n_kv_heads=2, n_q_heads=8), T, cap_extra=1)
    cache = tq.PackedKVCache(st.desc, st.blob)
    encs = _upload(tq, st, cache, T)
    for v_mode in (0, 1):
        for n_splits in (1, 2, 0):
            _check(tq, st, cache, encs, [T], T, v_mode, n_splits)


def test_decode_empty_and_clamped(tq):
    """A sequence of length 0 gives 0; a length above max_seq_len is clamped to it
    and flagged."""
    B, T = 3, 200
    st = _setup(tq, _workload(1, batch=B, n_kv_heads=2, n_q_heads=8), T)
    cache = tq.PackedKVCache(st.desc, st.blob)
    encs = _upload(tq, st, cache, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.tensor([0, 150, 200], dtype=torch.int32, device="cuda")
    out = cache.decode(q, sl, 160)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert not o[0].any()
    assert int(cache.status.item()) & tq.TQ_DEV_SEQ_OVER_MAX
    _check(tq, st, cache, {k: v for k, v in encs.items() if k[0] > 0}, [0, 150, 200], 160)


def test_prefix_plus_two_stage(tq):
    """Unquantised fp16 tokens plus a cache with two-stage keys
    (tq_decode_attention_prefix): the packed part's estimated scores and the
    unquantised part's exact ones, merged by log-sum-exp (each part's state from
    the oracle's functions)."""
    B, T, P = 2, 300, 96
    st = _setup(tq, _workload(2, batch=B, n_kv_heads=2, n_q_heads=8), T)
    cache = tq.PackedKVCache(st.desc, st.blob)
    encs = _upload(tq, st, cache, T)
    rng = np.random.default_rng([3, 0x5046])
    Kp = (rng.standard_normal((B, P, 2, 128)) * 2.0).astype(np.float16)
    Vp = rng.standard_normal((B, P, 2, 128)).astype(np.float16)
    plens, lens = np.array([P, 40], np.int32), np.array([T, 123], np.int32)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    out = cache.decode_prefix(q, torch.from_numpy(lens).cuda(), T, torch.from_numpy(Kp).cuda(),
                              torch.from_numpy(Vp).cuda(), torch.from_numpy(plens).cuda(), P)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    o = out.cpu().numpy()
    G = st.wl.group
    errs, scales = [], []
    for (b, h), (idx, sb, nr, ev) in encs.items():
        qh = W.as_float64(st.inp.q[b, h * G:(h + 1) * G], st.wl.in_dtype)
        L = int(lens[b])
        s = O.qjl_scores(qh, idx[:L], sb[:L], nr[:L].astype(np.float64), st.qspecs[h]) / np.sqrt(128.0)
        m1 = s.max(axis=1)
        p = np.exp(s - m1[:, None])
        vt = O.dequantize_rotated(ev.idx[:L], ev.norms[:L].astype(np.float64), st.vspecs[h])
        o1, l1 = (p @ vt) @ st.vspecs[h].R, p.sum(axis=1)
        n = int(plens[b])
        m2, l2, o2 = O.part_state(qh, Kp[b, :n, h].astype(np.float64), Vp[b, :n, h].astype(np.float64))
        M = np.maximum(m1, m2)
        w1, w2 = np.exp(m1 - M), np.exp(m2 - M)
        ref = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 * l1 + w2 * l2)[:, None]
        e, sc = att_error(o[b, h * G:(h + 1) * G], ref)
        errs.append(e)
        scales.append(sc)
    assert max(errs) <= ATT_TOL * max(scales), (max(errs), max(scales))
