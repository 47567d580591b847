"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI.

Write side: the kernel's packed codes must equal the oracle's except at
coordinates whose normalised rotated value lies within 1e-5 of a decision
boundary; those mismatches must be at most 1e-4 of all codes.  Stored norms
must be equal or adjacent fp16 values (fp32: within 4e-7 relative).

Read side: the oracle's packed cache is uploaded into the device cache and the
kernel's attention output must be within max-abs 2e-3 * max|o| of the
oracle's attention on that same cache."""
import numpy as np
import pytest

import workloads as W
from oracle import tq_oracle as O
from gpu_harness import (ATT_TOL, MAX_MISMATCH_FRAC, att_error, cache_norms, cache_records, compare_codes,
                         compare_norms, make_setup, oracle_attention, oracle_encode, pair_records, put_pair,
                         to_torch_input)

pytestmark = pytest.mark.gpu

# (workload, batch, T, mismatch fraction, near-boundary fraction normalised / scaled),
# printed at the end of the session
STATS = []

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rotated_bit_kv_gb300 as m
    m.build()
    m.lib()
    return m


def _workload(name):
    return {
        "tiny": W.tiny_single_head(),
        "llama8b": W.llama8b_decode(),
        "block32_tq3": W.block32(3),
        "block32_tq4": W.block32(4),
        "so4": W.so4_wht(),
        "mixed": W.mixed_rate_long(),
        # mixed-rate keys with four query heads per KV head
        "mixed_g4": W.mixed_rate_long().with_(n_q_heads=8),
        # natural-layout variants of the same formats (CUDA-core decode kernels):
        # 16 query heads per KV head, and fp32 norms with 32-wide blocks or with
        # mixed-rate keys
        "llama8b_g16": W.llama8b_decode().with_(n_kv_heads=2),
        "block32_f32": W.block32(3).with_(norm_dtype=W.F32),
        "mixed_f32": W.mixed_rate_long().with_(norm_dtype=W.F32),
        # mixed-rate keys in tight records: 3 bits on average (48 B), and 2 bits
        # with four query heads per KV head (32 B)
        "mixed_tight": W.mixed_rate_long().with_(tight_k=True),
        "mixed_tight2": W.mixed_rate_long().with_(tight_k=True, avg_bits=2, n_q_heads=8),
    }[name]


SMALL = {  # (batch, T) element-wise cases: several tiles and a ragged tail
    "tiny": (1, 256),
    "llama8b": (3, 333),
    "block32_tq3": (2, 333),
    "block32_tq4": (2, 333),
    "so4": (1, 333),
    "mixed": (1, 700),
    "mixed_g4": (2, 600),
    "llama8b_g16": (2, 333),
    "block32_f32": (2, 333),
    "mixed_f32": (1, 600),
    "mixed_tight": (1, 700),
    "mixed_tight2": (2, 600),
}
# TQ_LAYOUT_TILE16 caches (tensor-core decode kernel)
TILED = ["tiny", "llama8b", "block32_tq3", "block32_tq4", "so4", "mixed", "mixed_g4"]
# TQ_LAYOUT_NATURAL caches (CUDA-core decode kernels)
NATURAL = ["llama8b_g16", "block32_f32", "mixed_f32", "mixed_tight", "mixed_tight2"]


def _encode_on_gpu(tq, name, B, T, cap_extra=5, seq_lens=None):
    wl = _workload(name).with_(batch=B)
    inp = W.make_inputs(wl, seq_len=T, seq_lens=seq_lens)
    st = make_setup(tq, wl, inp, T + cap_extra)
    cache = tq.PackedKVCache(st.desc, st.blob)
    K = to_torch_input(torch, inp.K, wl.in_dtype)
    V = to_torch_input(torch, inp.V, wl.in_dtype)
    start = torch.zeros(B, dtype=torch.int32, device="cuda")
    cache.append(K, V, start)
    torch.cuda.synchronize()
    return st, cache


@pytest.mark.parametrize("name", list(SMALL))
def test_quantize_append_matches_oracle(tq, name):
    B, T = SMALL[name]
    st, cache = _encode_on_gpu(tq, name, B, T)
    assert int(cache.status.item()) == 0
    assert st.desc.layout == (tq.TQ_LAYOUT_TILE16 if name in TILED else tq.TQ_LAYOUT_NATURAL)
    kc, vc = cache_records(cache, "k", st), cache_records(cache, "v", st)
    kn, vn = cache_norms(cache, "k"), cache_norms(cache, "v")
    tot = bad = 0
    fws_all, fw_all = [], []
    for b in range(B):
        for h in range(st.wl.n_kv_heads):
            for which, codes, norms in (("k", kc, kn), ("v", vc, vn)):
                enc = oracle_encode(st, which, b, h)
                spec = st.specs[h][0 if which == "k" else 1]
                nbad, n, fw, fws, ok = compare_codes(codes[b, h, :T], enc, spec)
                assert ok, f"{which} b={b} h={h}: a mismatch outside the near-boundary window"
                bad += nbad
                tot += n
                fw_all.append(fw)
                fws_all.append(fws)
                assert compare_norms(norms[b, h, :T], enc), f"{which} norms b={b} h={h}"
                # slots beyond T stay untouched (zero)
                assert not codes[b, h, T:].any()
    assert bad / tot <= MAX_MISMATCH_FRAC, (bad, tot)
    # the near-boundary fraction, in the frame of the stored value n * y (|n (y - b)| <= 1e-5):
    # at most 1e-4 for uniform-rate caches; mixed-rate keys normalise small low-energy
    # groups whose norms are tiny, so there it is reported only (their mismatch fraction
    # is gated above like every other format's)
    if not st.wl.mixed_k:
        assert np.mean(fws_all) <= 1e-4, np.mean(fws_all)
    STATS.append((name, B, T, bad / tot, float(np.mean(fw_all)), float(np.mean(fws_all))))


def _check_codes_vs_oracle(st, cache, B, T):
    kc, vc = cache_records(cache, "k", st), cache_records(cache, "v", st)
    kn, vn = cache_norms(cache, "k"), cache_norms(cache, "v")
    tot = bad = 0
    for b in range(B):
        for h in range(st.wl.n_kv_heads):
            for which, codes, norms in (("k", kc, kn), ("v", vc, vn)):
                enc = oracle_encode(st, which, b, h)
                spec = st.specs[h][0 if which == "k" else 1]
                nbad, n, fw, fws, ok = compare_codes(codes[b, h, :T], enc, spec)
                assert ok, f"{which} b={b} h={h}: a mismatch outside the near-boundary window"
                bad += nbad
                tot += n
                assert compare_norms(norms[b, h, :T], enc), f"{which} norms b={b} h={h}"
    assert bad / tot <= MAX_MISMATCH_FRAC, (bad, tot)
    return kc, vc


@pytest.mark.parametrize("name", ["llama8b", "so4", "block32_tq4"])
def test_quantize_paths_agree(tq, name):
    """The write side has three kernels: whole prompts of 3-bit WHT128 caches with
    16-bit, 16-byte aligned inputs go through the tensor cores, other 16-byte
    aligned inputs (and short appends) through the half-warp kernel, inputs aligned
    to 8 bytes only (whole prompts or chunks) through the one-warp-per-vector
    kernel.  Each matches the oracle and the others."""
    B, T = SMALL[name]
    wl = _workload(name).with_(batch=B)
    inp = W.make_inputs(wl, seq_len=T)
    st = make_setup(tq, wl, inp, T + 5)
    K = to_torch_input(torch, inp.K, wl.in_dtype)
    V = to_torch_input(torch, inp.V, wl.in_dtype)
    out = []
    for mode, shift in (("whole", 0), ("chunks", 0), ("chunks", 4), ("whole", 4)):
        c = tq.PackedKVCache(st.desc, st.blob)
        if shift:   # an offset of 4 elements: 8-byte (bf16) aligned only
            kb = torch.empty(K.numel() + shift, dtype=K.dtype, device="cuda")
            vb = torch.empty(V.numel() + shift, dtype=V.dtype, device="cuda")
            kb[shift:].copy_(K.reshape(-1))
            vb[shift:].copy_(V.reshape(-1))
            Kx, Vx = kb[shift:].view(K.shape), vb[shift:].view(V.shape)
            assert Kx.data_ptr() % 16 == 8
        else:
            Kx, Vx = K, V
            assert Kx.data_ptr() % 16 == 0
        if mode == "chunks":   # appends of 40 tokens (short appends never take the tensor-core kernel)
            for t0 in range(0, T, 40):
                t1 = min(T, t0 + 40)
                kc, vc = Kx[:, t0:t1], Vx[:, t0:t1]
                if shift:   # keep the 8-byte alignment of the chunk copies
                    kc = torch.empty(kc.numel() + shift, dtype=K.dtype, device="cuda")[shift:].view(kc.shape)
                    vc = torch.empty(vc.numel() + shift, dtype=V.dtype, device="cuda")[shift:].view(vc.shape)
                    kc.copy_(Kx[:, t0:t1])
                    vc.copy_(Vx[:, t0:t1])
                else:
                    kc, vc = kc.contiguous(), vc.contiguous()
                c.append(kc, vc, torch.full((B,), t0, dtype=torch.int32, device="cuda"))
        else:
            c.append(Kx, Vx, torch.zeros(B, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert int(c.status.item()) == 0
        out.append(_check_codes_vs_oracle(st, c, B, T))
    for x in out[1:]:
        for a, b in zip(out[0], x):
            assert np.mean(a != b) <= MAX_MISMATCH_FRAC


@pytest.mark.parametrize("in_dtype,B,T,pairs", [
    (W.BF16, 2, 701, None),              # 4206 triples: a ragged last tile of 6
    (W.F16, 2, 701, None),               # fp16 operands
    (W.BF16, 2, 14001, [(0, 0), (1, 2)]),   # more tiles than warps: the grid-stride loop
])
def test_quantize_tc_heads_and_tails(tq, in_dtype, B, T, pairs):
    """Tensor-core write path with 3 KV heads (lanes of a warp on different heads;
    the warp count rounded to keep each lane on one head) against the oracle."""
    wl = W.llama8b_decode().with_(n_q_heads=12, n_kv_heads=3, batch=B, in_dtype=in_dtype)
    inp = W.make_inputs(wl, seq_len=T)
    st = make_setup(tq, wl, inp, T + 3)
    c = tq.PackedKVCache(st.desc, st.blob)
    K = to_torch_input(torch, inp.K, wl.in_dtype)
    V = to_torch_input(torch, inp.V, wl.in_dtype)
    c.append(K, V, torch.full((B,), 2, dtype=torch.int32, device="cuda"))   # slots 2 .. T+1
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    kc, vc = cache_records(c, "k", st), cache_records(c, "v", st)
    kn, vn = cache_norms(c, "k"), cache_norms(c, "v")
    bad = tot = 0
    for (b, h) in pairs or [(b, h) for b in range(B) for h in range(3)]:
        for which, codes, norms in (("k", kc, kn), ("v", vc, vn)):
            enc = oracle_encode(st, which, b, h)
            nb, n, _, _, ok = compare_codes(codes[b, h, 2:T + 2], enc, st.specs[h][0 if which == "k" else 1])
            assert ok, f"{which} b={b} h={h}"
            bad += nb
            tot += n
            assert compare_norms(norms[b, h, 2:T + 2], enc)
            assert not codes[b, h, :2].any() and not codes[b, h, T + 2:].any()
    assert bad / tot <= MAX_MISMATCH_FRAC


def test_quantize_tc_search_without_shared_table(tq):
    """The tensor-core write kernel searches through one cell table when every
    head's K and V boundaries are the same (they are whenever the library built
    the parameters); otherwise it falls back to a binary search per head.  Head 1's
    V boundaries moved up by one ulp force the fallback: every head still matches
    the oracle, and every other vector's codes equal those of the table search."""
    B, T = SMALL["llama8b"]
    wl = _workload("llama8b").with_(batch=B)
    inp = W.make_inputs(wl, seq_len=T)
    st = make_setup(tq, wl, inp, T + 5)
    bd = O.codebook(128, 3).boundaries.astype(np.float32)   # the library's fp32 boundaries
    raw = np.frombuffer(bytes(st.blob), dtype=np.uint8).copy()
    pat = bd.tobytes()
    hits = [i for i in range(0, raw.size - len(pat) + 1, 4) if raw[i:i + len(pat)].tobytes() == pat]
    assert len(hits) == 2 * wl.n_kv_heads, len(hits)   # K then V boundaries of each head, in head order
    moved = raw.copy()
    moved[hits[3]:hits[3] + len(pat)] = np.frombuffer(np.nextafter(bd, np.float32(np.inf)).tobytes(), np.uint8)
    K = to_torch_input(torch, inp.K, wl.in_dtype)
    V = to_torch_input(torch, inp.V, wl.in_dtype)
    res = []
    for blob in (raw, moved):
        c = tq.PackedKVCache(st.desc, blob)
        c.append(K, V, torch.zeros(B, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert int(c.status.item()) == 0
        res.append(_check_codes_vs_oracle(st, c, B, T))
    (k0, v0), (k1, v1) = res
    assert np.array_equal(k0, k1)
    keep = [h for h in range(wl.n_kv_heads) if h != 1]
    assert np.array_equal(v0[:, keep], v1[:, keep])


def _upload_oracle_cache(tq, st, cache, B, T):
    """Write the oracle's records into the device cache (in the cache's layout,
    converted by the harness); returns the encodings."""
    encs = {}
    for b in range(B):
        for h in range(st.wl.n_kv_heads):
            ek = oracle_encode(st, "k", b, h, 0, T)
            ev = oracle_encode(st, "v", b, h, 0, T)
            put_pair(torch, cache, "k", b, h, ek.codes, ek.norms, st=st)
            put_pair(torch, cache, "v", b, h, ev.codes, ev.norms, st=st)
            encs[(b, h)] = (ek, ev)
    torch.cuda.synchronize()
    return encs


def _check_decode(tq, st, cache, encs, q, seq_lens, max_seq, v_mode, n_splits, pairs=None):
    out = cache.decode(q, seq_lens, max_seq, v_mode=v_mode, n_splits=n_splits)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    G = st.wl.group
    errs, scales = [], []
    L = seq_lens.cpu().numpy()
    pairs = pairs or list(encs)
    for (b, h) in pairs:
        ek, ev = encs[(b, h)]
        ref = oracle_attention(st, ek, ev, b, h, int(min(L[b], max_seq)))
        e, s = att_error(o[b, h * G:(h + 1) * G], ref)
        errs.append(e)
        scales.append(s)
    err, scale = max(errs), max(scales)
    assert err <= ATT_TOL * scale, (err, scale)
    return err, scale


@pytest.mark.parametrize("n_splits", [1, 3, 0])
@pytest.mark.parametrize("name", list(SMALL))
def test_decode_matches_oracle(tq, name, n_splits):
    """The automatic kernel of every format (tensor cores on the tile layout, the
    crossover's CUDA-core kernel on the natural layout) with 1, 3 and the
    automatic number of splits (tensor cores: CTAs over all tiles)."""
    B, T = SMALL[name]
    seq_lens = W.ragged_lengths(B, T, 3) if B > 1 else None
    st, cache = _encode_on_gpu(tq, name, B, T, seq_lens=seq_lens)
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.from_numpy(st.inp.seq_lens).cuda()
    _check_decode(tq, st, cache, encs, q, sl, T, -1, n_splits)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("v_mode", [0, 1])
@pytest.mark.parametrize("n_splits", [1, 3, 0])
@pytest.mark.parametrize("name", NATURAL)
def test_decode_cuda_core_modes(tq, name, v_mode, n_splits):
    """Token- and dimension-parallel V accumulation on natural-layout caches."""
    B, T = SMALL[name]
    seq_lens = W.ragged_lengths(B, T, 3) if B > 1 else None
    st, cache = _encode_on_gpu(tq, name, B, T, seq_lens=seq_lens)
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.from_numpy(st.inp.seq_lens).cuda()
    _check_decode(tq, st, cache, encs, q, sl, T, v_mode, n_splits)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("T", [1, 2, 31, 127, 128, 129, 511, 512])
@pytest.mark.parametrize("name", ["so4", "llama8b_g16"])
def test_decode_short_and_tile_edges(tq, name, T):
    st, cache = _encode_on_gpu(tq, name, 1, T)
    encs = _upload_oracle_cache(tq, st, cache, 1, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.full((1,), T, dtype=torch.int32, device="cuda")
    modes = (-1, 2, 3) if name in TILED else (0, 1, -1)
    for v_mode in modes:
        _check_decode(tq, st, cache, encs, q, sl, T, v_mode, 0)


def test_v_mode_plan(tq):
    """Tile-layout caches take the tensor-core kernel at every length (and no
    CUDA-core kernel); natural-layout caches take dimension-parallel V
    accumulation at every length (their measured crossover is 0)."""
    for name in ("so4", "block32_tq3", "block32_tq4", "tiny"):
        st, _ = _encode_on_gpu(tq, name, 1, 8, cap_extra=601)     # any capacity (tiles are padded)
        for T in (8, 511, 512, 600):
            assert tq.tq_decode_plan(st.desc, T)[1] == tq.TQ_VMODE_TENSOR
        for vm in (tq.TQ_VMODE_TOKEN_PARALLEL, tq.TQ_VMODE_DIM_PARALLEL):
            with pytest.raises(tq.TQError) as e:
                tq.tq_decode_plan(st.desc, 512, vm)
            assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    for name in ("llama8b_g16", "block32_f32", "mixed_f32"):
        T0 = 600 if name == "mixed_f32" else 8   # mixed-rate keys calibrate on 512 tokens
        st, _ = _encode_on_gpu(tq, name, 1, T0, cap_extra=600)
        for T in (1, 511, 512):   # measured crossover 0: dimension-parallel at every length
            assert tq.tq_decode_plan(st.desc, T)[1] == tq.TQ_VMODE_DIM_PARALLEL
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_plan(st.desc, 512, tq.TQ_VMODE_TENSOR)
        assert e.value.status == tq.TQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("grid", [1, 3, 0])
@pytest.mark.parametrize("name", TILED)
def test_decode_tensor_matches_oracle(tq, name, grid):
    """Tensor-core kernel with 1, 3 and the automatic number of CTAs; ragged
    lengths and a capacity that is not a whole number of tiles."""
    B, T = SMALL[name]
    seq_lens = W.ragged_lengths(B, T, 4) if B > 1 else None
    st, cache = _encode_on_gpu(tq, name, B, T, cap_extra=3, seq_lens=seq_lens)
    assert st.desc.t_alloc % 16 == 0 and st.desc.t_alloc >= st.desc.t_capacity
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.from_numpy(st.inp.seq_lens).cuda()
    _check_decode(tq, st, cache, encs, q, sl, T, tq.TQ_VMODE_TENSOR, grid)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("T", [1, 15, 16, 17, 64, 100, 512, 1000])
@pytest.mark.parametrize("name", ["llama8b", "so4", "block32_tq3", "block32_tq4"])
def test_decode_tensor_tile_edges(tq, name, T):
    st, cache = _encode_on_gpu(tq, name, 1, T, cap_extra=1)
    encs = _upload_oracle_cache(tq, st, cache, 1, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.full((1,), T, dtype=torch.int32, device="cuda")
    for grid in (0, 1, 2):
        _check_decode(tq, st, cache, encs, q, sl, T, tq.TQ_VMODE_TENSOR, grid)


@pytest.mark.parametrize("n_splits", [77, 300])
@pytest.mark.parametrize("name,v_mode", [("so4", 2), ("block32_tq4", 2), ("llama8b", 2), ("block32_f32", 1),
                                         ("llama8b_g16", 0)])
def test_decode_many_splits(tq, name, v_mode, n_splits):
    """Many partials per pair: CUDA-core kernels with key-axis splits well beyond
    a warp's width (the merge walks the partials 32 at a time for the weights, 8
    at a time for the outputs), many of them empty; the tensor-core kernel with
    77 or 300 CTAs over few tiles (most CTAs hold a piece of one tile or none).
    Ragged lengths."""
    B, T = 2, 1000
    seq_lens = W.ragged_lengths(B, T, 7)
    st, cache = _encode_on_gpu(tq, name, B, T, seq_lens=seq_lens)
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.from_numpy(st.inp.seq_lens).cuda()
    _check_decode(tq, st, cache, encs, q, sl, T, v_mode, n_splits)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("name", ["tiny", "llama8b", "so4", "block32_tq3"])
def test_decode_streamk_matches_oracle(tq, name):
    """Ragged lengths put pair boundaries anywhere inside a CTA's range."""
    B, T = SMALL[name]
    B = max(B, 5)
    seq_lens = W.ragged_lengths(B, T, 6)
    st, cache = _encode_on_gpu(tq, name, B, T, seq_lens=seq_lens)
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.from_numpy(st.inp.seq_lens).cuda()
    for grid in (0, 7, 40):
        _check_decode(tq, st, cache, encs, q, sl, T, tq.TQ_VMODE_TENSOR_STREAMK, grid)
    assert int(cache.status.item()) == 0


def test_decode_streamk_empty_and_clamped(tq):
    B, T = 4, 200
    st, cache = _encode_on_gpu(tq, "llama8b", B, T)
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.tensor([0, T + 50, 0, 77], dtype=torch.int32, device="cuda")
    out = cache.decode(q, sl, T, v_mode=tq.TQ_VMODE_TENSOR_STREAMK)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert int(cache.status.item()) & tq.TQ_DEV_SEQ_OVER_CAPACITY
    G = st.wl.group
    for b, L in ((1, T), (3, 77)):
        for h in range(st.wl.n_kv_heads):
            ek, ev = encs[(b, h)]
            ref = oracle_attention(st, ek, ev, b, h, L)
            e, s = att_error(o[b, h * G:(h + 1) * G], ref)
            assert e <= ATT_TOL * s


def test_seq_len_zero_and_clamping(tq):
    B, T = 3, 200
    st, cache = _encode_on_gpu(tq, "llama8b", B, T, cap_extra=0)
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    # batch 0 empty, batch 1 over capacity (clamped to T), batch 2 normal
    sl = torch.tensor([0, T + 50, 77], dtype=torch.int32, device="cuda")
    out = cache.decode(q, sl, T)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.all(o[0] == 0)
    st_word = int(cache.status.item())
    assert st_word & tq.TQ_DEV_SEQ_OVER_CAPACITY
    G = st.wl.group
    for b, L in ((1, T), (2, 77)):
        for h in range(st.wl.n_kv_heads):
            ek, ev = encs[(b, h)]
            ref = oracle_attention(st, ek, ev, b, h, L)
            e, s = att_error(o[b, h * G:(h + 1) * G], ref)
            assert e <= ATT_TOL * s


def test_append_positions_and_incremental(tq):
    """Appending token by token at increasing positions gives the same cache
    as one whole-prompt call; positions outside the capacity are skipped and
    flagged."""
    B, T = 2, 40
    st, cache = _encode_on_gpu(tq, "llama8b", B, T)
    whole_k = cache.codes_view("k").clone()
    whole_kn = cache.norms_view("k").clone()
    whole_v = cache.codes_view("v").clone()
    whole_vn = cache.norms_view("v").clone()
    cache2 = tq.PackedKVCache(st.desc, st.blob)
    K = to_torch_input(torch, st.inp.K, st.wl.in_dtype)
    V = to_torch_input(torch, st.inp.V, st.wl.in_dtype)
    for t in range(0, T, 7):
        n = min(7, T - t)
        cache2.append(K[:, t:t + n].contiguous(), V[:, t:t + n].contiguous(),
                      torch.full((B,), t, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(cache2.codes_view("k"), whole_k)
    assert torch.equal(cache2.norms_view("k"), whole_kn)
    assert torch.equal(cache2.codes_view("v"), whole_v)   # value halves of one token never touch another's
    assert torch.equal(cache2.norms_view("v"), whole_vn)
    assert int(cache2.status.item()) == 0
    # out-of-range start position: skipped and flagged; n_new = 0 is a no-op
    before = cache_records(cache2, "v", st)
    cache2.append(K[:, :3].contiguous(), V[:, :3].contiguous(),
                  torch.tensor([st.desc.t_capacity - 1, -5], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(cache2.status.item()) & tq.TQ_DEV_BAD_POSITION
    after = cache_records(cache2, "v", st)
    cap = st.desc.t_capacity
    assert np.array_equal(after[1], before[1])             # batch 1 entirely skipped
    assert np.array_equal(after[0, :, :cap - 1], before[0, :, :cap - 1])
    assert np.array_equal(after[0, :, cap:], before[0, :, cap:])   # tile padding untouched
    tq.tq_quantize_append(st.desc, cache2.ptrs, K[:, :0].contiguous(), V[:, :0].contiguous(),
                          torch.zeros(B, dtype=torch.int32, device="cuda"), 0)


def test_quantize_tc_positions_outside_capacity(tq):
    """Whole-prompt (tensor-core) append whose positions leave [0, capacity) at
    either end: each token outside is skipped and flagged, the others encoded."""
    B, T = 2, 300                       # 4800 triples: the tensor-core kernel
    wl = _workload("llama8b").with_(batch=B)
    inp = W.make_inputs(wl, seq_len=T)
    cap = T + 5
    st = make_setup(tq, wl, inp, cap)
    c = tq.PackedKVCache(st.desc, st.blob)
    K = to_torch_input(torch, inp.K, wl.in_dtype)
    V = to_torch_input(torch, inp.V, wl.in_dtype)
    start = cap - 100   # batch 0: tokens 0..99 fit, 100.. run past the end
    c.append(K, V, torch.tensor([start, -5], dtype=torch.int32, device="cuda"))   # batch 1: tokens 0..4 before slot 0
    torch.cuda.synchronize()
    assert int(c.status.item()) & tq.TQ_DEV_BAD_POSITION
    for which in ("k", "v"):
        codes = cache_records(c, which, st)
        norms = cache_norms(c, which)
        assert not codes[0, :, :start].any() and not norms[0, :, :start].any()
        assert not codes[1, :, T - 5:].any() and not norms[1, :, T - 5:].any()
        for h in range(wl.n_kv_heads):
            spec = st.specs[h][0 if which == "k" else 1]
            for b, t0, t1, s0 in ((0, 0, 100, start), (1, 5, T, 0)):
                enc = oracle_encode(st, which, b, h, t0, t1)
                _, _, _, _, ok = compare_codes(codes[b, h, s0:s0 + t1 - t0], enc, spec)
                assert ok
                assert compare_norms(norms[b, h, s0:s0 + t1 - t0], enc)


def test_argument_errors(tq):
    st, cache = _encode_on_gpu(tq, "tiny", 1, 8)
    q = to_torch_input(torch, st.inp.q, st.wl.in_dtype)
    sl = torch.full((1,), 8, dtype=torch.int32, device="cuda")
    out = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError) as e:          # max_seq above capacity
        tq.tq_decode_attention(st.desc, cache.ptrs, q, sl, 10 ** 6, out, cache.workspace)
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    small_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TQError) as e:          # workspace too small for 4 CTAs
        tq.tq_decode_attention_ex(st.desc, cache.ptrs, q, sl, 8, out, small_ws, None, None, 2, 4)
    assert e.value.status == tq.TQ_ERR_WORKSPACE
    with pytest.raises(tq.TQError) as e:          # a CUDA-core kernel on a tile-layout cache
        tq.tq_decode_attention_ex(st.desc, cache.ptrs, q, sl, 8, out, cache.workspace, None, None, 1, 1)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    big = torch.empty(128 + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError) as e:          # output not 16-byte aligned
        tq.tq_decode_attention(st.desc, cache.ptrs, q, sl, 8, big[1:129].view(1, 1, 128), cache.workspace)
    assert e.value.status == tq.TQ_ERR_INVALID_ARG


# --------------------------------------------------------------------------
# full sizes, in the launch configuration the benchmark times (automatic plan)
FULL = {
    "llama8b": (W.llama8b_decode(), [(0, 0), (13, 5), (31, 7)]),
    "block32_tq3": (W.block32(3), [(0, 0), (5, 3), (7, 7)]),
    "block32_tq4": (W.block32(4), [(0, 0), (7, 7)]),
    "so4_2k": (W.so4_wht(seq_len=2048), [(0, 0), (0, 3)]),
    "so4_8k": (W.so4_wht(seq_len=8192), [(0, 1), (0, 2)]),
    "so4_32k": (W.so4_wht(seq_len=32768), [(0, 0), (0, 3)]),
    "mixed_131k": (W.mixed_rate_long(131072), [(0, 0), (0, 1)]),
    "mixed_524k": (W.mixed_rate_long(524288), [(0, 1)]),
    "mixed_tight_131k": (W.mixed_rate_long(131072).with_(tight_k=True), [(0, 0)]),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(tq, name):
    wl, pairs = FULL[name]
    T, B = wl.seq_len, wl.batch
    inp = W.make_inputs(wl)
    st = make_setup(tq, wl, inp, T)
    cache = tq.PackedKVCache(st.desc, st.blob)
    K = to_torch_input(torch, inp.K, wl.in_dtype)
    V = to_torch_input(torch, inp.V, wl.in_dtype)
    cache.append(K, V, torch.zeros(B, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    del K, V
    # write side on the sampled pairs
    encs = {}
    bad = tot = 0
    for (b, h) in pairs:
        ek = oracle_encode(st, "k", b, h)
        ev = oracle_encode(st, "v", b, h)
        for enc, which in ((ek, "k"), (ev, "v")):
            rec = pair_records(cache, which, b, h, st)[:T]
            nb, n, _, _, ok = compare_codes(rec, enc, st.specs[h][0 if which == "k" else 1])
            assert ok
            bad += nb
            tot += n
        encs[(b, h)] = (ek, ev)
    assert bad / tot <= MAX_MISMATCH_FRAC
    # read side: the sampled pairs carry the oracle's records
    for (b, h), (ek, ev) in encs.items():
        put_pair(torch, cache, "k", b, h, ek.codes, ek.norms, st=st)
        put_pair(torch, cache, "v", b, h, ev.codes, ev.norms, st=st)
    q = to_torch_input(torch, inp.q, wl.in_dtype)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    _check_decode(tq, st, cache, encs, q, sl, T, -1, 0, pairs=pairs)
    assert int(cache.status.item()) == 0
