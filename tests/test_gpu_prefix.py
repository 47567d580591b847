"""GPU parity of decode attention over unquantised tokens plus the packed cache
(tq_decode_attention_prefix) against the oracle's attend_prefix_packed, on the
oracle's own records in the device cache: tile and natural layouts, ragged
packed and unquantised lengths (0 included), fp16 / bf16 / fp32 unquantised
inputs, packed-only and unquantised-only calls, one and several sections."""
import numpy as np
import pytest

import workloads as W
from gpu_harness import ATT_TOL, att_error, to_torch_input
from oracle import tq_oracle as O
from test_gpu_parity import SMALL, _encode_on_gpu, _upload_oracle_cache

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rotated_bit_kv_gb300 as m
    m.build()
    m.lib()
    return m


def _prefix_inputs(wl, B, P, dtype, seed):
    """Unquantised K, V [B][P][Hkv][128] (the append input layout) as stored, and
    their exact fp64 values."""
    rng = np.random.default_rng([seed, 0x5046])
    K = rng.standard_normal((B, P, wl.n_kv_heads, 128)).astype(np.float32) * 2.0
    V = rng.standard_normal((B, P, wl.n_kv_heads, 128)).astype(np.float32)
    if dtype == W.F16:
        K, V = K.astype(np.float16), V.astype(np.float16)
    elif dtype == W.BF16:
        K, V = W.f32_to_bf16_bits(K), W.f32_to_bf16_bits(V)
    return K, V, W.as_float64(K, dtype), W.as_float64(V, dtype)


def _run(tq, name, P, plens, seq_lens_fn, dtype=W.F16, max_seq=None, seed=0):
    B, T = SMALL[name]
    seq_lens = W.ragged_lengths(B, T, 3) if B > 1 else None
    st, cache = _encode_on_gpu(tq, name, B, T, seq_lens=seq_lens)
    encs = _upload_oracle_cache(tq, st, cache, B, T)
    wl = st.wl
    q = to_torch_input(torch, st.inp.q, wl.in_dtype)
    L = seq_lens_fn(st.inp.seq_lens.copy(), T)
    sl = torch.from_numpy(L.astype(np.int32)).cuda()
    Kp, Vp, K64, V64 = _prefix_inputs(wl, B, P, dtype, seed)
    kp, vp = to_torch_input(torch, Kp, dtype), to_torch_input(torch, Vp, dtype)
    pl = torch.from_numpy(np.asarray(plens, dtype=np.int32)).cuda()
    ms = int(L.max()) if max_seq is None else max_seq
    out = cache.decode_prefix(q, sl, ms, kp, vp, pl, P)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    o = out.cpu().numpy()
    G = wl.group
    errs, scales = [], []
    for (b, h), (ek, ev) in encs.items():
        ks, vs = st.specs[h]
        qh = W.as_float64(st.inp.q[b, h * G:(h + 1) * G], wl.in_dtype)
        n = int(plens[b])
        ref = O.attend_prefix_packed(qh, K64[b, :n, h], V64[b, :n, h], ek.idx, ek.norms.astype(np.float64), ks,
                                     ev.idx, ev.norms.astype(np.float64), vs, int(min(L[b], ms)))
        e, s = att_error(o[b, h * G:(h + 1) * G], ref)
        errs.append(e)
        scales.append(s)
    assert max(errs) <= ATT_TOL * max(scales), (max(errs), max(scales))
    return cache, out


def _plens(B, P):
    """Ragged unquantised lengths in [0, P], including 0 and P."""
    p = np.linspace(P, 0, B).round().astype(np.int32) if B > 1 else np.array([P], dtype=np.int32)
    return p


@pytest.mark.parametrize("name", ["tiny", "llama8b", "so4", "mixed", "llama8b_g16", "block32_f32", "mixed_tight"])
def test_prefix_plus_packed(tq, name):
    B, _ = SMALL[name]
    _run(tq, name, 300, _plens(B, 300), lambda L, T: L)


@pytest.mark.parametrize("dtype", [W.BF16, W.F32])
def test_prefix_dtypes(tq, dtype):
    B, _ = SMALL["llama8b"]
    _run(tq, "llama8b", 77, _plens(B, 77), lambda L, T: L, dtype=dtype)


@pytest.mark.parametrize("P", [1, 64, 5000])
def test_prefix_lengths_and_sections(tq, P):
    """One token, one section, and many sections (the partial merge)."""
    B, _ = SMALL["so4"]
    _run(tq, "so4", P, _plens(B, P), lambda L, T: L)


def test_prefix_only_and_packed_only(tq):
    B, T = SMALL["llama8b"]
    # no packed token at all (max_seq_len = 0: the cache is not read)
    _run(tq, "llama8b", 200, _plens(B, 200), lambda L, T: np.zeros_like(L), max_seq=0)
    # no unquantised token: equals the packed decode
    _run(tq, "llama8b", 16, np.zeros(B, dtype=np.int32), lambda L, T: L)


def test_empty_everything_gives_zero(tq):
    B, _ = SMALL["llama8b"]
    cache, out = _run(tq, "llama8b", 8, np.zeros(B, dtype=np.int32), lambda L, T: np.zeros_like(L))
    assert not out.any()
