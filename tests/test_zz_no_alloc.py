"""GPU test of tq_decode_attention_noalloc, the decode entry point for callers
that cannot allocate device memory (code running inside another framework's
memory pool, plugins handed only their input and output buffers, paths where
an allocation would synchronise the device).  Its split-K scratch is a fixed
array in the library's device image instead of a caller workspace.

It is called through the C ABI and compared with tq_decode_attention (the
entry point that takes a workspace) and with the fp64 oracle on the same packed
cache, on two calls in a row, with a call on a different cache shape in between
so that the shared array holds another call's leftovers.  This file is
collected last on purpose."""
import numpy as np
import pytest

import workloads as W
from gpu_harness import ATT_TOL, att_error, make_setup, oracle_attention, oracle_encode, put_pair, to_torch_input

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


def _cache(tq, wl, B, T):
    wl = wl.with_(batch=B)
    inp = W.make_inputs(wl, seq_len=T, seq_lens=W.ragged_lengths(B, T, 5) if B > 1 else None)
    st = make_setup(tq, wl, inp, T)
    cache = tq.PackedKVCache(st.desc, st.blob)
    cache.append(to_torch_input(torch, inp.K, wl.in_dtype), to_torch_input(torch, inp.V, wl.in_dtype),
                 torch.zeros(B, dtype=torch.int32, device="cuda"))
    q = to_torch_input(torch, inp.q, wl.in_dtype)
    sl = torch.from_numpy(inp.seq_lens).cuda()
    # the oracle's records in the device cache, so that the oracle's attention on
    # them is the reference
    encs = {}
    for b in range(B):
        for h in range(wl.n_kv_heads):
            ek, ev = oracle_encode(st, "k", b, h), oracle_encode(st, "v", b, h)
            put_pair(torch, cache, "k", b, h, ek.codes, ek.norms, st=st)
            put_pair(torch, cache, "v", b, h, ev.codes, ev.norms, st=st)
            encs[(b, h)] = (ek, ev)
    cache.encs = encs
    return st, cache, q, sl


def _vs_oracle(st, cache, out, seq_lens):
    o = out.cpu().numpy()
    G = st.wl.group
    for (b, h), (ek, ev) in cache.encs.items():
        ref = oracle_attention(st, ek, ev, b, h, int(seq_lens[b]))
        err, scale = att_error(o[b, h * G:(h + 1) * G], ref)
        assert err <= ATT_TOL * scale, (b, h, err, scale)


def _close(a, ref):
    err = (a.double() - ref.double()).abs().max().item()
    scale = ref.double().abs().max().item()
    assert err <= ATT_TOL * scale, (err, scale)


def test_noalloc_matches_workspace_entry_point(tq):
    T1, T2 = 333, 600
    st1, c1, q1, l1 = _cache(tq, W.llama8b_decode(), 3, T1)
    st2, c2, q2, l2 = _cache(tq, W.so4_wht(), 1, T2)
    # both plans publish partials (several splits, or 0: the stream-K partition)
    assert tq.tq_decode_plan(st1.desc, T1)[0] != 1 and tq.tq_decode_plan(st2.desc, T2)[0] != 1
    ref1 = torch.empty(q1.shape, dtype=torch.float32, device="cuda")
    ref2 = torch.empty(q2.shape, dtype=torch.float32, device="cuda")
    tq.tq_decode_attention(st1.desc, c1.ptrs, q1, l1, T1, ref1, c1.workspace, c1.status)
    tq.tq_decode_attention(st2.desc, c2.ptrs, q2, l2, T2, ref2, c2.workspace, c2.status)
    outs = []
    for _ in range(2):
        o1 = torch.full(q1.shape, float("nan"), dtype=torch.float32, device="cuda")
        o2 = torch.full(q2.shape, float("nan"), dtype=torch.float32, device="cuda")
        tq.tq_decode_attention_noalloc(st1.desc, c1.ptrs, q1, l1, T1, o1, c1.status)
        tq.tq_decode_attention_noalloc(st2.desc, c2.ptrs, q2, l2, T2, o2, c2.status)
        outs.append((o1, o2))
    torch.cuda.synchronize()
    for o1, o2 in outs:
        _close(o1, ref1)
        _close(o2, ref2)
        _vs_oracle(st1, c1, o1, l1.cpu().numpy())
        _vs_oracle(st2, c2, o2, l2.cpu().numpy())
    assert int(c1.status.item()) == 0 and int(c2.status.item()) == 0


def test_noalloc_rejects_plans_beyond_the_fixed_scratch(tq):
    # 75 x 8 (batch, KV head) pairs at 16 query heads per KV head need two
    # splits of partials, about 10 MB: more than the fixed array holds.
    wl = W.llama8b_decode().with_(n_q_heads=128)
    B, T = 75, 64
    inp = W.make_inputs(wl.with_(batch=B), seq_len=T)
    st = make_setup(tq, wl.with_(batch=B), inp, 128)
    splits = tq.tq_decode_plan(st.desc, 128)[0]
    assert tq.tq_decode_workspace_bytes(st.desc, splits) > tq.tq_decode_noalloc_max_scratch_bytes()
    cache = tq.PackedKVCache(st.desc, st.blob, max_splits=1)
    q = to_torch_input(torch, inp.q, wl.in_dtype)
    sl = torch.full((B,), T, dtype=torch.int32, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention_noalloc(st.desc, cache.ptrs, q, sl, 128, out)
    assert e.value.status == tq.TQ_ERR_WORKSPACE
