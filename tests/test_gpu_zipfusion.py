"""GPU parity of the ZipFusion store and attention (tq_zip_store,
tq_zip_decode_attention) against the oracle: every stored block restores
bit-exactly through the oracle's decoder and compresses exactly when the oracle
says it can (b/2 recorded); attention on the pages equals fp64 attention on the
original bf16 values (the store is lossless) within 2e-3 max|o|; ragged lengths
with partial pages, 1 / 4 / 8 query heads per KV head, many sections; a page
offset outside the pool is flagged, not followed."""
import numpy as np
import pytest

import workloads as W
from gpu_harness import ATT_TOL, att_error, to_torch_input
from oracle import tq_oracle as O

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


def _store(tq, wl, B, T, cap, lens):
    inp = W.make_inputs(wl.with_(batch=B), seq_len=T)
    assert wl.in_dtype == W.BF16
    z = tq.ZipKVCache(B, wl.n_q_heads, wl.n_kv_heads, cap)
    K = to_torch_input(torch, inp.K, W.BF16)
    V = to_torch_input(torch, inp.V, W.BF16)
    z.store(K, V, torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda())
    torch.cuda.synchronize()
    return inp, z


def _pages_back(z, which, b, h, n_pages):
    """[n_pages][4] (mark, restored block bits) read back through the oracle."""
    pool = (z.k_pool if which == "k" else z.v_pool).cpu().numpy()
    meta = (z.k_meta if which == "k" else z.v_meta).cpu().numpy().view(np.uint32).reshape(-1, 2)
    pages = z.t_capacity // 16
    out = []
    for p in range(n_pages):
        off, marks = meta[(b * z.n_kv_heads + h) * pages + p]
        pos = int(off) * 256
        row = []
        for j in range(4):
            mk = (int(marks) >> (8 * j)) & 0xFF
            if mk == 0xFF:
                row.append((mk, pool[pos:pos + 1024].view(np.uint16).copy()))
                pos += 1024
            else:
                row.append((mk, O.zf_decode_block(mk, pool[pos:pos + 512], pool[pos + 512:pos + 768])))
                pos += 768
        out.append(row)
    return out


@pytest.mark.parametrize("name", ["llama8b", "so4"])
def test_store_is_lossless_and_compresses_as_the_oracle(tq, name):
    wl = W.llama8b_decode() if name == "llama8b" else W.so4_wht()
    B, T = 2, 333
    lens = [T, 200]
    inp, z = _store(tq, wl, B, T, 352, lens)
    assert int(z.status.item()) == 0
    n_comp = n_all = 0
    for b in range(B):
        for h in range(wl.n_kv_heads):
            for which, src in (("k", inp.K), ("v", inp.V)):
                n_pages = (lens[b] + 15) // 16
                for p, row in enumerate(_pages_back(z, which, b, h, n_pages)):
                    page = np.zeros((16, 128), dtype=np.uint16)
                    n = min(16, lens[b] - 16 * p)
                    page[:n] = src[b, 16 * p:16 * p + n, h]
                    blocks = O.zf_page_blocks(page, which)
                    for j, (mk, bits) in enumerate(row):
                        np.testing.assert_array_equal(bits, blocks[j])
                        if n == 16 and O.zf_compressible(blocks[j]):
                            assert mk == O.zf_base(blocks[j]) // 2
                            n_comp += 1
                        else:
                            assert mk == 0xFF
                        n_all += 1
    assert 0 < n_comp < n_all   # the recipe's outlier channels leave some blocks raw


def _check_attention(tq, wl, B, T, cap, lens, max_seq=None):
    inp, z = _store(tq, wl, B, T, cap, lens)
    q = to_torch_input(torch, inp.q, W.BF16)
    sl = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    ms = max(lens) if max_seq is None else max_seq
    out = z.decode(q, sl, ms)
    torch.cuda.synchronize()
    clamped = max(lens) > ms
    assert int(z.status.item()) == (tq.TQ_DEV_SEQ_OVER_MAX if clamped else 0)
    o = out.cpu().numpy()
    G = wl.group
    errs, scales = [], []
    for b in range(B):
        for h in range(wl.n_kv_heads):
            qh = W.as_float64(inp.q[b, h * G:(h + 1) * G], W.BF16)
            L = min(lens[b], ms)
            ref = O.attend_exact(qh, W.as_float64(inp.K[b, :L, h], W.BF16), W.as_float64(inp.V[b, :L, h], W.BF16), L)
            e, s = att_error(o[b, h * G:(h + 1) * G], ref)
            errs.append(e)
            scales.append(s)
    assert max(errs) <= ATT_TOL * max(scales), (max(errs), max(scales))
    return z


@pytest.mark.parametrize("name", ["single", "llama8b", "so4"])
def test_attention_matches_oracle(tq, name):
    wl = {"single": W.llama8b_decode().with_(n_q_heads=8, n_kv_heads=8), "llama8b": W.llama8b_decode(),
          "so4": W.so4_wht()}[name]
    _check_attention(tq, wl, 3, 333, 352, [333, 1, 170])


def test_attention_many_sections(tq):
    wl = W.so4_wht()
    _check_attention(tq, wl, 1, 4000, 4000, [4000])          # several sections per (batch, KV head)
    _check_attention(tq, wl, 2, 600, 608, [600, 599], max_seq=512)   # clamped to max_seq_len


def test_bad_page_offset_is_flagged(tq):
    wl = W.llama8b_decode()
    inp, z = _store(tq, wl, 1, 64, 64, [64])
    meta = z.k_meta.view(torch.int32)
    meta[2] = 0x7FFFFFF0                      # page 1 of head 0: far outside the pool
    q = to_torch_input(torch, inp.q, W.BF16)
    z.decode(q, torch.tensor([64], dtype=torch.int32, device="cuda"), 64)
    torch.cuda.synchronize()
    assert int(z.status.item()) & tq.TQ_DEV_BAD_METADATA
