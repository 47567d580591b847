"""CPU tests of the C ABI: the shared library loads, exports every entry point
declared in include/tq.h, and its host-side functions (Lloyd-Max solver, block
energy, greedy allocation, descriptor) agree with the fp64 oracle.  No GPU call
is made here."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle import tq_oracle as O


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tq_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tq_codebook", "tq_quantize_append", "tq_decode_attention", "tq_block_bit_alloc"):
        assert n in names


def test_every_declared_symbol_is_exported(tqlib):
    h = tqlib.lib()
    missing = [n for n in declared_functions() if not hasattr(h, n)]
    assert not missing, missing


def test_status_strings(tqlib):
    assert tqlib.tq_status_string(0) == "TQ_OK"
    assert tqlib.tq_status_string(5) == "TQ_ERR_WORKSPACE"
    assert tqlib.tq_status_string(99) == "TQ_ERR_UNKNOWN"


@pytest.mark.parametrize("d,bits", [(128, 3), (128, 4), (32, 3), (32, 4), (24, 1), (18, 2), (20, 3), (66, 4),
                                    (2, 4), (3, 2), (128, 1), (128, 2)])
def test_codebook_matches_oracle(tqlib, d, bits):
    c, b = tqlib.tq_codebook(d, bits)
    cb = O.codebook(d, bits)
    np.testing.assert_array_equal(c, cb.centroids.astype(np.float32))
    np.testing.assert_array_equal(b, cb.boundaries.astype(np.float32))


def test_codebook_invalid_args(tqlib):
    for d, bits in ((1, 3), (128, 0), (128, 5), (5000, 3)):
        with pytest.raises(tqlib.TQError) as e:
            tqlib.tq_codebook(d, bits)
        assert e.value.status == tqlib.TQ_ERR_INVALID_ARG


def test_block_energy_matches_oracle(tqlib):
    rng = np.random.default_rng(0)
    q = rng.standard_normal((64, 8, 128)).astype(np.float32)
    k = (rng.standard_normal((64, 128)) * 3).astype(np.float32)
    np.testing.assert_allclose(tqlib.tq_block_energy(q, k), O.block_energy(q, k), rtol=1e-13)


@pytest.mark.parametrize("seed", range(25))
def test_bit_alloc_matches_oracle(tqlib, seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 80))
    bmin = int(rng.integers(0, 3))
    bmax = int(rng.integers(bmin, 6))
    B = int(rng.integers(L * bmin, L * bmax + 1))
    s = rng.lognormal(0, 3, size=L)
    if seed % 4 == 0:
        s = np.round(s)          # exact ties
    np.testing.assert_array_equal(tqlib.tq_block_bit_alloc(s, bmin, bmax, B), O.greedy_bit_alloc(s, bmin, bmax, B))


def test_bit_alloc_infeasible(tqlib):
    with pytest.raises(tqlib.TQError):
        tqlib.tq_block_bit_alloc(np.ones(4), 1, 4, 3)
    with pytest.raises(tqlib.TQError):
        tqlib.tq_block_bit_alloc(np.ones(4), 1, 4, 17)
    with pytest.raises(tqlib.TQError):
        tqlib.tq_block_bit_alloc(np.array([1.0, np.nan]), 1, 4, 4)


def test_desc_sizes(tqlib):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 32, 8, 32, 8192, tq.TQ_ROT_WHT128, 3, 3, tq.TQ_F16)
    assert (d.group, d.k_code_bytes, d.v_code_bytes, d.k_norm_slots, d.norm_bytes) == (4, 48, 48, 1, 2)
    assert tq.tq_cache_bytes(d, tq.TQ_PART_K_CODES) == 32 * 8 * 8192 * 48
    assert tq.tq_cache_bytes(d, tq.TQ_PART_V_NORMS) == 32 * 8 * 8192 * 2
    d = tq.tq_cache_desc_init(128, 32, 8, 8, 8192, tq.TQ_ROT_WHT32, 4, 4, tq.TQ_F16)
    assert (d.k_code_bytes, d.k_norm_slots, d.v_norm_slots) == (64, 4, 4)
    # 72 B per block-32 TQ4 vector (64 B codes + 4 fp16 norms)
    assert d.k_code_bytes + d.k_norm_slots * d.norm_bytes == 72
    d = tq.tq_cache_desc_init(128, 16, 2, 1, 1024, tq.TQ_ROT_WHT128, 0, 3, tq.TQ_F16, 1)
    assert (d.k_code_bytes, d.k_norm_slots, d.v_code_bytes, d.v_norm_slots) == (64, 4, 48, 1)
    assert d.params_bytes == 2 * 3200 + 2 * 128 * 128 * 4


@pytest.mark.parametrize("args,status", [
    ((64, 32, 8, 1, 16, 0, 3, 3, 1), 2),      # head_dim != 128
    ((128, 30, 8, 1, 16, 0, 3, 3, 1), 1),     # n_q not a multiple of n_kv
    ((128, 32, 8, 0, 16, 0, 3, 3, 1), 1),     # batch 0
    ((128, 32, 8, 1, 16, 7, 3, 3, 1), 1),     # bad rotation
    ((128, 32, 8, 1, 16, 0, 2, 2, 1), 2),     # 2-bit V codes not built
    ((128, 32, 8, 1, 16, 1, 2, 3, 1), 2),     # two-stage keys with 32-wide blocks
    ((128, 32, 8, 1, 16, 0, 5, 3, 1), 2),     # 5-bit keys
    ((128, 32, 8, 1, 16, 0, 3, 4, 1), 2),     # K and V widths differ
    ((128, 64, 2, 1, 16, 0, 3, 3, 1), 2),     # group 32 > 16
    ((128, 32, 8, 1, 16, 0, 3, 3, 2), 1),     # bf16 norms
])
def test_desc_errors(tqlib, args, status):
    with pytest.raises(tqlib.TQError) as e:
        tqlib.tq_cache_desc_init(*args)
    assert e.value.status == status


def test_params_blob_contents(tqlib):
    tq = tqlib
    rng = np.random.default_rng(1)
    d = tq.tq_cache_desc_init(128, 4, 2, 1, 64, tq.TQ_ROT_WHT128, 0, 3, tq.TQ_F16, 1)
    signs = np.where(rng.random((2, 128)) < 0.5, -1.0, 1.0).astype(np.float32)
    bb = rng.integers(1, 5, size=(2, 64)).astype(np.int32)
    mats = []
    for h in range(2):
        for b, cs in O.group_layout(bb[h]):
            a = rng.standard_normal((cs.size, cs.size))
            qm, r = np.linalg.qr(a)
            mats.append((qm * np.sign(np.diag(r))).astype(np.float32).ravel())
    blob = tq.tq_params_build(d, signs=signs, k_block_bits=bb, k_group_mats=np.concatenate(mats))
    assert blob.size == d.params_bytes
    rec = blob[:3200]
    np.testing.assert_array_equal(rec[:512].view(np.float32), signs[0])
    starts = rec[1536:1556].view(np.int32)
    lay = O.group_layout(bb[0])
    want = [0]
    for b in range(1, 5):
        want.append(want[-1] + sum(cs.size for bb_, cs in lay if bb_ == b))
    np.testing.assert_array_equal(starts, want)
    # missing inputs are argument errors: in the binding, and in the library
    with pytest.raises(ValueError):
        tq.tq_params_build(d, signs=signs)
    out = np.zeros(int(d.params_bytes), np.uint8)
    assert tq.lib().tq_params_build(ctypes.byref(d), signs.ctypes.data, None, None, None,
                                    out.ctypes.data) == tq.TQ_ERR_INVALID_ARG


def test_decode_plan_host_only(tqlib):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 32, 8, 32, 8192, tq.TQ_ROT_WHT128, 3, 3, tq.TQ_F16)
    assert d.layout == tq.TQ_LAYOUT_TILE16 and d.t_alloc == 8192
    sp, vm = tq.tq_decode_plan(d, 8192)
    # tensor-core path: 131072 tiles over one wave of persistent CTAs (2 per SM)
    assert (sp, vm) == (304, tq.TQ_VMODE_TENSOR)
    with pytest.raises(tq.TQError) as e:   # no CUDA-core kernel reads the tile layout
        tq.tq_decode_plan(d, 8192, tq.TQ_VMODE_DIM_PARALLEL)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    # any capacity: the tile layout pads it to whole tiles
    d2 = tq.tq_cache_desc_init(128, 32, 8, 32, 8190, tq.TQ_ROT_WHT128, 3, 3, tq.TQ_F16)
    assert d2.layout == tq.TQ_LAYOUT_TILE16 and d2.t_alloc == 8192
    assert tq.tq_cache_bytes(d2, tq.TQ_PART_K_CODES) == 32 * 8 * 8192 * 48
    assert tq.tq_cache_bytes(d2, tq.TQ_PART_V_NORMS) == 32 * 8 * 8192 * 2
    assert tq.tq_decode_plan(d2, 8190) == (304, tq.TQ_VMODE_TENSOR)
    sp, vm = tq.tq_decode_plan(d, 100)
    assert vm == tq.TQ_VMODE_TENSOR and sp == 224                       # 1792 tiles, 8 per CTA (one a warp)
    assert tq.tq_decode_plan(d, 100, tq.TQ_VMODE_TENSOR, 7) == (7, tq.TQ_VMODE_TENSOR)
    # natural layout (16 query heads per KV head): dimension-parallel at every
    # length (the measured crossover is 0)
    d3 = tq.tq_cache_desc_init(128, 32, 2, 32, 8190, tq.TQ_ROT_WHT128, 3, 3, tq.TQ_F16)
    assert d3.layout == tq.TQ_LAYOUT_NATURAL and d3.t_alloc == 8190
    sp, vm = tq.tq_decode_plan(d3, 100)
    assert vm == tq.TQ_VMODE_DIM_PARALLEL and sp <= 2
    assert tq.tq_decode_plan(d3, 1)[1] == tq.TQ_VMODE_DIM_PARALLEL
    sp, vm = tq.tq_decode_plan(d3, 8190)
    assert vm == tq.TQ_VMODE_DIM_PARALLEL and 1 <= sp <= tq.TQ_MAX_SPLITS
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_plan(d3, 8190, tq.TQ_VMODE_TENSOR)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    with pytest.raises(tq.TQError):
        tq.tq_decode_plan(d, 0)
    with pytest.raises(tq.TQError):
        tq.tq_decode_plan(d, 9000)


def test_prefix_workspace_and_argument_checks(tqlib):
    """Host-side behaviour of the prefix entry point: workspace sizes grow with the
    unquantised length and hold the packed decode's; bad arguments are refused
    before any device work (every call below fails its checks)."""
    d = tqlib.tq_cache_desc_init(128, 32, 8, 4, 1000, 0, 3, 3, 1)
    w0 = tqlib.tq_decode_prefix_workspace_bytes(d, 0)
    w1 = tqlib.tq_decode_prefix_workspace_bytes(d, 4096)
    assert w0 >= tqlib.tq_decode_workspace_bytes(d, 1) and w1 > w0
    assert tqlib.tq_decode_prefix_workspace_bytes(d, -1) == 0
    h = tqlib.lib()
    c = tqlib.tq_cache_ptrs(16, 16, 16, 16, 16)
    w50 = tqlib.tq_decode_prefix_workspace_bytes(d, 50)
    args = dict(q=256, qdt=tqlib.TQ_F16, sl=256, msl=10, kp=256, vp=256, pdt=tqlib.TQ_F16, cap=100, pl=256, mpl=50,
                out=256, ws=256, wsb=w50)

    def call(**kw):
        a = dict(args, **kw)
        return h.tq_decode_attention_prefix(ctypes.byref(d), ctypes.byref(c), a["q"], a["qdt"], a["sl"], a["msl"],
                                            a["kp"], a["vp"], a["pdt"], a["cap"], a["pl"], a["mpl"], a["out"], a["ws"],
                                            a["wsb"], None, None)
    assert call(out=0) == tqlib.TQ_ERR_INVALID_ARG
    assert call(pl=0) == tqlib.TQ_ERR_INVALID_ARG
    assert call(pdt=7) == tqlib.TQ_ERR_INVALID_ARG
    assert call(mpl=101) == tqlib.TQ_ERR_INVALID_ARG          # above the capacity
    assert call(kp=0) == tqlib.TQ_ERR_INVALID_ARG             # unquantised tokens without K
    assert call(kp=258) == tqlib.TQ_ERR_INVALID_ARG           # misaligned
    assert call(wsb=w50 - 1) == tqlib.TQ_ERR_WORKSPACE
    assert call(ws=0) == tqlib.TQ_ERR_WORKSPACE


@pytest.mark.parametrize("fmt", ["g16", "wht32_f32", "mixed_f32"])
def test_crossover_per_format(tqlib, fmt, monkeypatch):
    tq = tqlib
    """Natural-layout formats: dimension-parallel from length 1 (measured crossover
    0); TQ_V_CROSSOVER = X moves the switch to X (token-parallel at X - 1,
    dimension-parallel at X)."""
    if fmt == "g16":
        d = tq.tq_cache_desc_init(128, 32, 2, 4, 4096, tq.TQ_ROT_WHT128, 3, 3, tq.TQ_F16)
    elif fmt == "wht32_f32":
        d = tq.tq_cache_desc_init(128, 32, 8, 4, 4096, tq.TQ_ROT_WHT32, 3, 3, tq.TQ_F32)
    else:
        d = tq.tq_cache_desc_init(128, 16, 2, 1, 4096, tq.TQ_ROT_WHT128, 0, 3, tq.TQ_F32, 1)
    assert d.layout == tq.TQ_LAYOUT_NATURAL
    monkeypatch.delenv("TQ_V_CROSSOVER", raising=False)
    for T in (1, 511, 512, 4096):
        assert tq.tq_decode_plan(d, T)[1] == tq.TQ_VMODE_DIM_PARALLEL
    monkeypatch.setenv("TQ_V_CROSSOVER", "512")
    assert tq.tq_decode_plan(d, 511)[1] == tq.TQ_VMODE_TOKEN_PARALLEL
    assert tq.tq_decode_plan(d, 512)[1] == tq.TQ_VMODE_DIM_PARALLEL


def test_block_energy_shape_check(tqlib):
    """The binding refuses calibration keys whose token count differs from the
    queries' (the C function reads T rows of both)."""
    q = np.zeros((16, 4, 128), dtype=np.float32)
    with pytest.raises(ValueError):
        tqlib.tq_block_energy(q, np.zeros((8, 128), dtype=np.float32))


def test_zip_sizes_and_argument_checks(tqlib):
    """ZipFusion host side: a 4096-byte slot and 8 metadata bytes per 16-token page;
    capacities not a multiple of 16 and more than 8 query heads per KV head are
    refused before any device work."""
    assert tqlib.tq_zip_pool_bytes(2, 8, 64) == 2 * 8 * 4 * 4096
    assert tqlib.tq_zip_meta_bytes(2, 8, 64) == 2 * 8 * 4 * 8
    assert tqlib.tq_zip_pool_bytes(2, 8, 65) == 0
    assert tqlib.tq_zip_workspace_bytes(2, 32, 8, 64) > 0
    assert tqlib.tq_zip_workspace_bytes(2, 32, 2, 64) == 0          # 16 heads per KV head
    h = tqlib.lib()
    ws = tqlib.tq_zip_workspace_bytes(2, 32, 8, 64)
    args = [256, tqlib.TQ_BF16, 2, 32, 8, 64, 256, 256, 256, 256, 256, 64, 256, 256, ws, None, None]

    def call(i, v):
        a = list(args)
        a[i] = v
        return h.tq_zip_decode_attention(*a)
    assert call(5, 65) == tqlib.TQ_ERR_INVALID_ARG                   # capacity not whole pages
    assert call(11, 65) == tqlib.TQ_ERR_INVALID_ARG                  # max_seq_len above capacity
    assert call(4, 2) == tqlib.TQ_ERR_UNSUPPORTED                    # 16 query heads per KV head
    assert call(14, ws - 1) == tqlib.TQ_ERR_WORKSPACE
    assert call(6, 128) == tqlib.TQ_ERR_INVALID_ARG                  # pool not 256-byte aligned
    assert h.tq_zip_store(256, 256, 2, 8, 0, 64, 256, 256, 256, 256, 256, None, None) == tqlib.TQ_ERR_INVALID_ARG
