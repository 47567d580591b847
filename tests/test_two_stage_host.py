"""CPU tests of the host side of two-stage keys (a (b-1)-bit MSE code plus a 1-bit
QJL code, b = k_bits = 1 or 2)  [TQ-MNN §2.4]: descriptor sizes and layout, the
parameter blob (codebook, segments, the projection stored transposed), argument
checks in the binding and in the C library, and the host plan.  No GPU call."""
import ctypes

import numpy as np
import pytest

import workloads as W
from oracle import tq_oracle as O

PARAMS = 3200          # bytes of one KV head's parameter record
OFF_K_SEG_START, OFF_K_SEG_BITS, OFF_K_NSEG = 1536, 1556, 1572
OFF_K_CENT, OFF_K_BOUND, OFF_GCOORD = 1664, 1920, 2688


@pytest.mark.parametrize("k_bits,v_bits", [(1, 3), (2, 3), (2, 4), (1, 4)])
def test_desc_sizes(tqlib, k_bits, v_bits):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 32, 8, 4, 1000, tq.TQ_ROT_WHT128, k_bits, v_bits, tq.TQ_F16)
    assert d.layout == tq.TQ_LAYOUT_NATURAL and d.t_alloc == 1000
    assert (d.k_code_bytes, d.k_norm_slots) == (16 * k_bits, 2)
    assert d.k_code_bytes == O.qjl_record_bytes(k_bits - 1)
    assert (d.v_code_bytes, d.v_norm_slots) == (48 if v_bits == 3 else 64, 1)
    assert d.params_bytes == 8 * PARAMS + 8 * 128 * 128 * 4
    assert tq.tq_cache_bytes(d, tq.TQ_PART_K_CODES) == 4 * 8 * 1000 * 16 * k_bits
    assert tq.tq_cache_bytes(d, tq.TQ_PART_K_NORMS) == 4 * 8 * 1000 * 2 * 2
    d = tq.tq_cache_desc_init(128, 8, 8, 1, 64, tq.TQ_ROT_SO4_WHT128, k_bits, v_bits, tq.TQ_F32)
    assert d.layout == tq.TQ_LAYOUT_NATURAL and d.norm_bytes == 4


def test_desc_rejects(tqlib):
    tq = tqlib
    with pytest.raises(tq.TQError) as e:
        tq.tq_cache_desc_init(128, 32, 8, 1, 16, tq.TQ_ROT_WHT32, 2, 3, tq.TQ_F16)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    # with k_mixed the key width comes from the allocation: k_bits is ignored
    d = tq.tq_cache_desc_init(128, 16, 2, 1, 64, tq.TQ_ROT_WHT128, 2, 3, tq.TQ_F16, 1)
    assert d.k_mixed == 1 and d.k_code_bytes == 64 and d.k_norm_slots == 4


@pytest.mark.parametrize("k_bits", [1, 2])
def test_params_blob(tqlib, k_bits):
    tq = tqlib
    wl = W.two_stage_keys(k_bits).with_(n_q_heads=8, n_kv_heads=2, batch=1)
    d = tq.tq_cache_desc_init(128, 8, 2, 1, 64, wl.rot, k_bits, 3, wl.norm_dtype)
    rng = np.random.default_rng(2)
    signs = np.where(rng.random((2, 128)) < 0.5, -1.0, 1.0).astype(np.float32)
    S = np.stack([W.two_stage_projection(128, 0, h) for h in range(2)])
    blob = tq.tq_params_build(d, signs=signs, k_group_mats=S)
    assert blob.size == d.params_bytes
    for h in range(2):
        rec = blob[h * PARAMS:(h + 1) * PARAMS]
        assert rec[OFF_K_SEG_START:OFF_K_SEG_START + 20].view(np.int32).tolist() == [0, 128, 128, 128, 128]
        assert rec[OFF_K_SEG_BITS:OFF_K_SEG_BITS + 4].view(np.int32)[0] == k_bits - 1
        assert rec[OFF_K_NSEG:OFF_K_NSEG + 4].view(np.int32)[0] == 1
        cent = rec[OFF_K_CENT:OFF_K_CENT + 8].view(np.float32)
        bound = rec[OFF_K_BOUND:OFF_K_BOUND + 4].view(np.float32)
        if k_bits == 2:
            np.testing.assert_array_equal(cent, O.codebook(128, 1).centroids.astype(np.float32))
            assert bound[0] == 0.0
        else:
            assert not cent.any()
        np.testing.assert_array_equal(rec[OFF_GCOORD:PARAMS].view(np.int32), np.arange(128))
    # the projections follow the records, each stored transposed
    tail = blob[2 * PARAMS:].view(np.float32).reshape(2, 128, 128)
    for h in range(2):
        np.testing.assert_array_equal(tail[h], S[h].T)


def test_params_argument_checks(tqlib):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 8, 2, 1, 64, tq.TQ_ROT_WHT128, 2, 3, tq.TQ_F16)
    signs = np.ones((2, 128), np.float32)
    with pytest.raises(ValueError):
        tq.tq_params_build(d, signs=signs)                                 # projections missing
    with pytest.raises(ValueError):
        tq.tq_params_build(d, signs=signs, k_group_mats=np.zeros((1, 128, 128), np.float32))   # one head short
    with pytest.raises(ValueError):
        tq.tq_params_build(d, signs=np.ones((1, 128), np.float32), k_group_mats=np.zeros((2, 128, 128)))
    # the C library itself refuses a missing projection
    blob = np.zeros(int(d.params_bytes), np.uint8)
    st = tq.lib().tq_params_build(ctypes.byref(d), signs.ctypes.data, None, None, None, blob.ctypes.data)
    assert st == tq.TQ_ERR_INVALID_ARG


def test_mixed_rate_matrix_size_check(tqlib):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 4, 1, 1, 64, tq.TQ_ROT_WHT128, 0, 3, tq.TQ_F16, 1)
    bb = np.full((1, 64), 3, np.int32)
    with pytest.raises(ValueError):
        tq.tq_params_build(d, signs=np.ones((1, 128), np.float32), k_block_bits=bb,
                           k_group_mats=np.zeros(128 * 128 - 1, np.float32))
    blob = tq.tq_params_build(d, signs=np.ones((1, 128), np.float32), k_block_bits=bb,
                              k_group_mats=np.eye(128, dtype=np.float32))
    assert blob.size == d.params_bytes


def test_plan_is_cuda_core(tqlib):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 32, 8, 8, 8192, tq.TQ_ROT_WHT128, 2, 3, tq.TQ_F16)
    sp, vm = tq.tq_decode_plan(d, 8192)
    assert vm == tq.TQ_VMODE_DIM_PARALLEL and 1 <= sp <= 128
    assert tq.tq_decode_plan(d, 500, tq.TQ_VMODE_TOKEN_PARALLEL, 3) == (3, tq.TQ_VMODE_TOKEN_PARALLEL)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_plan(d, 8192, tq.TQ_VMODE_TENSOR)
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
