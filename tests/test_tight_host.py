"""CPU tests of the host side of tight mixed-rate key records (each code at its
group's width, concatenated; k_mixed = 2)  [Block-GTQ, packed cache]:
descriptor sizes and layout, the budget check of the parameter blob, the plan.
No GPU call."""
import numpy as np
import pytest

from oracle import tq_oracle as O


@pytest.mark.parametrize("avg,nbytes", [(2, 32), (3, 48)])
def test_desc_sizes(tqlib, avg, nbytes):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 16, 2, 1, 1000, tq.TQ_ROT_WHT128, avg, 3, tq.TQ_F16, 2)
    assert d.layout == tq.TQ_LAYOUT_NATURAL and d.t_alloc == 1000
    assert (d.k_mixed, d.k_bits, d.k_code_bytes, d.k_norm_slots) == (2, avg, nbytes, 4)
    assert d.params_bytes == 2 * 3200 + 2 * 128 * 128 * 4
    # the nibble record of the same allocation: 64 B
    n = tq.tq_cache_desc_init(128, 16, 2, 1, 1000, tq.TQ_ROT_WHT128, 0, 3, tq.TQ_F16, 1)
    assert n.k_code_bytes == 64 and n.layout == tq.TQ_LAYOUT_TILE16


@pytest.mark.parametrize("args,status", [
    ((128, 16, 2, 1, 16, 0, 4, 3, 1, 2), 2),    # 4 bits on average: the nibble record already
    ((128, 16, 2, 1, 16, 0, 1, 3, 1, 2), 2),
    ((128, 16, 2, 1, 16, 1, 3, 3, 1, 2), 2),    # 32-wide blocks
    ((128, 16, 2, 1, 16, 0, 3, 3, 1, 3), 1),    # no k_mixed 3
])
def test_desc_errors(tqlib, args, status):
    with pytest.raises(tqlib.TQError) as e:
        tqlib.tq_cache_desc_init(*args)
    assert e.value.status == status


def _mats(bb, rng):
    flat = []
    for b, cs in O.group_layout(bb):
        qm, r = np.linalg.qr(rng.standard_normal((cs.size, cs.size)))
        flat.append((qm * np.sign(np.diag(r))).astype(np.float32).ravel())
    return np.concatenate(flat)


def test_params_budget(tqlib):
    """Every head's allocation must fill the record exactly: 3 * 64 block bits for
    48-byte records."""
    tq = tqlib
    rng = np.random.default_rng(4)
    d = tq.tq_cache_desc_init(128, 4, 1, 1, 64, tq.TQ_ROT_WHT128, 3, 3, tq.TQ_F16, 2)
    signs = np.ones((1, 128), np.float32)
    bb = O.greedy_bit_alloc(rng.lognormal(0, 2, 64), 1, 4, 3 * 64).astype(np.int32)[None]
    blob = tq.tq_params_build(d, signs=signs, k_block_bits=bb, k_group_mats=_mats(bb[0], rng))
    assert blob.size == d.params_bytes
    short = bb.copy()
    short[0, np.argmax(short[0])] -= 1          # 191 bits: does not fill the record
    with pytest.raises(tq.TQError) as e:
        tq.tq_params_build(d, signs=signs, k_block_bits=short, k_group_mats=_mats(short[0], rng))
    assert e.value.status == tq.TQ_ERR_INVALID_ARG


def test_plan_is_cuda_core(tqlib):
    tq = tqlib
    d = tq.tq_cache_desc_init(128, 16, 2, 1, 131072, tq.TQ_ROT_WHT128, 3, 3, tq.TQ_F16, 2)
    sp, vm = tq.tq_decode_plan(d, 131072)
    assert vm == tq.TQ_VMODE_DIM_PARALLEL and 1 <= sp <= 128
    with pytest.raises(tq.TQError):
        tq.tq_decode_plan(d, 131072, tq.TQ_VMODE_TENSOR)
