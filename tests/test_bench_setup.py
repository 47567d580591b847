"""Host side of `bench.py` on CPU: the library setup of every workload the
benchmark times (descriptor and blob through the library alone) and the
per-step byte counts the roofline divides by.  No GPU call."""
import numpy as np
import pytest

import bench
import workloads as W


def _cases():
    return [
        W.llama8b_decode(seq_len=64, batch=2),
        W.block32(3, seq_len=64, batch=2),
        W.so4_wht(seq_len=64),
        W.mixed_rate_long(seq_len=600),
        W.mixed_rate_long(seq_len=600).with_(tight_k=True),
        W.mixed_rate_long(seq_len=600).with_(norm_dtype=W.F32),
        W.llama8b_decode(seq_len=64, batch=2).with_(n_kv_heads=2),
        W.two_stage_keys(1, seq_len=64, batch=2),
        W.two_stage_keys(2, seq_len=64, batch=2),
    ]


@pytest.mark.parametrize("i", range(len(_cases())))
def test_library_setup(tqlib, i):
    wl = _cases()[i]
    inp = W.make_inputs(wl, seq_len=wl.seq_len)
    desc, blob = bench.library_setup(tqlib, wl, inp, wl.seq_len)
    assert blob.size == desc.params_bytes
    if wl.mixed_k:
        assert desc.k_mixed == (2 if wl.tight_k else 1)
        assert desc.k_code_bytes == (16 * wl.avg_bits if wl.tight_k else 64)
    elif wl.k_bits in (1, 2):
        assert desc.k_code_bytes == 16 * wl.k_bits and desc.k_norm_slots == 2
    else:
        assert desc.k_code_bytes == (48 if wl.k_bits == 3 else 64)
    b = bench.step_bytes(wl, wl.seq_len, desc)
    per = desc.k_code_bytes + desc.v_code_bytes + (desc.k_norm_slots + desc.v_norm_slots) * desc.norm_bytes
    assert b["decode"] >= wl.batch * wl.n_kv_heads * wl.seq_len * per
    assert b["step"] == b["decode"] + b["append"]


def test_bench_workload_bytes():
    """The bench line's algorithmic bytes: llama8b, batch 32, T = 8192, 3-bit K and V
    with fp16 norms: 100 B per (token, KV head), plus q (bf16) and out (fp32)."""
    class D:
        k_code_bytes = v_code_bytes = 48
        k_norm_slots = v_norm_slots = 1
        norm_bytes = 2
    wl = W.llama8b_decode()
    b = bench.step_bytes(wl, 8192, D)
    assert b["decode"] == 32 * 8 * 8192 * 100 + 32 * 32 * 128 * (2 + 4) == 210501632
