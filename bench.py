#!/usr/bin/env python
"""Benchmark of one decode step of the rotation-quantised packed KV cache on
the Llama-3.1-8B-shaped decode workload: batch 32, 32 query heads, 8 KV heads,
head_dim 128, T = 8192 cached tokens per sequence, bf16 q/K/V, 3-bit K and V,
128-point sign-flipped WHT, fp16 norms.

A step is one pass of the whole hot path: quantise-and-append the new token's
K and V for every sequence (write side) and decode attention for every query
head over T tokens on the packed codes (read side).

Prints one JSON line.  `value` is the algorithmic HBM throughput of the step
(codes + norms read, q read, out written, appended bytes) in GB/s, summed over
ranks; `us_per_step` is the device time per step.  The roofline block reports
the decode kernel alone against the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  (N > 1 under torch.distributed.run: independent replicas, one per GPU)
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "packed 3-bit KV decode attention: µs/step and HBM GB/s as % of GB300 peak"
NREF = 8               # distinct (batch, KV head) pairs the oracle arm encodes
DTYPE = "f16*f16->f32" # tensor-core operands fp16, accumulation and softmax fp32
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(wl: W.Workload, T: int, desc) -> dict:
    B, Hkv, Hq, d = wl.batch, wl.n_kv_heads, wl.n_q_heads, wl.head_dim
    per_tok = desc.k_code_bytes + desc.v_code_bytes + (desc.k_norm_slots + desc.v_norm_slots) * desc.norm_bytes
    in_b = 4 if wl.in_dtype == W.F32 else 2
    decode = B * T * Hkv * per_tok + B * Hq * d * in_b + B * Hq * d * 4
    append = B * Hkv * 2 * d * in_b + B * Hkv * per_tok
    return {"decode": decode, "append": append, "step": decode + append}


def workload_name(wl, T):
    return (f"llama8b_decode: batch {wl.batch}, {wl.n_q_heads} q heads / {wl.n_kv_heads} KV heads, d=128, "
            f"T={T}, bf16 q/K/V, 3-bit K and V, 128-point sign-flipped WHT, fp16 norms")


class ClockSampler:
    """nvidia-smi samples during the timed region (started before, stopped after)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"tq_clocks_{os.getpid()}.csv")
        try:
            gpu_index = self._index_of(local_rank)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_index, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _index_of(local_rank: int) -> str:
        """nvidia-smi index of the CUDA device this rank uses, matched by UUID."""
        import torch
        uuid = str(torch.cuda.get_device_properties(local_rank).uuid)
        out = subprocess.run(["nvidia-smi", "--query-gpu=index,uuid", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout
        rows = [r.split(",") for r in out.strip().splitlines() if "," in r]
        for idx, u in rows:
            if uuid.replace("GPU-", "") in u:
                return idx.strip()
        return rows[0][0].strip() if len(rows) == 1 else str(local_rank)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("tq_decode.cu", "tq_decode_tile.cu", "tq_tile.cuh", "tq_mma.cuh", "tq_decode_common.cuh",
              "tq_device.cuh", "tq_internal.h"):
        with open(os.path.join(ROOT, "rotated_bit_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-launch DRAM bytes of the decode kernel from a committed ncu summary
    taken on the current kernel source (else None)."""
    d = os.path.join(ROOT, "profiles")
    want = kernel_source_hash()
    for f in sorted(os.listdir(d)) if os.path.isdir(d) else []:
        if not f.endswith(".md"):
            continue
        src, traffic = None, None
        for line in open(os.path.join(d, f)):
            if line.startswith("kernel_source_sha256_16:"):
                src = line.split(":", 1)[1].strip()
            if line.startswith("dram_bytes_per_launch:"):
                traffic = float(line.split(":", 1)[1].strip())
        if src == want and traffic is not None:
            return traffic
    return None


# ----------------------------------------------------------------------------
# CPU leg: the oracle as it stands, on a bounded sample of the same step
class OracleLeg:
    """The oracle as it stands, timed on a bounded sample of the step: for a few
    (batch, KV head) pairs, encode the new token's K and V and run attention
    over T cached tokens (the cache itself is encoded once, untimed)."""

    def __init__(self, wl, T, n_pairs):
        from gpu_harness import Setup, oracle_encode
        from oracle import tq_oracle as O
        self.O = O
        self.wl, self.T = wl.with_(batch=1), T
        self.inp = W.make_inputs(self.wl, seq_len=T)
        self.specs = O.head_specs(self.wl, self.inp)
        self.st = Setup(self.wl, self.inp, None, None, self.specs, None, None)
        self.heads = list(range(min(n_pairs, wl.n_kv_heads)))
        self.encs = {h: (oracle_encode(self.st, "k", 0, h), oracle_encode(self.st, "v", 0, h)) for h in self.heads}

    def run_pairs(self, n_pairs):
        """Seconds for n_pairs pair-steps (encode the new K and V token, attend over T),
        cycling over the encoded pairs."""
        from gpu_harness import oracle_attention
        O, wl, T, inp = self.O, self.wl, self.T, self.inp
        t0 = time.perf_counter()
        for i in range(n_pairs):
            h = self.heads[i % len(self.heads)]
            x = W.as_float64(inp.K[0, T - 1:T, h], wl.in_dtype)
            O.quantize(x, self.specs[h][0], O.norm_dtype_name(wl))
            x = W.as_float64(inp.V[0, T - 1:T, h], wl.in_dtype)
            O.quantize(x, self.specs[h][1], O.norm_dtype_name(wl))
            ek, ev = self.encs[h]
            oracle_attention(self.st, ek, ev, 0, h, T)
        return time.perf_counter() - t0

    def seconds_per_pair(self, reps=1):
        from gpu_harness import oracle_attention
        O, wl, T, inp = self.O, self.wl, self.T, self.inp
        t0 = time.perf_counter()
        n = 0
        for _ in range(reps):
            for h in self.heads:
                x = W.as_float64(inp.K[0, T - 1:T, h], wl.in_dtype)
                O.quantize(x, self.specs[h][0], O.norm_dtype_name(wl))
                x = W.as_float64(inp.V[0, T - 1:T, h], wl.in_dtype)
                O.quantize(x, self.specs[h][1], O.norm_dtype_name(wl))
                ek, ev = self.encs[h]
                oracle_attention(self.st, ek, ev, 0, h, T)
                n += 1
        return (time.perf_counter() - t0) / n


def bench_config(wl, T, sb, world):
    return {"workload": workload_name(wl, T), "batch": wl.batch, "seq_len": T,
            "parallelism": "replicas" if world == 1 else f"replicas x{world}",
            "l2": "inputs larger than L2 (%.0f MB read per step vs 129 MB L2); two cache copies "
                  "alternated between steps" % (sb["decode"] / 1e6)}


def accuracy_stats(tq, wl, T, inp, cache, out, pairs):
    """Statistics of the GPU path against the oracle on sampled (batch, KV head)
    pairs, from the GPU's own packed cache: near-boundary fractions of the
    oracle's rotated coordinates (normalised frame: |y - b| <= 1e-5; scaled frame:
    |n (y - b)| <= 1e-5), the fraction of codes that differ, the attention error
    against the oracle on that same cache (and its margin to 2e-3 max|o|), and
    the error against exact fp64 attention on the unquantised inputs."""
    from gpu_harness import OracleEnc, Setup, compare_codes, oracle_encode, pair_norms, pair_records
    from oracle import tq_oracle as O
    st = Setup(wl, inp, None, None, O.head_specs(wl, inp), None, None)
    o = out.float().cpu().numpy()
    G = wl.group
    nbad = ntot = 0
    fw, fws, margin, exact_rel, exact_rms = [], [], [], [], []
    for b, h in pairs:
        recs = {}
        for which in ("k", "v"):
            enc = oracle_encode(st, which, b, h, 0, T)
            spec = st.specs[h][0 if which == "k" else 1]
            rec = pair_records(cache, which, b, h, st)[:T]
            nb_, n_, f1, f2, _ = compare_codes(rec, enc, spec)
            nbad, ntot = nbad + nb_, ntot + n_
            fw.append(f1)
            fws.append(f2)
            recs[which] = OracleEnc(rec, O.unpack(rec, spec, 128), pair_norms(cache, which, b, h)[:T], enc.y)
        ks, vs = st.specs[h]
        q = W.as_float64(inp.q[b, h * G:(h + 1) * G], wl.in_dtype)
        ref = O.attend_rotated(q, recs["k"].idx, recs["k"].norms.astype(np.float64), ks, recs["v"].idx,
                               recs["v"].norms.astype(np.float64), vs, T)
        got = o[b, h * G:(h + 1) * G].astype(np.float64)
        scale = float(np.max(np.abs(ref)))
        margin.append(float(np.max(np.abs(got - ref))) / (2e-3 * scale))
        Kx = W.as_float64(inp.K[b, :T, h], wl.in_dtype)
        Vx = W.as_float64(inp.V[b, :T, h], wl.in_dtype)
        ex = O.attend_exact(q, Kx, Vx, T)
        exact_rel.append(float(np.max(np.abs(got - ex))) / float(np.max(np.abs(ex))))
        exact_rms.append(float(np.sqrt(np.mean((got - ex) ** 2)) / np.sqrt(np.mean(ex ** 2))))
    return {"pairs": [list(p) for p in pairs], "mismatch_frac": nbad / ntot,
            "near_boundary_frac_normalised": float(np.mean(fw)), "near_boundary_frac_scaled": float(np.mean(fws)),
            "parity_margin": max(margin), "exact_attention_rel_err": max(exact_rel),
            "exact_attention_rms_rel_err": max(exact_rms),
            "note": "margin = max|o - oracle on the same cache| / (2e-3 max|o|); exact = max|o - fp64 attention "
                    "on the unquantised inputs| / max|exact| (and the same in root-mean-square terms)"}


def cpu_cores():
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(v):
            return int(os.environ[v])
    return os.cpu_count()


def run_reference(args, wl, T, rank, world):
    """The oracle as it stands on the host cores: every step encodes the new
    token's K and V and runs attention over T cached tokens for every (batch, KV
    head) pair of the workload.  The cached codes of NREF distinct pairs are
    encoded once (untimed) and cycled over the pairs: the oracle's work does not
    depend on the values."""
    if rank != 0:
        return
    from rotated_bit_kv_gb300 import tq_cache_desc
    d = tq_cache_desc()
    d.k_code_bytes = d.v_code_bytes = 48
    d.k_norm_slots = d.v_norm_slots = 1
    d.norm_bytes = 2
    sb = step_bytes(wl, T, d)
    pairs_total = wl.batch * wl.n_kv_heads
    leg = OracleLeg(wl, T, n_pairs=NREF)
    for _ in range(args.warmup):
        leg.run_pairs(pairs_total)
    times = []
    for _ in range(args.steps):
        times.append(leg.run_pairs(pairs_total))
    step_s = statistics.mean(times)
    val = sb["step"] / step_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "us_per_step": step_s * 1e6,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(wl, T, sb, world),
        "cpu_baseline": {"kind": "oracle", "value": val, "unit": "GB/s", "cores": cpu_cores(),
                         "sample": f"every step: oracle encode of the new token + attention over T={T} for all "
                                   f"{pairs_total} (batch, KV head) pairs (the cached codes of {NREF} distinct "
                                   f"pairs, encoded once, cycled over them)"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def reduce_max_over_ranks(x, dist, device):
    """Largest of x over the ranks of the default process group (x itself
    without one); the job's time is the slowest rank's."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _to_torch(torch, x, dtype, device):
    """A workload array (bf16 kept as its 16-bit patterns) as a device tensor."""
    if dtype == W.BF16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


# ----------------------------------------------------------------------------
def run_ours(args, wl, T, rank, world, local_rank):
    import torch

    import rotated_bit_kv_gb300 as tq

    tq.build()
    lib = tq.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
    inp = W.make_inputs(wl, seq_len=T)
    # descriptor and parameter blob from the library alone (uniform-rate keys)
    desc = tq.tq_cache_desc_init(wl.head_dim, wl.n_q_heads, wl.n_kv_heads, wl.batch, T, wl.rot, wl.k_bits, wl.v_bits,
                                 wl.norm_dtype, 0)
    blob = tq.tq_params_build(desc, signs=inp.signs, quats=inp.quats, k_block_bits=None, k_group_mats=None)
    # two cache copies alternated between steps: each step reads ~210 MB, more
    # than L2, and never the copy the previous step read
    caches = [tq.PackedKVCache(desc, blob, device=dev) for _ in range(2)]
    K = _to_torch(torch, inp.K, wl.in_dtype, dev)
    V = _to_torch(torch, inp.V, wl.in_dtype, dev)
    zero = torch.zeros(wl.batch, dtype=torch.int32, device=dev)
    pf = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    for i, c in enumerate(caches):
        if i == 1:
            pf[0].record()
        c.append(K, V, zero)
        if i == 1:
            pf[1].record()
    torch.cuda.synchronize()
    # whole-prompt append (write side W1-W4 over every token), timed on the second cache
    pf_us = pf[0].elapsed_time(pf[1]) * 1e3
    pf_bytes = (K.numel() + V.numel()) * K.element_size() + 2 * wl.batch * wl.n_kv_heads * T * (48 + 2)
    prefill = {"tokens": wl.batch * T, "us": pf_us, "GB/s": pf_bytes / (pf_us * 1e-6) / 1e9,
               "bytes": pf_bytes}
    k_new = K[:, T - 1:T].contiguous()
    v_new = V[:, T - 1:T].contiguous()
    del K, V
    q = _to_torch(torch, inp.q, wl.in_dtype, dev)
    start = torch.full((wl.batch,), T - 1, dtype=torch.int32, device=dev)
    seq = torch.full((wl.batch,), T, dtype=torch.int32, device=dev)
    out = torch.empty((wl.batch, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
    splits, vmode = tq.tq_decode_plan(desc, T, tq.TQ_VMODE_TENSOR_STREAMK if args.streamk else tq.TQ_VMODE_AUTO,
                                      args.splits)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    in_code = tq._dtype_code(q)
    dref = ctypes.byref(desc)
    pref = [ctypes.byref(c.ptrs) for c in caches]

    def step(i, ev=None, qd=q, kd=k_new, vd=v_new, sd=start, ld=seq, od=out):
        c = caches[i & 1]
        st_ = lib.tq_quantize_append(dref, pref[i & 1], kd.data_ptr(), vd.data_ptr(), in_code, sd.data_ptr(), 1,
                                     c.status.data_ptr(), sptr)
        if ev is not None:
            ev[0].record(stream)
        st2 = lib.tq_decode_attention_ex(dref, pref[i & 1], qd.data_ptr(), in_code, ld.data_ptr(), T, od.data_ptr(),
                                         c.workspace.data_ptr(), c.workspace.numel(), c.status.data_ptr(), sptr,
                                         vmode, splits)
        if ev is not None:
            ev[1].record(stream)
        if st_ or st2:
            raise RuntimeError(f"library error {st_} {st2}")

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return reduce_max_over_ranks(x, dist, dev)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)   # nvidia-smi is running before the timed region starts
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_a.record(stream)
    for i in range(args.steps):
        step(i, kev[i])
    t_b.record(stream)
    barrier()
    elapsed_ms = max_over_ranks(t_a.elapsed_time(t_b))
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    # clock window: the same steps repeated for at least a second after the timed
    # region, so that the sampler sees the GPU under this load
    w_a, w_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_win = max(1, int(math.ceil(1.2 / max(elapsed_ms / args.steps * 1e-3, 1e-6))))
    w_a.record(stream)
    for i in range(n_win):
        step(i)
    w_b.record(stream)
    barrier()
    win_us = w_a.elapsed_time(w_b) * 1e3 / n_win
    clocks = sampler.stop() if sampler else None
    if clocks is not None:
        clocks["window"] = {"steps": n_win, "seconds": win_us * n_win * 1e-6, "us_per_step": win_us,
                            "note": "clocks sampled over the timed steps and a window of the same steps after them"}
    for c in caches:
        if int(c.status.item()) != 0:
            raise RuntimeError(f"device status {int(c.status.item())}")

    # end to end through the C ABI with host buffers: pinned H2D of the step's
    # inputs (q, new K/V token, positions, lengths) and D2H of the output
    # the step's host inputs live in one pinned buffer and go over in one copy
    parts = [q, k_new, v_new, start, seq]
    offs, off = [], 0
    for x in parts:
        offs.append(off)
        off += (x.numel() * x.element_size() + 255) // 256 * 256
    hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(off, dtype=torch.uint8, device=dev)
    dviews = []
    for x, o in zip(parts, offs):
        nb = x.numel() * x.element_size()
        hbuf[o:o + nb].copy_(x.reshape(-1).view(torch.uint8).cpu())
        dviews.append(dbuf[o:o + nb].view(x.dtype).view(x.shape))
    dq, dk, dv, ds, dl = dviews
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = off
    d2h = hout.numel() * hout.element_size()

    def e2e_step(i):
        dbuf.copy_(hbuf, non_blocking=True)
        step(i, None, dq, dk, dv, ds, dl, out)
        hout.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    barrier()
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e_b.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e_a.elapsed_time(e_b))

    sb = step_bytes(wl, T, desc)
    step_ms = elapsed_ms / args.steps
    value = world * sb["step"] / (step_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    achieved = sb["decode"] / (dec_ms * 1e-3) / 1e9
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "us_per_step": step_ms * 1e3,
        "pct_of_peak": 100.0 * (value / world) / peak, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": bench_config(wl, T, sb, world),
        "decode_plan": {"ctas": splits, "v_mode": vmode},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(), "kernel": "decode attention",
                     "us_per_launch": dec_ms * 1e3, "algorithmic_bytes_per_launch": sb["decode"],
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy kernel; spec ~7900)"},
        "e2e": {"value": world * sb["step"] / (e2e_ms / args.steps * 1e-3) / 1e9, "unit": "GB/s",
                "us_per_step": e2e_ms / args.steps * 1e3, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "prefill_append": prefill,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["stats"] = accuracy_stats(tq, wl, T, inp, caches[(args.steps - 1) & 1], out,
                                       [(0, 0), (wl.batch - 1, wl.n_kv_heads - 1)])
        leg = OracleLeg(wl, T, n_pairs=2)
        npairs = len(leg.heads)
        dt = leg.seconds_per_pair(reps=4)
        pairs_total = wl.batch * wl.n_kv_heads
        cpu_step = dt * pairs_total
        line["cpu_baseline"] = {
            "kind": "oracle", "value": sb["step"] / cpu_step / 1e9, "unit": "GB/s", "cores": cpu_cores(),
            "sample": f"oracle (fp64 NumPy) encode of the new token + attention over T={T} for {npairs} (batch, KV "
                      f"head) pairs x4, scaled linearly to all {pairs_total} pairs"}
    print(json.dumps(line), flush=True)


def library_setup(tq, wl, inp, t_capacity):
    """Descriptor and parameter blob through the library alone.  Mixed-rate keys:
    block energies and the greedy allocation from the library's own entry
    points, one seeded Haar matrix per non-empty same-width group (ascending
    width) of each KV head.  Two-stage keys: one seeded projection per KV head."""
    block_bits = mats = None
    if wl.mixed_k:
        G = wl.group
        kc = W.as_float64(inp.K[0, :wl.calib_tokens], wl.in_dtype).astype(np.float32)
        qc = W.as_float64(inp.q_calib, wl.in_dtype).astype(np.float32)
        bbs, flat = [], []
        for h in range(wl.n_kv_heads):
            s_h = tq.tq_block_energy(qc[:, h * G:(h + 1) * G], kc[:, h])
            bb = tq.tq_block_bit_alloc(s_h, wl.b_min, wl.b_max, wl.avg_bits * (wl.head_dim // 2))
            bbs.append(bb)
            for b in range(wl.b_min, wl.b_max + 1):
                n = 2 * int(np.count_nonzero(np.asarray(bb) == b))
                if n:
                    flat.append(W.haar_orthogonal(n, wl.seed, h, b).ravel())
        block_bits = np.stack(bbs).astype(np.int32)
        mats = np.concatenate(flat)
    k_mixed = (2 if wl.tight_k else 1) if wl.mixed_k else 0
    k_bits = (wl.avg_bits if wl.tight_k else 0) if wl.mixed_k else wl.k_bits
    if not wl.mixed_k and wl.k_bits in (1, 2):   # two-stage keys: the projections
        mats = np.stack([W.two_stage_projection(wl.head_dim, wl.seed, h) for h in range(wl.n_kv_heads)])
    desc = tq.tq_cache_desc_init(wl.head_dim, wl.n_q_heads, wl.n_kv_heads, wl.batch, t_capacity, wl.rot,
                                 k_bits, wl.v_bits, wl.norm_dtype, k_mixed)
    blob = tq.tq_params_build(desc, signs=inp.signs, quats=inp.quats, k_block_bits=block_bits, k_group_mats=mats)
    return desc, blob


def _cold_launch_us(torch, flush, launch, steps):
    """Median device time of one launch with a cold L2: each timed launch follows
    a write of a buffer larger than L2, then a device-side wait of about 50 us so
    that the host has queued the start event and the launch before the device
    reaches them (the interval then holds the kernel alone, not the host's
    submission latency).  CUDA events on the current stream."""
    for _ in range(3):
        launch()
    times = []
    for _ in range(steps):
        flush.zero_()
        torch.cuda._sleep(100_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        times.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(x.elapsed_time(y) for x, y in times) * 1e3


def run_sweep(args):
    """Decode time on every synthetic workload (not the bench line): one cache
    filled by a whole-prompt append, the library's plan, L2 flushed before each
    timed launch, CUDA events around the decode alone."""
    import torch

    import rotated_bit_kv_gb300 as tq

    tq.build()
    dev = torch.device("cuda", 0)
    peak, _ = measured_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cases = [(W.llama8b_decode(seq_len=t), t) for t in (128, 256, 512, 2048, 8192)]
    cases += [(W.block32(3), 8192), (W.block32(4), 8192)]
    cases += [(W.so4_wht(seq_len=t), t) for t in (128, 256, 512, 2048, 8192, 32768)]
    cases += [(W.mixed_rate_long(seq_len=t), t) for t in (131072, 524288)]
    # mixed-rate keys in tight records (natural layout, CUDA-core kernels)
    cases += [(W.mixed_rate_long(seq_len=131072).with_(tight_k=True, name="mixed_rate_long_tight"), 131072)]
    print("| workload | B | T | plan (splits, V mode) | decode us | GB/s | of measured peak |")
    print("|---|---|---|---|---|---|---|")
    for wl, T in cases:
        if args.only and args.only not in wl.name:
            continue
        wl = wl.with_(batch=wl.batch, seq_len=T)
        inp = W.make_inputs(wl, seq_len=T)
        desc, blob = library_setup(tq, wl, inp, T)
        cache = tq.PackedKVCache(desc, blob, device=dev)
        K = _to_torch(torch, inp.K, wl.in_dtype, dev)
        V = _to_torch(torch, inp.V, wl.in_dtype, dev)
        cache.append(K, V, torch.zeros(wl.batch, dtype=torch.int32, device=dev))
        del K, V
        q = _to_torch(torch, inp.q, wl.in_dtype, dev)
        seq = torch.full((wl.batch,), T, dtype=torch.int32, device=dev)
        out = torch.empty((wl.batch, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
        splits, vmode = tq.tq_decode_plan(desc, T, tq.TQ_VMODE_AUTO, args.splits)
        us = _cold_launch_us(torch, flush, lambda: cache.decode(q, seq, T, out=out, n_splits=args.splits), args.steps)
        if int(cache.status.item()) != 0:
            raise RuntimeError(f"device status {int(cache.status.item())}")
        nbytes = step_bytes(wl, T, desc)["decode"]
        gbs = nbytes / (us * 1e-6) / 1e9
        print(f"| {wl.name} | {wl.batch} | {T} | {splits}, {vmode} | {us:.1f} | {gbs:.0f} | {100 * gbs / peak:.1f} % |",
              flush=True)
        del cache, q, out
        torch.cuda.empty_cache()


def run_crossover(args):
    """Token- against dimension-parallel V accumulation on the caches that use those
    kernels (natural layout: 16 query heads per KV head, fp32 norms with mixed-rate
    keys or with 32-wide blocks, tight mixed-rate records, two-stage keys): decode time of
    each kernel over a range of lengths (one cache per workload filled to its longest
    length, the same launches as the sweep)."""
    import torch

    import rotated_bit_kv_gb300 as tq

    tq.build()
    dev = torch.device("cuda", 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    lengths = [64, 128, 256, 384, 512, 768, 1024, 2048, 4096]
    cases = [W.mixed_rate_long(seq_len=max(lengths)).with_(norm_dtype=W.F32),
             W.llama8b_decode(seq_len=max(lengths), batch=8).with_(n_kv_heads=2),
             W.block32(3, seq_len=max(lengths), batch=8).with_(norm_dtype=W.F32),
             W.mixed_rate_long(seq_len=max(lengths)).with_(tight_k=True, name="mixed_rate_long_tight"),
             W.two_stage_keys(2, seq_len=max(lengths), batch=8)]
    if args.only:
        cases = [wl for wl in cases if args.only in wl.name]
    print("| workload | B | T | token-parallel us | dimension-parallel us | faster |")
    print("|---|---|---|---|---|---|")
    for wl in cases:
        Tm = max(lengths)
        inp = W.make_inputs(wl, seq_len=Tm)
        desc, blob = library_setup(tq, wl, inp, Tm)
        assert desc.layout == tq.TQ_LAYOUT_NATURAL
        cache = tq.PackedKVCache(desc, blob, device=dev)
        K = _to_torch(torch, inp.K, wl.in_dtype, dev)
        V = _to_torch(torch, inp.V, wl.in_dtype, dev)
        cache.append(K, V, torch.zeros(wl.batch, dtype=torch.int32, device=dev))
        del K, V
        q = _to_torch(torch, inp.q, wl.in_dtype, dev)
        out = torch.empty((wl.batch, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
        name = wl.name + f" (G={wl.group}, {'fp32' if wl.norm_dtype == W.F32 else 'fp16'} norms)"
        for T in lengths:
            seq = torch.full((wl.batch,), T, dtype=torch.int32, device=dev)
            res = []
            for vm in (tq.TQ_VMODE_TOKEN_PARALLEL, tq.TQ_VMODE_DIM_PARALLEL):
                res.append(_cold_launch_us(torch, flush, lambda: cache.decode(q, seq, T, out=out, v_mode=vm),
                                           args.steps))
            print(f"| {name} | {wl.batch} | {T} | {res[0]:.1f} | {res[1]:.1f} | "
                  f"{'token' if res[0] < res[1] else 'dimension'} |", flush=True)
        del cache, q, out
        torch.cuda.empty_cache()


def run_prefix(args):
    """Decode over unquantised (fp16) tokens plus the packed cache: time of the
    packed decode alone and of the whole call (packed decode, then the fp16
    kernel with the log-sum-exp merge), cold L2 as in the sweep; bytes = the
    packed part's decode bytes + the unquantised K and V read."""
    import torch

    import rotated_bit_kv_gb300 as tq

    tq.build()
    dev = torch.device("cuda", 0)
    peak, _ = measured_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cases = [(W.llama8b_decode(seq_len=6144), 6144, 2048, "fp16 prefix 2048 + packed 6144"),
             (W.llama8b_decode(seq_len=512), 512, 8192, "deferred prefill: fp16 prompt 8192 + packed 512"),
             (W.mixed_rate_long(131072), 131072, 128, "recent-token buffer: fp16 128 + packed 131072"),
             (W.so4_wht(seq_len=128), 128, 32768, "fp16 prompt 32768 + packed 128")]
    print("| workload | B | packed T | fp16 P | packed decode us | whole call us | fp16 part us | "
          "whole-call GB/s | of measured peak |")
    print("|---|---|---|---|---|---|---|---|---|")
    for wl, T, P, what in cases:
        if args.only and args.only not in wl.name:
            continue
        inp = W.make_inputs(wl, seq_len=T)
        desc, blob = library_setup(tq, wl, inp, T)
        cache = tq.PackedKVCache(desc, blob, device=dev)
        K = _to_torch(torch, inp.K, wl.in_dtype, dev)
        V = _to_torch(torch, inp.V, wl.in_dtype, dev)
        cache.append(K, V, torch.zeros(wl.batch, dtype=torch.int32, device=dev))
        del K, V
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        kp = torch.randn((wl.batch, P, wl.n_kv_heads, 128), generator=g, device=dev).to(torch.float16)
        vp = torch.randn((wl.batch, P, wl.n_kv_heads, 128), generator=g, device=dev).to(torch.float16)
        q = _to_torch(torch, inp.q, wl.in_dtype, dev)
        seq = torch.full((wl.batch,), T, dtype=torch.int32, device=dev)
        pl = torch.full((wl.batch,), P, dtype=torch.int32, device=dev)
        out = torch.empty((wl.batch, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device=dev)
        us_p = _cold_launch_us(torch, flush, lambda: cache.decode(q, seq, T, out=out), args.steps)
        us_w = _cold_launch_us(torch, flush, lambda: cache.decode_prefix(q, seq, T, kp, vp, pl, P, out=out),
                               args.steps)
        if int(cache.status.item()) != 0:
            raise RuntimeError(f"device status {int(cache.status.item())}")
        nbytes = step_bytes(wl, T, desc)["decode"] + 2 * kp.numel() * kp.element_size()
        gbs = nbytes / (us_w * 1e-6) / 1e9
        print(f"| {wl.name} ({what}) | {wl.batch} | {T} | {P} | {us_p:.1f} | {us_w:.1f} | {us_w - us_p:.1f} | "
              f"{gbs:.0f} | {100 * gbs / peak:.1f} % |", flush=True)
        del cache, q, out, kp, vp
        torch.cuda.empty_cache()


def run_zip(args):
    """ZipFusion store and attention (a table): the llama8b shape at the pages'
    measured setting (batch 32, 2048 tokens, bf16 K/V with the llama8b channel
    recipe), and longer contexts.  Time of the attention on the compressed pages
    and of the same tensor-core attention on the raw bf16 rows (the unquantised-
    token path with no packed token), cold L2; bytes = what each one reads."""
    import torch

    import rotated_bit_kv_gb300 as tq

    tq.build()
    dev = torch.device("cuda", 0)
    peak, _ = measured_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    print("| workload | B | T | stored / raw bytes | zip attention us | raw bf16 attention us | zip GB/s read | "
          "of measured peak | raw-equivalent GB/s |")
    print("|---|---|---|---|---|---|---|---|---|")
    for wl, T in ((W.llama8b_decode(seq_len=2048), 2048), (W.llama8b_decode(seq_len=8192), 8192)):
        inp = W.make_inputs(wl, seq_len=T)
        K = _to_torch(torch, inp.K, W.BF16, dev)
        V = _to_torch(torch, inp.V, W.BF16, dev)
        q = _to_torch(torch, inp.q, W.BF16, dev)
        lens = torch.full((wl.batch,), T, dtype=torch.int32, device=dev)
        z = tq.ZipKVCache(wl.batch, wl.n_q_heads, wl.n_kv_heads, T, device=dev)
        z.store(K, V, lens)
        torch.cuda.synchronize()
        if int(z.status.item()) != 0:
            raise RuntimeError(f"device status {int(z.status.item())}")
        # bytes the attention reads: every block at its stored size (+ metadata, q, out)
        stored = 0
        for meta in (z.k_meta, z.v_meta):
            m = meta.cpu().numpy().view(np.uint32).reshape(-1, 2)[:, 1]
            marks = np.stack([(m >> (8 * j)) & 0xFF for j in range(4)])
            stored += int(np.where(marks == 0xFF, 1024, 768).sum()) + m.size * 8
        raw = 2 * K.numel() * 2
        qo = q.numel() * 2 + q.numel() * 4
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
        us_z = _cold_launch_us(torch, flush, lambda: z.decode(q, lens, T, out=out), args.steps)
        # the raw rows through the prefix entry (no packed token)
        desc = tq.tq_cache_desc_init(128, wl.n_q_heads, wl.n_kv_heads, wl.batch, 16, W.ROT_WHT128, 3, 3, W.F16)
        blob = tq.tq_params_build(desc, signs=inp.signs[:, :])
        cache = tq.PackedKVCache(desc, blob, device=dev)
        zero = torch.zeros(wl.batch, dtype=torch.int32, device=dev)
        us_r = _cold_launch_us(torch, flush, lambda: cache.decode_prefix(q, zero, 0, K, V, lens, T, out=out), args.steps)
        gbs = (stored + qo) / (us_z * 1e-6) / 1e9
        eq = (raw + qo) / (us_z * 1e-6) / 1e9
        print(f"| {wl.name} (bf16, ZipFusion pages) | {wl.batch} | {T} | {stored / raw:.3f} | {us_z:.1f} | {us_r:.1f} | "
              f"{gbs:.0f} | {100 * gbs / peak:.1f} % | {eq:.0f} |", flush=True)
        del z, K, V, cache
        torch.cuda.empty_cache()


def run_two_stage(args):
    """Two-stage keys (a (k_bits - 1)-bit MSE code plus a 1-bit QJL code of the
    residual) on the llama8b head shape (a table): the whole-prompt append and the
    decode (CUDA-core kernels on the natural layout, the library's plan), cold L2;
    bytes = K and V records and norms read + q + out."""
    import torch

    import rotated_bit_kv_gb300 as tq

    tq.build()
    dev = torch.device("cuda", 0)
    peak, _ = measured_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    print("| workload | B | T | K bytes / token-head | plan (splits, V mode) | append us | decode us | GB/s | "
          "of measured peak |")
    print("|---|---|---|---|---|---|---|---|---|")
    for k_bits in (1, 2):
        wl = W.two_stage_keys(k_bits, seq_len=args.seq_len, batch=8)
        T = wl.seq_len
        inp = W.make_inputs(wl, seq_len=T)
        desc = tq.tq_cache_desc_init(128, wl.n_q_heads, wl.n_kv_heads, wl.batch, T, wl.rot, wl.k_bits, wl.v_bits,
                                     wl.norm_dtype)
        S = np.stack([W.two_stage_projection(128, wl.seed, h) for h in range(wl.n_kv_heads)])
        cache = tq.PackedKVCache(desc, tq.tq_params_build(desc, signs=inp.signs, k_group_mats=S), device=dev)
        K = _to_torch(torch, inp.K, W.BF16, dev)
        V = _to_torch(torch, inp.V, W.BF16, dev)
        q = _to_torch(torch, inp.q, W.BF16, dev)
        start = torch.zeros(wl.batch, dtype=torch.int32, device=dev)
        us_a = _cold_launch_us(torch, flush, lambda: cache.append(K, V, start), max(3, args.steps // 4))
        if int(cache.status.item()) != 0:
            raise RuntimeError(f"device status {int(cache.status.item())}")
        lens = torch.full((wl.batch,), T, dtype=torch.int32, device=dev)
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
        us = _cold_launch_us(torch, flush, lambda: cache.decode(q, lens, T, out=out), args.steps)
        pairs = wl.batch * wl.n_kv_heads
        per = desc.k_code_bytes + desc.k_norm_slots * desc.norm_bytes + desc.v_code_bytes + desc.norm_bytes
        nbytes = pairs * T * per + q.numel() * 2 + q.numel() * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        sp, vm = tq.tq_decode_plan(desc, T)
        print(f"| {wl.name} | {wl.batch} | {T} | {desc.k_code_bytes + 2 * desc.norm_bytes} | {sp}, {vm} | "
              f"{us_a:.1f} | {us:.1f} | {gbs:.0f} | {100 * gbs / peak:.1f} % |", flush=True)
        del cache, K, V
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seq-len", type=int, default=8192)
    ap.add_argument("--batch", type=int, default=32, help="smaller batches are for profiling captures only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--splits", type=int, default=0, help="key-axis splits (0: the library's plan)")
    ap.add_argument("--streamk", action="store_true", help="tensor-core kernel with the stream-K partition")
    ap.add_argument("--sweep", action="store_true",
                    help="decode time on every synthetic workload (a table, not the bench line)")
    ap.add_argument("--only", default="", help="sweep: workloads whose name contains this")
    ap.add_argument("--crossover", action="store_true",
                    help="token- against dimension-parallel decode on natural-layout caches (a table)")
    ap.add_argument("--prefix", action="store_true",
                    help="decode over fp16 tokens plus the packed cache (a table)")
    ap.add_argument("--zip", action="store_true", help="ZipFusion store and attention (a table)")
    ap.add_argument("--two-stage", action="store_true",
                    help="keys at 1-2 bits with the QJL residual stage: append and decode (a table)")
    args = ap.parse_args()
    if args.two_stage:
        run_two_stage(args)
        return
    if args.zip:
        run_zip(args)
        return
    if args.prefix:
        run_prefix(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.crossover:
        run_crossover(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = W.llama8b_decode(seq_len=args.seq_len, batch=args.batch)
    if args.impl == "reference":
        run_reference(args, wl, args.seq_len, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, wl, args.seq_len, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
