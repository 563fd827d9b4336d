#!/usr/bin/env python
"""Benchmark of the OSCAR INT2 KV-cache decode step on GB300.

Workload: one Qwen3-8B-shaped attention layer (32 query / 8 KV heads, head_dim 128) at 100,000 tokens
of context = 64 BF16 sink + 99,680 INT2 history (paged, shuffled page table, partial last page) + 256
BF16 recent, batch 1, group 128, clip 0.9, covariance-aligned rotations computed on the GPU from
synthetic anisotropic calibration samples.  One step = append the new token (demoting the oldest
recent token into the INT2 history) + decode attention over the whole pool.  Steps rotate over
several layer buffers whose total size exceeds the L2 cache, so every step reads its KV from HBM.

Metric: KV tokens/s (tokens of context attended per second, one layer, all heads), with the history
kernel's achieved HBM bandwidth against the measured peak.  Synthetic data (seeded); no weights.
"""
from __future__ import annotations

import argparse
import ctypes as C
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

L_CTX, HQ, HKV, D, GROUP, CLIP = 100_000, 32, 8, 128, 128, 0.9
SINK, RECENT, PAGE = 64, 256, 64
CALIB_T = 4096
ATTN_KERNEL = "v1::attn_kernel (INT2 history + BF16 sink/recent CTAs)"
ATTN_KERNEL_KEY = "v1::attn_kernel"
# the sources the attention kernel is compiled from (a traffic record holds only while they are unchanged)
ATTN_SRC = [os.path.join(ROOT, "bit_rotated_kv_02_gb300", "csrc", f)
            for f in ("decode_v1.cu", "bf16_part.cuh", "split.cuh", "oscar_internal.cuh", "ptx.cuh")]
# the BF16 sink/window bytes are read by the same launch (its BF16 CTAs)
ATTN_HAS_BF16 = True
METRIC = "INT2-KV decode attn: KV tokens/s, HBM GB/s as frac of GB300 peak; demote tok/s"
WORKLOAD = "qwen3-8b-layer decode, 100k context (64 sink + 99,680 INT2 history + 256 recent), batch 1"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=10,
                    help="rotating layer buffers (working set >= 4x the 129 MB L2)")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["decode100k", "batch-sweep", "bulk", "mixed", "bf16-compare",
                                           "shared-prefix", "quality", "codebook"],
                    default="decode100k",
                    help="decode100k is the headline line; the others measure the remaining workloads")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-cores", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-kind", choices=["decode", "bulk", "demote"], default="decode", help=argparse.SUPPRESS)
    ap.add_argument("--roofline-launches", type=int, default=64,
                    help="attention launches timed one by one with CUDA events after the run")
    return ap.parse_args()


# ---------------------------------------------------------------------------------------------
# Oracle CPU baseline (the only place besides --impl reference that runs oracle/): decode steps of one KV
# head (its 4 query heads), i.e. 1/8 of the layer's step each, within a time budget.  On all cores every
# process runs the same sample on its own copy (processes started with spawn, one thread each).
def _oracle_sample_setup():
    import numpy as np
    import synth
    from oracle import pool as opool
    from oracle import rotation as orot
    ch = synth.outlier_channels(7, 1, D, 4)
    K = synth.outlier_kv(8, L_CTX + 512, 1, D, ch)
    V = synth.outlier_kv(9, L_CTX + 512, 1, D, ch)
    q = synth.outlier_q(10, 1, HQ // HKV, 1, D, ch)
    R = orot.to_f32(orot.rotation_from_gaussian(synth.gaussian_matrix(11, D)))[None]
    hist = L_CTX - SINK - RECENT
    pages = -(-(hist + 512) // PAGE) + 2
    O = opool.Pool(1, HQ // HKV, 1, D, GROUP, pages, pages, R, R, [CLIP], [CLIP])
    O.page_table[0] = synth.shuffled_pages(12, pages)
    O.prefill(0, K[:L_CTX], V[:L_CTX])
    return O, K, V, q


def oracle_sample_steps(n_steps: int, budget_s: float = 1e9):
    """(per-step seconds, tokens attended) of up to n_steps oracle decode steps of KV head 0 at 100k
    context (append with demotion + float64 attention), stopping once budget_s is spent."""
    O, K, V, q = _oracle_sample_setup()
    times, ctx = [], []
    for n in range(min(n_steps, 512)):
        t0 = time.perf_counter()
        O.append(K[L_CTX + n][None], V[L_CTX + n][None])
        O.decode(q)
        times.append(time.perf_counter() - t0)
        ctx.append(L_CTX + n + 1)
        if sum(times) >= budget_s:
            break
    return times, ctx


def _oracle_worker(args):
    budget_s, = args
    import os as _os
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        _os.environ[k] = "1"
    times, ctx = oracle_sample_steps(10 ** 9, budget_s)
    return sum(times), sum(ctx)


SAMPLE_NOTE = ("decode steps of KV head 0 (4 of 32 query heads, 1/8 of the layer) at 100k context, append with "
               "demotion + float64 attention; KV tokens/s scaled to the full layer (x 1/8)")


def cpu_baseline_child(budget_s: float, cores: int) -> dict:
    if cores <= 1:
        t, c = _oracle_worker((budget_s,))
        return {"value": c / t / HKV, "unit": "KV tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"{SAMPLE_NOTE}; one process", "seconds": round(t, 3)}
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(budget_s,)] * cores)
    # every process ran for about the budget at once: aggregate tokens over the slowest process's time
    t = max(r[0] for r in res)
    return {"value": sum(r[1] for r in res) / t / HKV, "unit": "KV tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{SAMPLE_NOTE}; {cores} processes of one thread each, the same sample", "seconds": round(t, 3)}


def cpu_bulk_child(budget_s: float) -> dict:
    """Oracle bulk quantize (exactly rounded rotation, clip, scale/zero, codes) on batches of 2,048 synthetic
    vectors of one KV head, one thread, for about budget_s; tokens/s of K and V of all Hkv heads."""
    import synth
    from oracle import quant as oq, rotation as orot
    ch = synth.outlier_channels(7, 1, D, 2)
    R = orot.to_f32(orot.rotation_from_gaussian(synth.gaussian_matrix(11, D)))
    x = synth.outlier_kv(8, 2048, 1, D, ch)[:, 0, :]
    n, t = 0, 0.0
    while t < budget_s:
        t0 = time.perf_counter()
        oq.quantize_vectors_many(x, R, CLIP, 128)
        t += time.perf_counter() - t0
        n += x.shape[0]
    return {"value": n / t / (2 * 8), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} vectors of one KV head (oracle quantize_vectors_many, batches of 2,048); tokens/s = "
                      "vectors/s / (K and V x 8 KV heads); one process", "seconds": round(t, 3)}


def cpu_demote_child(budget_s: float) -> dict:
    """Oracle append with demotion (the window's oldest K and V vectors rotated, clipped, quantized exactly into
    the history) on a one-sequence, one-KV-head pool, one thread, for about budget_s; tokens/s of a sequence
    with 8 KV heads."""
    import synth
    from oracle import pool as opool, rotation as orot
    ch = synth.outlier_channels(7, 1, D, 4)
    n_tok = SINK + RECENT + 4096
    K = synth.outlier_kv(8, n_tok + 4096, 1, D, ch)
    V = synth.outlier_kv(9, n_tok + 4096, 1, D, ch)
    R = orot.to_f32(orot.rotation_from_gaussian(synth.gaussian_matrix(11, D)))[None]
    pages = -(-(n_tok + 4096) // PAGE) + 1
    O = opool.Pool(1, HQ // HKV, 1, D, GROUP, pages, pages, R, R, [CLIP], [CLIP])
    O.page_table[0] = synth.shuffled_pages(12, pages)
    O.prefill(0, K[:SINK + RECENT], V[:SINK + RECENT])
    n, t = 0, 0.0
    while t < budget_s and n < 4096:
        t0 = time.perf_counter()
        O.append(K[SINK + RECENT + n][None], V[SINK + RECENT + n][None])
        t += time.perf_counter() - t0
        n += 1
    return {"value": n / t / 8, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} appends with demotion on a one-KV-head pool (oracle Pool.append); tokens/s = appends/s "
                      "/ 8 KV heads; one process", "seconds": round(t, 3)}


def run_cpu_baseline(budget_s: float, cores: int = 1, kind: str = "decode") -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", "--cpu-seconds",
                        str(budget_s), "--cpu-cores", str(cores), "--cpu-kind", kind], capture_output=True, text=True,
                       env=env, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": "KV tokens/s", "cores": cores, "kind": "oracle",
                "sample": "failed: " + r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"}
    return json.loads(r.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------------------------------------
# Multi-GPU: one replica of the workload per rank (the path shards into independent sequences and
# has no exchange step), a barrier before and after the timed region, the slowest rank's time.
def max_over_ranks(value: float) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, max_ms: float, world: int) -> float:
    """Whole-job units per second: every rank processed units_per_rank in at most max_ms."""
    return world * units_per_rank / (max_ms * 1e-3)


# ---------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_index, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        """Summarise the samples taken between wall-clock times t0 and t1 (the timed region)."""
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if not (t0 <= ts <= t1):
                    continue
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def sources_sha(paths) -> str:
    """First 16 hex digits of the SHA-256 of the concatenated source files (in the given order)."""
    h = hashlib.sha256()
    for p in paths:
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str, kernel_srcs):
    """DRAM bytes per launch of `kernel` from profiles/traffic.json (written from an ncu capture, with the
    capture's command), if the kernel's source files have not changed since that capture (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[kernel]
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("source_sha256_16") != sources_sha(kernel_srcs):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------------------------
def setup_layers(n_layers: int, extra_tokens: int, seed: int = 2024):
    import torch
    import numpy as np
    import bit_rotated_kv_02_gb300 as ok
    import synth
    dev = torch.device("cuda")
    G = HQ // HKV
    # covariance-aligned rotations from synthetic calibration samples (one set shared by the layers)
    ch = synth.outlier_channels(seed, HKV, D, 4)
    Rk, Rv = [], []
    for h in range(HKV):
        chh = ch[h:h + 1]
        Qc = synth.calib_samples(seed + 10 + h, CALIB_T, G, D, chh, heads_per_channel_set=G)
        KVc = synth.calib_samples(seed + 50 + h, CALIB_T, 2, D, chh, heads_per_channel_set=2)
        tq = torch.from_numpy(Qc.view(np.int16)).view(torch.bfloat16).to(dev)
        tk = torch.from_numpy(np.ascontiguousarray(KVc[:, 0]).view(np.int16)).view(torch.bfloat16).to(dev)
        tv = torch.from_numpy(np.ascontiguousarray(KVc[:, 1]).view(np.int16)).view(torch.bfloat16).to(dev)
        Rk.append(ok.oscar_make_rotation(ok.oscar_calib_covariance_k(tq), ok.ROT_COVARIANCE)[1])
        Rv.append(ok.oscar_make_rotation(ok.oscar_calib_covariance_v(tq, tk, tv), ok.ROT_COVARIANCE)[1])
    Rk, Rv = torch.stack(Rk), torch.stack(Rv)
    clip = torch.full((HKV,), CLIP, dtype=torch.float32)
    hist = L_CTX - SINK - RECENT
    pages = -(-(hist + extra_tokens) // PAGE) + 1
    gen = torch.Generator(device=dev)
    chan = torch.from_numpy(ch.astype(np.int64)).to(dev)
    layers = []
    for l in range(n_layers):
        gen.manual_seed(seed + 1000 + l)
        P = ok.Pool(1, HQ, HKV, GROUP, pages, pages, Rk, Rv, clip, clip)
        P.set_page_table(torch.randperm(pages, generator=gen, device=dev).to(torch.int32)[None])
        for which in range(2):
            x = torch.randn((L_CTX, HKV, D), generator=gen, device=dev)
            x.scatter_(2, chan[None].expand(L_CTX, -1, -1), x.gather(2, chan[None].expand(L_CTX, -1, -1)) * 20)
            if which == 0:
                kx = x.to(torch.bfloat16)
            else:
                vx = x.to(torch.bfloat16)
        ok.oscar_prefill_pool(P, 0, kx, vx)
        del kx, vx
        layers.append(P)
    torch.cuda.synchronize()
    for P in layers:
        assert P.err() == 0
    return layers


# ---------------------------------------------------------------------------------------------
# The other workloads (one JSON line each): synthetic data generated on the GPU from seeded torch
# generators (N(0,1) with outlier channels x20), Haar rotations built by the library.
def _gpu_rotations(ok, n, d, seed):
    import torch
    import synth
    return torch.stack([ok.oscar_make_rotation(torch.from_numpy(synth.gaussian_matrix(seed + i, d)).cuda(),
                                               ok.ROT_HAAR)[1] for i in range(n)])


def _gpu_kv(gen, n, hkv, chan, factor=20.0):
    import torch
    x = torch.randn((n, hkv, D), generator=gen, device="cuda")
    idx = chan[None].expand(n, -1, -1)
    x.scatter_(2, idx, x.gather(2, idx) * factor)
    return x.to(torch.bfloat16)


def _time(fn, steps, warmup):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps   # ms per step


def bf16_compare(args, peak):
    """The 100k-context, batch-1 decode step with the whole history in a BF16 paged cache against the
    same step over the INT2 pool, in one process on the same GPU (the pages' batch-1 speed-up over BF16,
    "评估结果" Fig. 5, measured at kernel level).  Both arms append one token per step."""
    import numpy as np
    import torch
    import bit_rotated_kv_02_gb300 as ok
    import synth
    lib = ok.lib()
    steps, warm = max(3, min(args.steps, 2000)), max(3, min(args.warmup, 50))
    n_bf = 4                                      # 410 MB of KV per layer: every step reads HBM
    per_layer = -(-(steps + warm) // n_bf) + 8
    pages = -(-(L_CTX + per_layer) // PAGE)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5151)
    chan = torch.from_numpy(synth.outlier_channels(2024, HKV, D, 4).astype(np.int64)).cuda()
    caches = []
    for _ in range(n_bf):
        Cc = ok.BF16Cache(1, HQ, HKV, pages, pages)
        Cc.set_page_table(torch.randperm(pages, generator=gen, device="cuda").to(torch.int32)[None])
        ok.oscar_bf16_prefill(Cc, 0, _gpu_kv(gen, L_CTX, HKV, chan), _gpu_kv(gen, L_CTX, HKV, chan))
        caches.append(Cc)
    q = (torch.randn((1, HQ, D), generator=gen, device="cuda") * 3).to(torch.bfloat16)
    kn, vn = _gpu_kv(gen, 1, HKV, chan), _gpu_kv(gen, 1, HKV, chan)
    out = torch.empty((1, HQ, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(ok.oscar_bf16_decode_workspace_size(caches[0]), dtype=torch.uint8, device="cuda")
    EVERY = 8
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(-(-steps // EVERY))]
    for e2 in evs:
        for e in e2:
            e.record()

    def bf_step(i, ev=None):
        if ev is not None:
            lib.oscar_profile_events(0, C.c_void_p(ev[0].cuda_event), C.c_void_p(ev[1].cuda_event))
        ok.oscar_bf16_decode_step(caches[i % n_bf], kn, vn, q, out=out, ws=ws)

    for i in range(warm):
        bf_step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        bf_step(warm + i, evs[i // EVERY] if i % EVERY == 0 else None)
    t1.record()
    torch.cuda.synchronize()
    bf_ms = t0.elapsed_time(t1) / steps
    attn_us = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) * 1e3
    for Cc in caches:
        assert Cc.err() == 0, hex(Cc.err())
    ctx = L_CTX + (steps + warm) / (2 * n_bf)        # mean tokens held over the timed steps
    attn_bytes = ctx * HKV * 2 * D * 2 + 4 * math.ceil(ctx / PAGE) + HQ * D * 2
    del caches, ws
    torch.cuda.empty_cache()
    # the INT2 arm: the headline step over the three-segment pool (3 launches per step)
    NL = 8
    layers = setup_layers(NL, -(-(steps + warm) // NL) + 8)
    ws2 = torch.empty(ok.oscar_decode_workspace_size(layers[0], 0), dtype=torch.uint8, device="cuda")
    step2 = lambda i: ok.oscar_decode_step(layers[i % NL], kn, vn, q, out=out, ws=ws2)
    for i in range(warm):
        step2(i)
    torch.cuda.synchronize()
    t0.record()
    for i in range(steps):
        step2(warm + i)
    t1.record()
    torch.cuda.synchronize()
    int2_ms = t0.elapsed_time(t1) / steps
    achieved = attn_bytes / (attn_us * 1e-6) / 1e9
    return [{"metric": "decode step, BF16 paged cache vs INT2 pool: KV tokens/s", "workload":
             "qwen3-8b-layer decode, 100k context, batch 1: BF16 paged history vs OSCAR INT2 pool",
             "value": L_CTX / (bf_ms * 1e-3), "unit": "KV tokens/s", "ms_per_step": bf_ms, "steps": steps,
             "int2_ms_per_step": int2_ms, "int2_value": L_CTX / (int2_ms * 1e-3),
             "speedup_int2_over_bf16": bf_ms / int2_ms,
             "config": {"num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": D, "page_tokens": PAGE,
                        "l2": f"{n_bf} rotating BF16 caches of {attn_bytes / 1e6:.0f} MB (> L2)"},
             "roofline": {"bound": "hbm", "kernel": "bf::attn_kernel (BF16 paged history)", "achieved": achieved,
                          "peak": peak, "unit": "GB/s", "frac": achieved / peak, "mean_launch_us": attn_us,
                          "algorithmic_bytes_per_launch": attn_bytes, "timed_launches": len(evs),
                          "sampling": f"every {EVERY}th step of the timed region"},
             "gpu_launches": steps * 3}]


def shared_prefix(args, peak):
    """Decode step throughput against the fraction of history pages shared by every sequence of the
    batch (a common prompt prefix held once through the page tables: the prefix-cache use of the paged
    history, "评估结果" Fig. 6).  16 sequences x 32k context, Qwen3-8B layer shapes."""
    import numpy as np
    import torch
    import bit_rotated_kv_02_gb300 as ok
    import synth
    B, L, Hq, Hkv = 16, 32_768, HQ, HKV
    hist = L - SINK - RECENT
    steps = max(3, min(args.steps, 300))
    warm = max(3, min(args.warmup, 20))
    own = -(-(hist + steps + warm + 8) // PAGE)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(6161)
    chan = torch.from_numpy(synth.outlier_channels(2024, Hkv, D, 4).astype(np.int64)).cuda()
    Rk, Rv = _gpu_rotations(ok, Hkv, D, 100), _gpu_rotations(ok, Hkv, D, 200)
    clip = torch.full((Hkv,), 0.9)
    lines = []
    for frac in (0.0, 0.5, 0.9):
        share = int(frac * (hist // PAGE))
        P = ok.Pool(B, Hq, Hkv, 128, B * own, own, Rk, Rv, clip, clip)
        pt = torch.randperm(B * own, generator=gen, device="cuda").to(torch.int32).reshape(B, own)
        pt[1:, :share] = pt[0, :share]
        P.set_page_table(pt)
        K0, V0 = _gpu_kv(gen, L, Hkv, chan), _gpu_kv(gen, L, Hkv, chan)
        ok.oscar_prefill_pool(P, 0, K0, V0)
        for b in range(1, B):
            K, V = _gpu_kv(gen, L, Hkv, chan), _gpu_kv(gen, L, Hkv, chan)
            n = SINK + share * PAGE
            K[:n], V[:n] = K0[:n], V0[:n]
            ok.oscar_prefill_pool_shared(P, b, K, V, share)
        del K0, V0
        q = (torch.randn((B, Hq, D), generator=gen, device="cuda") * 3).to(torch.bfloat16)
        kn, vn = _gpu_kv(gen, B, Hkv, chan), _gpu_kv(gen, B, Hkv, chan)
        out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        ws = torch.empty(ok.oscar_decode_workspace_size(P), dtype=torch.uint8, device="cuda")
        ms = _time(lambda: ok.oscar_decode_step(P, kn, vn, q, out=out, ws=ws), steps, warm)
        assert P.err() == 0, hex(P.err())
        per_tok = Hkv * 2 * (D // 4 + 4)
        unique = (hist + (B - 1) * (hist - share * PAGE)) * per_tok + B * (SINK + RECENT) * Hkv * 2 * D * 2
        lines.append({"metric": "decode step with shared prefix pages: KV tokens/s", "workload":
                      f"qwen3-8b-layer decode, batch {B} x 32k context, {share} of {hist // PAGE} history pages shared",
                      "shared_fraction": share / (hist // PAGE), "value": B * L / (ms * 1e-3), "unit": "KV tokens/s",
                      "ms_per_step": ms, "steps": steps, "unique_bytes_per_step": unique,
                      "unique_gbs": unique / (ms * 1e-3) / 1e9, "unique_frac_of_peak": unique / (ms * 1e-3) / 1e9 / peak})
        del P, ws
        torch.cuda.empty_cache()
    return lines


def codebook_compare(args, peak):
    """The 100k-context, batch-1 decode step over a pool whose history carries Lloyd-Max codebooks
    (calibrated by the library on the first 4,096 tokens of each layer's keys and values) against the
    same step over uniform-INT2 pools, round-robin over 4 layers per arm (history larger than L2)."""
    import numpy as np
    import torch
    import bit_rotated_kv_02_gb300 as ok
    import synth
    steps, warm = max(3, min(args.steps, 400)), max(3, min(args.warmup, 20))
    n_layers, hist = 4, L_CTX - SINK - RECENT
    pages = -(-(hist + (steps + warm) // n_layers + 16) // PAGE)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7171)
    chan = torch.from_numpy(synth.outlier_channels(2024, HKV, D, 4).astype(np.int64)).cuda()
    Rk, Rv = _gpu_rotations(ok, HKV, D, 100), _gpu_rotations(ok, HKV, D, 200)
    clip = torch.full((HKV,), CLIP)
    arms = {"uniform": [], "lloyd_max": []}
    t0 = time.time()
    for l in range(n_layers):
        K, V = _gpu_kv(gen, L_CTX, HKV, chan), _gpu_kv(gen, L_CTX, HKV, chan)
        cbk = ok.oscar_lloyd_max_codebook(K[:4096].contiguous(), Rk.cuda(), clip.cuda())
        cbv = ok.oscar_lloyd_max_codebook(V[:4096].contiguous(), Rv.cuda(), clip.cuda())
        pt = torch.randperm(pages, generator=gen, device="cuda").to(torch.int32)[None]
        for name, cbs in (("uniform", (None, None)), ("lloyd_max", (cbk, cbv))):
            P = ok.Pool(1, HQ, HKV, GROUP, pages, pages, Rk, Rv, clip, clip, codebook_k=cbs[0], codebook_v=cbs[1])
            P.set_page_table(pt)
            ok.oscar_prefill_pool(P, 0, K, V)
            arms[name].append(P)
        del K, V
    torch.cuda.synchronize()
    calib_s = time.time() - t0
    q = (torch.randn((1, HQ, D), generator=gen, device="cuda") * 3).to(torch.bfloat16)
    kn, vn = _gpu_kv(gen, 1, HKV, chan), _gpu_kv(gen, 1, HKV, chan)
    out = torch.empty((1, HQ, D), dtype=torch.float32, device="cuda")
    lines = []
    byts = hist * HKV * 2 * (D // 4 + 4) + (SINK + RECENT) * HKV * 2 * D * 2
    for name, layers in arms.items():
        ws = torch.empty(ok.oscar_decode_workspace_size(layers[0]), dtype=torch.uint8, device="cuda")
        it = [0]

        def step():
            ok.oscar_decode_step(layers[it[0] % n_layers], kn, vn, q, out=out, ws=ws)
            it[0] += 1
        ms = _time(step, steps, warm)
        for P in layers:
            assert P.err() == 0, hex(P.err())
        lines.append({"metric": "decode step (append+demote + attention): KV tokens/s", "variant": name,
                      "workload": WORKLOAD + (", Lloyd-Max codebooks" if name == "lloyd_max" else ", uniform INT2"),
                      "value": L_CTX / (ms * 1e-3), "unit": "KV tokens/s", "ms_per_step": ms, "steps": steps,
                      "step_gbs": byts / (ms * 1e-3) / 1e9, "frac_of_peak": byts / (ms * 1e-3) / 1e9 / peak,
                      "decode_path": "tensor-core INT2" if name == "uniform" else "tensor-core, three indicator planes",
                      "setup_s_incl_calibration": calib_s})
        del ws
    return lines


def quality_workload(args):
    """Attention quality of the four variants of the pages' Fig. 1 (naive INT2, Hadamard-only, clip-only,
    OSCAR) on one Qwen3-8B-shaped layer (32 query / 8 KV heads): calibration-style synthetic activations
    (anisotropic spectrum, four outlier channels per KV head: x4 in q, x10 in K and V), 2,048 calibration
    tokens, one decode query per head over 4,416 tokens of context."""
    import numpy as np
    import torch
    import synth
    import quality_harness as quality
    T, L, G = 2048, 4416, HQ // HKV
    ch = synth.outlier_channels(77, HKV, D, 4)
    Qs = synth.calib_samples(78, T + 1, HQ, D, ch, heads_per_channel_set=G, factor=4.0)
    KV = [synth.calib_samples(79 + h, T + L, 2, D, ch[h:h + 1], heads_per_channel_set=2, factor=10.0)
          for h in range(HKV)]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    K = dev(np.stack([kv[:, 0] for kv in KV], 1))
    V = dev(np.stack([kv[:, 1] for kv in KV], 1))
    Qd = dev(Qs)
    lines = []
    vs = quality.variants(Qd[:T], K[:T], V[:T])
    runs = [(name, Rk, Rv, c, None) for name, (Rk, Rv, c) in vs.items()]
    Rk, Rv, c = vs["oscar"]
    # OSCAR's rotation plus Lloyd-Max codebooks calibrated on the same calibration keys and values
    runs.append(("oscar_lloyd_max", Rk, Rv, c, quality.lloyd_max_codebooks(K[:T], V[:T], Rk, Rv, c)))
    for name, Rk, Rv, c, cbs in runs:
        cbk, cbv = (None, None) if cbs is None else cbs
        kl, err = quality.measure(K[T:], V[T:], Qd[T], Rk, Rv, [c] * HKV, [c] * HKV, codebook_k=cbk,
                                  codebook_v=cbv)
        lines.append({"metric": "attention quality vs exact BF16 attention (score KL, relative output error)",
                      "variant": name, "score_kl": kl, "output_rel_sq_error": err, "clip": c,
                      "workload": "qwen3-8b-layer, calibration-style synthetic activations, 4,416-token context",
                      "data": "synthetic"})
    return lines


def other_workload(args):
    import numpy as np
    import torch
    import bit_rotated_kv_02_gb300 as ok
    import synth
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs") or 6800.0
    if args.workload == "bf16-compare":
        return bf16_compare(args, peak)
    if args.workload == "shared-prefix":
        return shared_prefix(args, peak)
    if args.workload == "quality":
        return quality_workload(args)
    if args.workload == "codebook":
        return codebook_compare(args, peak)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4242)
    lines = []
    if args.workload == "bulk":
        wl = synth.BULK_128K
        N, Hkv = wl.context[0], wl.num_kv_heads
        chan = torch.from_numpy(synth.outlier_channels(wl.seed, Hkv, D, wl.n_outliers).astype(np.int64)).cuda()
        K, V = _gpu_kv(gen, N, Hkv, chan), _gpu_kv(gen, N, Hkv, chan)
        Rk, Rv = _gpu_rotations(ok, Hkv, D, 10), _gpu_rotations(ok, Hkv, D, 50)
        clip = torch.full((Hkv,), 0.9, device="cuda")
        out = [ok.oscar_quantize_kv(K, Rk, clip, 128), ok.oscar_quantize_kv(V, Rv, clip, 128)]

        def step():
            ok.oscar_quantize_kv(K, Rk, clip, 128, *out[0])
            ok.oscar_quantize_kv(V, Rv, clip, 128, *out[1])
        ms = _time(step, max(3, args.steps), max(3, args.warmup))
        byts = 2 * (N * Hkv * D * 2 + N * Hkv * (D // 4 + 4))
        lines.append({"metric": "bulk prefill quantize: tokens/s (K and V of all KV heads)", "value": N / (ms * 1e-3),
                      "unit": "tokens/s", "ms_per_step": ms, "workload": wl.name,
                      "config": {"tokens": N, "num_kv_heads": Hkv, "head_dim": D, "group_size": 128, "clip": 0.9,
                                 "l2": "inputs 537 MB > L2"},
                      "roofline": {"bound": "hbm", "achieved": byts / (ms * 1e-3) / 1e9, "peak": peak,
                                   "frac": byts / (ms * 1e-3) / 1e9 / peak, "unit": "GB/s",
                                   "algorithmic_bytes": byts,
                                   "flops_fp32_rotation": 2.0 * 2 * N * Hkv * D * D,
                                   "tensor_pipe_pct_ncu": 19.5,
                                   "note": "tensor-pipe share from the ncu capture in profiles/quant_tc_kernel_bulk128k.md"},
                      "cpu_baseline": None if args.no_cpu_baseline else run_cpu_baseline(min(args.cpu_seconds, 5.0),
                                                                                         kind="bulk")})
        return lines
    if args.workload == "batch-sweep":
        for B in (1, 16, 64, 256):
            wl = synth.batch_sweep(B)
            L, Hq, Hkv = wl.context[0], wl.num_q_heads, wl.num_kv_heads
            hist = L - SINK - RECENT
            steps = max(3, min(args.steps, 200 if B < 64 else 40))
            pages = -(-(hist + 2 * steps + args.warmup + 8) // PAGE)  # the steps, then as many appends timed alone
            chan = torch.from_numpy(synth.outlier_channels(wl.seed, Hkv, D, 4).astype(np.int64)).cuda()
            Rk, Rv = _gpu_rotations(ok, Hkv, D, 100), _gpu_rotations(ok, Hkv, D, 200)
            clip = torch.full((Hkv,), 0.9)
            P = ok.Pool(B, Hq, Hkv, 128, B * pages, pages, Rk, Rv, clip, clip)
            P.set_page_table(torch.randperm(B * pages, generator=gen, device="cuda").to(torch.int32).reshape(B, pages))
            for b in range(B):
                ok.oscar_prefill_pool(P, b, _gpu_kv(gen, L, Hkv, chan), _gpu_kv(gen, L, Hkv, chan))
            q = (torch.randn((B, Hq, D), generator=gen, device="cuda") * 3).to(torch.bfloat16)
            kn, vn = _gpu_kv(gen, B, Hkv, chan), _gpu_kv(gen, B, Hkv, chan)
            out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
            ws = torch.empty(ok.oscar_decode_workspace_size(P), dtype=torch.uint8, device="cuda")

            def step():
                ok.oscar_decode_step(P, kn, vn, q, out=out, ws=ws)
            ms = _time(step, steps, max(3, min(args.warmup, 20)))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                ok.oscar_append_kv(P, kn, vn)
            e1.record()
            torch.cuda.synchronize()
            dem_ms = e0.elapsed_time(e1) / steps
            assert P.err() == 0, hex(P.err())
            byts = B * (hist * Hkv * 2 * (D // 4 + 4) + (SINK + RECENT) * Hkv * 2 * D * 2)
            lines.append({"metric": "decode step (append+demote + attention): KV tokens/s", "batch": B,
                          "value": B * L / (ms * 1e-3), "unit": "KV tokens/s", "decode_steps_per_s": 1e3 / ms,
                          "ms_per_step": ms, "workload": wl.name,
                          "demote": {"ms_per_call": dem_ms, "tokens_per_s": B / (dem_ms * 1e-3)},
                          "step_gbs": byts / (ms * 1e-3) / 1e9, "frac_of_peak": byts / (ms * 1e-3) / 1e9 / peak})
            del P, ws
            torch.cuda.empty_cache()
        return lines
    # mixed long-context batch (group 32, per-head clip ratios in [0.8, 1.0])
    wl = synth.mixed_long()
    Hq, Hkv, B = wl.num_q_heads, wl.num_kv_heads, wl.batch
    lens = list(wl.context)
    pages_b = [-(-(max(L - SINK - RECENT, 0) + 64) // PAGE) for L in lens]
    chan = torch.from_numpy(synth.outlier_channels(wl.seed, Hkv, D, 4).astype(np.int64)).cuda()
    Rk, Rv = _gpu_rotations(ok, Hkv, D, 300), _gpu_rotations(ok, Hkv, D, 400)
    ck = torch.from_numpy(synth.clip_ratios(wl.seed, Hkv, 0.8, 1.0))
    cv = torch.from_numpy(synth.clip_ratios(wl.seed + 1, Hkv, 0.8, 1.0))
    mp = max(pages_b)
    P = ok.Pool(B, Hq, Hkv, 32, sum(pages_b), mp, Rk, Rv, ck, cv)
    perm = torch.randperm(sum(pages_b), generator=gen, device="cuda").to(torch.int32).cpu()
    pt = torch.full((B, mp), -1, dtype=torch.int32)
    o = 0
    for b, n in enumerate(pages_b):
        pt[b, :n] = perm[o:o + n]
        o += n
    P.set_page_table(pt)
    for b, L in enumerate(lens):
        ok.oscar_prefill_pool(P, b, _gpu_kv(gen, L, Hkv, chan), _gpu_kv(gen, L, Hkv, chan))
    q = (torch.randn((B, Hq, D), generator=gen, device="cuda") * 3).to(torch.bfloat16)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(ok.oscar_decode_workspace_size(P), dtype=torch.uint8, device="cuda")
    ms = _time(lambda: ok.oscar_decode_attention(P, q, out=out, ws=ws), max(3, min(args.steps, 100)), 5)
    # the history kernel alone: CUDA events around it (on the call's stream) in a loop of calls
    lib = ok.lib()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for ev in evs:   # record once so that the CUDA events exist (the library records them again)
        ev[0].record()
        ev[1].record()
    torch.cuda.synchronize()
    for ev in evs:
        lib.oscar_profile_events(0, C.c_void_p(ev[0].cuda_event), C.c_void_p(ev[1].cuda_event))
        ok.oscar_decode_attention(P, q, out=out, ws=ws)
    torch.cuda.synchronize()
    hist_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    assert P.err() == 0, hex(P.err())
    hist = sum(max(L - SINK - RECENT, 0) for L in lens)
    ng = D // 32
    hist_byts = hist * Hkv * 2 * (D // 4 + 2 * 2 * ng) + sum(pages_b) * 4   # codes + scale/zero + page table
    byts = hist_byts + B * (SINK + RECENT) * Hkv * 2 * D * 2
    lines.append({"metric": "decode attention: KV tokens/s", "value": sum(lens) / (ms * 1e-3), "unit": "KV tokens/s",
                  "ms_per_step": ms, "workload": wl.name, "lengths": lens,
                  "gbs": byts / (ms * 1e-3) / 1e9, "frac_of_peak": byts / (ms * 1e-3) / 1e9 / peak,
                  "roofline": {"bound": "hbm", "kernel": f"tc::hist_kernel<{Hq // Hkv}, {ng}> (INT2 history, tcgen05)",
                               "achieved": hist_byts / (hist_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                               "frac": hist_byts / (hist_ms * 1e-3) / 1e9 / peak,
                               "algorithmic_bytes_per_launch": hist_byts, "mean_launch_us": hist_ms * 1e3,
                               "timed_launches": len(evs)}})
    return lines


def main():
    args = parse()
    if args.cpu_baseline_child:
        if args.cpu_kind == "bulk":
            print(json.dumps(cpu_bulk_child(args.cpu_seconds)))
        elif args.cpu_kind == "demote":
            print(json.dumps(cpu_demote_child(args.cpu_seconds)))
        else:
            print(json.dumps(cpu_baseline_child(args.cpu_seconds, args.cpu_cores)))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            # W untimed + K timed oracle steps, each one decode step of the sample (1/8 of the layer)
            times, ctx = oracle_sample_steps(args.warmup + args.steps)
            times, ctx = times[args.warmup:], ctx[args.warmup:]
            sec = sum(times)
            val = sum(ctx) / sec / HKV if sec > 0 else None
            cpu = {"value": val, "unit": "KV tokens/s", "cores": 1, "kind": "oracle",
                   "sample": f"{SAMPLE_NOTE}; each step of this line is one such sample step", "seconds": round(sec, 3)}
            print(json.dumps({"impl": "reference", "metric": METRIC, "value": val, "unit": "KV tokens/s",
                              "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
                              "ms_per_step": 1e3 * sec / max(len(times), 1), "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                              "config": {"workload": WORKLOAD + " (oracle sample: KV head 0 per step)"},
                              "cpu_baseline": cpu,
                              "e2e": {"value": val, "unit": "KV tokens/s", "h2d_bytes_per_step": 0,
                                      "d2h_bytes_per_step": 0}}))
        return

    import torch
    import torch.distributed as dist
    import __graft_entry__
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    __graft_entry__.build()
    import bit_rotated_kv_02_gb300 as ok
    from bit_rotated_kv_02_gb300 import _lib
    lib = ok.lib()
    if args.workload != "decode100k":
        if rank == 0:
            for line in other_workload(args):
                print(json.dumps(line))
        return

    NL = args.layers
    DEM_N = 200  # appends timed on their own after the run
    HOT_N, HOT_W = 500, 20  # the L2-hot steps (layer 0 only) after the run
    total = args.warmup + args.steps + args.e2e_steps + max(1, args.e2e_steps // 4) + DEM_N + max(50, args.roofline_launches)
    per_layer = -(-total // NL)
    layers = setup_layers(NL, per_layer + HOT_N + HOT_W + 8)
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(77 + rank)
    NQ = 64
    qs = (torch.randn((NQ, 1, HQ, D), generator=gen, device=dev) * 3).to(torch.bfloat16)
    kn = (torch.randn((NQ, 1, HKV, D), generator=gen, device=dev) * 3).to(torch.bfloat16)
    vn = (torch.randn((NQ, 1, HKV, D), generator=gen, device=dev) * 3).to(torch.bfloat16)
    outs = [torch.empty((1, HQ, D), dtype=torch.float32, device=dev) for _ in range(NL)]
    ws_bytes = ok.oscar_decode_workspace_size(layers[0], 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = C.c_void_p(stream.cuda_stream)
    scale = 1.0 / math.sqrt(D)
    appended = [0] * NL

    def step(i, ev=None):
        l = i % NL
        P = layers[l]
        if ev is not None:
            lib.oscar_profile_events(0, C.c_void_p(ev[0].cuda_event), C.c_void_p(ev[1].cuda_event))
        j = i % NQ
        st = lib.oscar_decode_step(P.ref, C.c_void_p(kn[j].data_ptr()), C.c_void_p(vn[j].data_ptr()),
                                   C.c_void_p(qs[j].data_ptr()), C.c_void_p(outs[l].data_ptr()), scale,
                                   C.c_void_p(ws.data_ptr()), ws_bytes, sp)
        if st:
            raise RuntimeError(lib.oscar_last_error_string().decode())
        appended[l] += 1
        return L_CTX + appended[l]      # tokens attended in this step

    # nvidia-smi samples SM clocks and throttle reasons every 20 ms from before the warm-up until after the
    # last GPU loop below: the timed region itself (steps x ~0.02-0.04 ms) is shorter than one sample
    # interval, so the line reports the samples of the whole window of GPU work around it.
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0] or "0"
    clocks = ClockSampler(gpu_index)
    time.sleep(0.3)
    wall0 = time.time()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tokens = 0
    t_start.record()
    for i in range(args.steps):
        tokens += step(args.warmup + i)
    t_stop.record()
    torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_stop)
    ms = max_over_ranks(ms)
    for P in layers:
        if P.err() != 0:
            raise RuntimeError(f"device error flags {P.err():#x}")

    # End to end through the public API with the step's inputs (q, k_new, v_new) in pinned host memory and its
    # result read back into pinned host memory, every step.  Main figure: the host buffers are passed to the
    # call itself, whose kernels read the inputs from and write the result to host memory over the host link
    # (no separate copy; the calls stay back to back on the stream).  Second figure: one explicit copy of the
    # inputs in and one of the result out per step around a call on device buffers.
    nq, nk = HQ * D, HKV * D
    hin = torch.empty(nq + 2 * nk, dtype=torch.bfloat16).pin_memory()
    hin[:nq].copy_(qs[0].reshape(-1).cpu()); hin[nq:nq + nk].copy_(kn[0].reshape(-1).cpu())
    hin[nq + nk:].copy_(vn[0].reshape(-1).cpu())
    hq, hk, hv = hin[:nq].view(1, HQ, D), hin[nq:nq + nk].view(1, HKV, D), hin[nq + nk:].view(1, HKV, D)
    hout = torch.empty((1, HQ, D), dtype=torch.float32).pin_memory()
    din = torch.empty_like(hin, device="cuda")
    dq, dk, dv = din[:nq].view(1, HQ, D), din[nq:nq + nk].view(1, HKV, D), din[nq + nk:].view(1, HKV, D)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    base = args.warmup + args.steps

    def e2e_loop(explicit: bool, n: int, first: int):
        tok = 0
        e0.record()
        for i in range(n):
            l = (first + i) % NL
            if explicit:
                din.copy_(hin, non_blocking=True)
                ok.oscar_decode_step(layers[l], dk, dv, dq, out=outs[l], ws=ws)
                hout.copy_(outs[l], non_blocking=True)
            else:
                ok.oscar_decode_step(layers[l], hk, hv, hq, out=hout, ws=ws)
            appended[l] += 1
            tok += L_CTX + appended[l]
        e1.record()
        torch.cuda.synchronize()
        return tok, max_over_ranks(e0.elapsed_time(e1))

    e2e_tokens, e2e_ms = e2e_loop(False, args.e2e_steps, base)
    e2x_steps = max(1, args.e2e_steps // 4)
    e2x_tokens, e2x_ms = e2e_loop(True, e2x_steps, base + args.e2e_steps)
    # the demotion + append kernel on its own (oscar_append_kv: one token per step, window full)
    e0.record()
    for i in range(DEM_N):
        ok.oscar_append_kv(layers[i % NL], dk, dv)
    e1.record()
    torch.cuda.synchronize()
    dem_ms = e0.elapsed_time(e1) / DEM_N
    # The dominant kernel on its own: CUDA events recorded on the step's stream immediately before and
    # after the attention kernel of each of these steps (an event between two kernels ends their
    # programmatic overlap, so these launches include the kernel's whole start-up; the layers rotate, so
    # every launch reads its history from HBM).
    RL = max(50, args.roofline_launches)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(RL)]
    for e2 in evs:              # torch creates the CUDA event on first record; create them all now
        for e in e2:
            e.record()
    torch.cuda.synchronize()
    rl_tokens = 0
    base = args.warmup + args.steps + args.e2e_steps + e2x_steps
    for i in range(RL):
        rl_tokens += step(base + i, evs[i])
    torch.cuda.synchronize()
    hist_ms = [e[0].elapsed_time(e[1]) for e in evs]
    rl_hist_avg = rl_tokens / RL - SINK - RECENT
    # L2-hot: the same step on one layer again and again, so that its ~58 MB stay in the 129 MB L2
    hot_tokens = 0

    def hot_step():
        st = lib.oscar_decode_step(layers[0].ref, C.c_void_p(kn[0].data_ptr()), C.c_void_p(vn[0].data_ptr()),
                                   C.c_void_p(qs[0].data_ptr()), C.c_void_p(outs[0].data_ptr()), scale,
                                   C.c_void_p(ws.data_ptr()), ws_bytes, sp)
        if st:
            raise RuntimeError(lib.oscar_last_error_string().decode())
        appended[0] += 1
        return L_CTX + appended[0]
    for _ in range(HOT_W):
        hot_step()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(HOT_N):
        hot_tokens += hot_step()
    e1.record()
    torch.cuda.synchronize()
    hot_ms = e0.elapsed_time(e1)
    clk = clocks.stop(wall0, time.time())
    clk["window"] = "warm-up, timed steps, e2e steps, demotion, roofline launches and L2-hot steps"
    for P in layers:
        if P.err() != 0:
            raise RuntimeError(f"device error flags {P.err():#x}")

    # algorithmic bytes per launch of the history kernel: codes + scale/zero + page-table entries + q of the
    # history; the step adds the BF16 sink and window (their own kernel), q, out, the new token and the
    # demoted row
    def hist_bytes_for(hist_tokens):
        b = hist_tokens * HKV * 2 * (D // 4 + 4 * (D // GROUP)) + 4 * math.ceil(hist_tokens / PAGE) + HQ * D * 2
        return b + ((SINK + RECENT) * HKV * 2 * D * 2 if ATTN_HAS_BF16 else 0)
    hist_tokens_avg = (tokens / args.steps) - SINK - RECENT
    step_bytes = hist_bytes_for(hist_tokens_avg) + (0 if ATTN_HAS_BF16 else (SINK + RECENT) * HKV * 2 * D * 2) \
        + HQ * D * 4 + HKV * 2 * D * 2 * 3 + HKV * 2 * (D // 4 + 4)
    attn_bytes = hist_bytes_for(rl_hist_avg)
    hist_mean_ms = statistics.mean(hist_ms)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    achieved = attn_bytes / (hist_mean_ms * 1e-3) / 1e9
    value = replica_throughput(tokens, ms, world)
    cpu = cpu_all = cpu_demote = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args.cpu_seconds)
        cpu_all = run_cpu_baseline(args.cpu_seconds, os.cpu_count() or 1)
        cpu_demote = run_cpu_baseline(min(args.cpu_seconds, 5.0), kind="demote")
    if rank == 0:
        rec = {
            "metric": METRIC, "value": value, "unit": "KV tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int2-kv/f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": D,
                       "group_size": GROUP, "clip": CLIP, "page_tokens": PAGE, "rotation": "covariance (GPU calib)",
                       "l2": f"{NL} rotating layer buffers ({NL * step_bytes / 1e6:.0f} MB >= 4x L2)",
                       "parallelism": f"replicas x{world}"},
            "decode_steps_per_s": world * args.steps / (ms * 1e-3),
            "bytes_per_step": step_bytes,
            "step_gbs": step_bytes * args.steps / (ms * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "kernel": ATTN_KERNEL,
                         "achieved": achieved, "peak": peak,
                         "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                         "frac_of_nominal_8tbs": achieved / 8000.0,
                         "traffic": traffic_from_profiles(ATTN_KERNEL_KEY, ATTN_SRC),
                         "algorithmic_bytes_per_launch": attn_bytes, "mean_launch_us": hist_mean_ms * 1e3,
                         "timed_launches": len(hist_ms),
                         "sampling": "a loop of decode steps after the run, CUDA events around each attention launch"},
            "demote": {"tokens_per_s": 1.0 / (dem_ms * 1e-3), "mean_call_us": dem_ms * 1e3,
                       "note": "oscar_append_kv (demotion + append kernel), timed on its own after the run; in "
                               "the decode step the attention kernel's sink CTAs perform the demotion",
                       "cpu_baseline": cpu_demote},
            "l2_hot": {"value": hot_tokens / (hot_ms * 1e-3), "unit": "KV tokens/s", "ms_per_step": hot_ms / HOT_N,
                       "steps": HOT_N, "note": "one layer's step repeated: its history stays in L2"},
            "e2e": {"value": replica_throughput(e2e_tokens, e2e_ms, world), "unit": "KV tokens/s",
                    "h2d_bytes_per_step": hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2,
                    "d2h_bytes_per_step": hout.numel() * 4, "steps": args.e2e_steps,
                    "transfer": "the call's kernels read q, k_new, v_new from pinned host memory and write the "
                                "output to pinned host memory over the host link",
                    "explicit_copies": {"value": replica_throughput(e2x_tokens, e2x_ms, world), "steps": e2x_steps,
                                        "transfer": "one host-to-device copy of the inputs and one device-to-host "
                                                    "copy of the output per step, around a call on device buffers"}},
            "gpu_launches": args.steps * 3,   # q rotation, attention (history + BF16 CTAs + demotion), merge
            "clocks": clk,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
        }
        print(json.dumps(rec))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
