#!/usr/bin/env python3
"""Decode-step benchmark of the persistent megakernel on B300.

Headline workload: the ~2B dense decoder (25 layers, d 2048, 16/4 heads, hd 128,
SwiGLU 8192, vocab 128256, BF16 weights ~N(0, 0.02)), batch 1, KV cache pre-filled
with seeded N(0, 1) BF16 to 8192 tokens on randomly permuted 16-token pages, greedy
decode whose tokens are fed back on the device; positions cycle through
8192..8447 (256 steps) so any --steps count repeats that workload.
Secondary (reported under "batch8"): the same model at batch 8, lengths uniform in
[512, 8192], sliding window 4096 on odd layers, two sequences replaced by fresh
512-token contexts every 64 steps (continuous batching).

One JSON line on rank 0. All inputs are synthetic and seeded; every step reads the
whole model (4.1 GB) and KV, far more than the 126 MB L2, so no L2 flush is needed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode tokens/s/GPU at batch 1 and 8; achieved HBM GB/s as % of 8 TB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
CTX = 8192
CYCLE = 256
PROFILE = os.path.join(ROOT, "profiles", "decode_step_dense2b_b1.md")
KERNEL_SOURCES = ["persistent_megakernel_05_b300/csrc/mk_kernel.cuh",
                  "persistent_megakernel_05_b300/csrc/mk_ptx.cuh",
                  "persistent_megakernel_05_b300/csrc/mk_api.cu"]


# ------------------------------------------------------------------ helpers
def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    try:
        txt = open(PROFILE).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    m_traffic = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", txt)
    if not m_hash or not m_traffic or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_traffic.group(1))


def algorithmic_bytes(cfg, batch, positions_per_layer_lo, positions, moe_union=None, kv_rows=None):
    """Bytes a decode step must move: every weight once (embedding: only the B rows; a
    MoE layer: its router and the experts in the union of the rows' routes, counts per
    layer in `moe_union`), the cached K/V rows attended (keys [lo, pos-1] per layer and
    row; `kv_rows` overrides the count, e.g. a shared prefix read once), the new K/V
    rows written, and the fp32 logits written."""
    d, hd, Hq, Hkv = cfg.d_model, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    attn = (Hq + 2 * Hkv) * hd * d + d * Hq * hd + 2 * d
    if cfg.is_moe:
        experts = sum(cfg.n_experts * d + u * 3 * cfg.expert_ffn_dim * d for u in moe_union)
        layer_params = cfg.n_layers * attn + experts
    else:
        layer_params = cfg.n_layers * (attn + 3 * cfg.ffn_dim * d)
    weights = 2 * (layer_params + cfg.vocab * d + d + batch * d)
    row = 2 * Hkv * hd * 2  # K and V of one position, one layer
    kv_read = 0
    if kv_rows is not None:
        kv_read = kv_rows * row
    else:
        for l in range(cfg.n_layers):
            for b in range(batch):
                kv_read += (positions[b] - positions_per_layer_lo[l][b]) * row
    kv_write = cfg.n_layers * batch * row
    return weights + kv_read + kv_write + batch * cfg.vocab * 4


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mk_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ replicas (N > 1)
def init_replicas(backend=None):
    """One process per GPU, each a full replica of the decode path (the step does not
    shard). Reads RANK / WORLD_SIZE / LOCAL_RANK from the environment and, for N > 1,
    joins the process group: NCCL on GPUs, gloo where there is no GPU. Returns
    (rank, world, local_rank, torch.distributed or None)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world <= 1:
        return rank, world, local, None
    import torch
    import torch.distributed as dist_mod
    if backend is None:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist_mod.init_process_group(backend)
    return rank, world, local, dist_mod


def max_over_ranks(x, dist, device="cpu"):
    """The largest of every rank's x (the slowest replica's time); x itself at N = 1."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, rows, steps, elapsed_ms):
    """Tokens per second of the whole job: every replica decodes `rows` tokens a step for
    `steps` steps, over the slowest replica's elapsed time."""
    return world * rows * steps / (elapsed_ms / 1000.0)


def emit(line, rank):
    """Rank 0 alone prints the JSON line."""
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ workloads
def setup_b1(cfg, W, device, steps_total, mk):
    import torch
    import synth
    npages = (CTX + CYCLE) // 16 + 2
    model = mk.DecodeModel(cfg, W, npages, device=device)
    synth.fill_normal_bf16_(model.kv(), 11)
    rng = np.random.default_rng(1)
    pt = synth.random_page_tables(rng, npages, [npages - 2], max_pages=npages - 2)
    dev = f"cuda:{device}"
    pos = torch.tensor([[CTX + (t % CYCLE)] for t in range(steps_total)], dtype=torch.int32, device=dev)
    toks = torch.zeros((steps_total + 1, 1), dtype=torch.int32, device=dev)
    toks[0, 0] = int(synth.random_tokens(rng, cfg.vocab, 1)[0])
    return {"model": model, "pt": torch.tensor(pt, device=dev), "pos": pos, "sl": pos + 1,
            "toks": toks, "pt_host": pt, "tok0": int(toks[0, 0]), "B": 1,
            "logits": torch.empty((1, cfg.vocab), dtype=torch.float32, device=dev)}


def setup_b8(cfg, W, device, steps_total, mk):
    """Batch 8 with ragged lengths, SWA on odd layers, continuous batching."""
    import torch
    import synth
    rng = np.random.default_rng(2)
    B = 8
    lens = rng.integers(512, CTX + 1, size=B).astype(np.int64)
    n_events = steps_total // 64
    max_len = CTX + steps_total + 16
    maxp = (max_len + 15) // 16 + 1
    fresh_pages = (512 + 4 * 64 + 16) // 16 + 1  # a refilled slot lives <= 4 events
    npages = B * maxp + 2 * n_events * fresh_pages + 16
    model = mk.DecodeModel(cfg, W, npages, device=device)
    synth.fill_normal_bf16_(model.kv(), 12)
    perm = list(rng.permutation(npages))
    pts, pos_rows, tok_fix = [], [], []
    cur_pt = np.full((B, maxp), -1, np.int32)
    for b in range(B):
        n = (int(lens[b]) + steps_total) // 16 + 1
        cur_pt[b, :n] = [perm.pop() for _ in range(n)]
    cur_pos = lens.copy()
    pts.append(cur_pt.copy())
    pt_index = []
    for t in range(steps_total):
        if t > 0 and t % 64 == 0:
            k = t // 64 - 1
            for slot in synth.replacement_slots(k, B):
                cur_pos[slot] = 512
                cur_pt[slot, :] = -1
                cur_pt[slot, :fresh_pages] = [perm.pop() for _ in range(fresh_pages)]
                tok_fix.append((t, slot, int(synth.random_tokens(rng, cfg.vocab, 1)[0])))
            pts.append(cur_pt.copy())
        pt_index.append(len(pts) - 1)
        pos_rows.append(cur_pos.copy())
        cur_pos = cur_pos + 1
    dev = f"cuda:{device}"
    toks = torch.zeros((steps_total + 1, B), dtype=torch.int32, device=dev)
    toks[0] = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device=dev)
    pos = torch.tensor(np.stack(pos_rows).astype(np.int32), device=dev)
    return {"model": model, "pts": torch.tensor(np.stack(pts), device=dev), "pt_index": pt_index,
            "pos": pos, "sl": pos + 1, "toks": toks, "tok_fix": tok_fix, "B": B,
            "pos_host": np.stack(pos_rows), "logits": torch.empty((B, cfg.vocab), dtype=torch.float32, device=dev)}


def run_device_loop(S, steps, warmup, cfg, batch8=False):
    """Device-resident decode loop; returns per-step kernel durations (ms) and total."""
    import torch
    model = S["model"]
    stream = torch.cuda.current_stream()
    fixes = {}
    for (t, slot, tok) in S.get("tok_fix", []):
        fixes.setdefault(t, []).append((slot, tok))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]

    def one(t, timed_idx=None):
        for (slot, tok) in fixes.get(t, []):
            S["toks"][t, slot] = tok
        pt = S["pts"][S["pt_index"][t]] if batch8 else S["pt"]
        if timed_idx is not None:
            starts[timed_idx].record(stream)
        model.step(S["toks"][t], S["pos"][t], pt, S["sl"][t], S["toks"][t + 1], S["logits"])
        if timed_idx is not None:
            ends[timed_idx].record(stream)

    for t in range(warmup):
        one(t)
    torch.cuda.synchronize()
    code, task = model.status()
    if code != 0:
        raise RuntimeError(f"warm-up step failed: status {code} task {task}")
    return one, starts, ends


def multi_step_loop(S, launches, warmup, n):
    """The same decode loop, n steps per launch (mk_decode_steps): each launch starts at
    the next position of the cycle and takes the previous launch's last token. Returns
    the mean milliseconds per step of the timed launches (CUDA events)."""
    import torch
    model = S["model"]
    dev = S["pos"].device
    total = warmup + launches
    starts = torch.tensor([[CTX + (n * i) % CYCLE] for i in range(total)], dtype=torch.int32, device=dev)
    sls = starts + 1
    bufs = [torch.zeros((n, 1), dtype=torch.int32, device=dev) for _ in range(2)]
    bufs[1][n - 1, 0] = S["tok0"]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def one(i):
        model.steps(n, bufs[(i + 1) % 2][n - 1], starts[i], S["pt"], sls[i], bufs[i % 2])

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    ev[0].record()
    for i in range(warmup, total):
        one(i)
    ev[1].record()
    torch.cuda.synchronize()
    code, task = model.status()
    if code != 0:
        raise RuntimeError(f"multi-step launches failed: status {code} task {task}")
    return ev[0].elapsed_time(ev[1]) / (launches * n)


def timed_region(one, warmup, steps, dist):
    import torch
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record()
    for i in range(steps):
        one(warmup + i, i)
    ev1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist:
        dist.barrier()
    return ev0.elapsed_time(ev1), wall


def e2e_loop(S, cfg, steps, warmup):
    """End to end through the public API with HOST buffers: every step calls
    mk_decode_step_host, which packs the step's inputs into one host-to-device copy, runs
    the step, and returns the device status word and the next tokens in one
    device-to-host copy; the host feeds the tokens to the following step. Returns the
    wall time (s) of the timed steps and the bytes copied each way per step."""
    import numpy as np
    model = S["model"]
    B = S["B"]
    pt_host = np.ascontiguousarray(S["pt_host"], dtype=np.int32)
    maxp = pt_host.shape[1]
    h_tok = np.zeros(B, dtype=np.int32)
    h_pos = np.zeros(B, dtype=np.int32)
    h_sl = np.zeros(B, dtype=np.int32)
    h_next = np.zeros(B, dtype=np.int32)
    h_tok[0] = S["tok0"]
    h2d = (3 * B + B * maxp) * 4        # tokens, positions, seq_lens, page table: one copy
    d2h = (4 + B) * 4                   # status word (+ 2 spare ints) and next tokens: one copy

    def one(t):
        p = CTX + (t % CYCLE)
        h_pos.fill(p)
        h_sl.fill(p + 1)
        model.step_host(h_tok, h_pos, pt_host, h_sl, h_next)
        h_tok[:] = h_next

    for t in range(warmup):
        one(t)
    t0 = time.perf_counter()
    for i in range(steps):
        one(warmup + i)
    wall = time.perf_counter() - t0
    return wall, h2d, d2h


# ------------------------------------------------------------------ the other model configs
def other_config(mk, local, name, B, ctx, steps, warmup, prefix_pages=0, private_pages=0, layers=0):
    """One more decode workload on its own seeded weights: B rows at context ~ctx (or
    rows sharing a page-aligned prefix run), greedy tokens fed back on device. Returns
    tokens/s, per-step time, and the achieved GB/s over the algorithmic bytes (a MoE
    layer counts the experts of its measured routed union)."""
    import torch
    import synth
    cfg = synth.CONFIGS[name]
    if layers:  # profiling only: the same shapes with fewer layers
        cfg = cfg.with_(name=f"{name}-{layers}l", n_layers=layers)
    dev = f"cuda:{local}"
    seed = {"moe-64x768": 3, "dense-8b": 4 if not prefix_pages else 5}[name]
    W = synth.make_weights(cfg, seed, device=dev)
    rng = np.random.default_rng(seed)
    total = warmup + steps
    if prefix_pages:
        npages = prefix_pages + B * private_pages + 2
        maxp = prefix_pages + private_pages
        pt = synth.prefix_shared_page_tables(rng, npages, B, prefix_pages, private_pages, maxp)
        start = np.array([prefix_pages * 16 + 256 + 100 * b for b in range(B)], np.int64)
    else:
        per = (ctx + total + 15) // 16 + 1
        npages = B * per + 2
        pt = synth.random_page_tables(rng, npages, [per] * B, per)
        start = np.full(B, ctx, np.int64)
    model = mk.DecodeModel(cfg, W, npages, device=local)
    if prefix_pages:  # the rows' shared prefix is read once per kv head for the batch
        model.set_shared_prefix([0] * B, [prefix_pages] * B)
    synth.fill_normal_bf16_(model.kv(), seed + 100)
    pos = torch.tensor(np.stack([start + t for t in range(total)]).astype(np.int32), device=dev)
    toks = torch.zeros((total + 1, B), dtype=torch.int32, device=dev)
    toks[0] = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device=dev)
    ptd = torch.tensor(pt, device=dev)
    sl = pos + 1

    def run(t0, n, union_log=None):
        for t in range(t0, t0 + n):
            model.step(toks[t], pos[t], ptd, sl[t], toks[t + 1], None)
            if union_log is not None:
                ptr, nbytes = mk.mk_debug_buffer(model.handle, mk.MK_BUF_MOE_UNION)
                src = torch.as_tensor(mk._CudaArray(ptr, (cfg.n_layers,), "<i4"), device=dev)
                union_log[t - t0].copy_(src, non_blocking=True)

    run(0, warmup)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    run(warmup, steps)
    ev1.record()
    torch.cuda.synchronize()
    code, task = model.status()
    if code != 0:
        raise RuntimeError(f"{name} B={B} steps failed: status {code} task {task}")
    ms = ev0.elapsed_time(ev1) / steps
    unions = None
    if cfg.is_moe:
        # replay the same steps (same tokens, positions, pages: the same routing) and log
        # each step's per-layer routed union
        log = torch.zeros((steps, cfg.n_layers), dtype=torch.int32, device=dev)
        run(warmup, steps, log)
        torch.cuda.synchronize()
        unions = log.cpu().numpy()
    row = 2 * cfg.n_kv_heads * cfg.head_dim * 2
    byts, naive = 0, 0
    for i in range(steps):
        p = [int(x) for x in pos[warmup + i].tolist()]
        lo = [[0] * B for _ in range(cfg.n_layers)]
        un = unions[i].tolist() if unions is not None else None
        if prefix_pages:
            shared = prefix_pages * 16
            rows = cfg.n_layers * (shared + sum(x - shared for x in p))
            byts += algorithmic_bytes(cfg, B, lo, p, un, kv_rows=rows)
        else:
            byts += algorithmic_bytes(cfg, B, lo, p, un)
        naive += algorithmic_bytes(cfg, B, lo, p, un)
    gbs = byts / steps / (ms / 1000.0) / 1e9
    out = {"tokens_per_s": round(B * 1000.0 / ms, 2), "ms_per_step": round(ms, 4), "steps": steps,
           "batch": B, "hbm_gbs": round(gbs, 1), "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
           "algorithmic_bytes_per_step": int(byts / steps)}
    if prefix_pages:
        out["naive_bytes_per_step"] = int(naive / steps)
        out["workload"] = (f"{name}, batch {B} sharing a {prefix_pages * 16}-token prefix page run "
                           f"(declared: read once per kv head), {private_pages * 16}-token private runs; "
                           f"prefix KV counted once in the bytes")
    else:
        out["workload"] = f"{name}, batch {B}, {ctx}-token seeded paged KV per row"
    if unions is not None:
        out["mean_routed_union_per_layer"] = round(float(unions.mean()), 2)
    model.close()
    del W
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU baseline (oracle)
def cpu_model() -> str:
    """The host CPU's model name (lscpu), or '' if unavailable."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return ""


def oracle_sample(cfg, W_cpu, kv_host, pt, budget_s=12.0, max_steps=16, B=1):
    """Times the CPU oracle, as it stands, on a bounded sample of the same workload:
    consecutive decode steps at positions 8192, 8193, ... until the budget is spent, on
    every core the process may use; then one step on a single thread."""
    import oracle
    om = oracle.OracleModel(cfg, W_cpu)
    threads = oracle.default_threads()
    tok = 1
    done, t_sum = 0, 0.0
    while done < max_steps and t_sum < budget_s:
        pos = CTX + done
        t0 = time.perf_counter()
        _, nx = om.decode_step(kv_host, [tok] * B, [pos] * B, np.repeat(pt[:1], B, 0), [pos + 1] * B,
                               nthreads=threads)
        t_sum += time.perf_counter() - t0
        tok = int(nx[0])
        done += 1
    pos = CTX + done
    t0 = time.perf_counter()
    om.decode_step(kv_host, [tok] * B, [pos] * B, np.repeat(pt[:1], B, 0), [pos + 1] * B, nthreads=1)
    t1 = time.perf_counter() - t0
    return {"value": B * done / t_sum, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "single_thread_value": B / t1, "cpu_model": cpu_model(),
            "sample": f"{done} consecutive decode steps of the dense-2b batch-{B} workload "
                      f"(context {CTX}..{CTX + done - 1}), {t_sum:.1f} s on {threads} threads, then "
                      f"step {CTX + done} on 1 thread ({t1:.1f} s); plain C fp32, OpenMP over output rows"}


def reference_arm(args, rank, world):
    """--impl reference: the CPU oracle on this arm's workload (rank 0 only)."""
    if rank != 0:
        return
    import torch
    import synth
    cfg = synth.DENSE_2B
    W = synth.make_weights(cfg, 1, device="cpu")
    npages = (CTX + CYCLE) // 16 + 2
    kv = torch.empty(synth.kv_pool_shape(cfg, npages), dtype=torch.bfloat16)
    synth.fill_normal_bf16_(kv, 11)
    kv_host = synth.bf16_bits(kv).copy()
    rng = np.random.default_rng(1)
    pt = synth.random_page_tables(rng, npages, [npages - 2], max_pages=npages - 2)
    import oracle
    om = oracle.OracleModel(cfg, W)
    threads = oracle.default_threads()
    # warm-up: W steps, as the repo arm; timed: up to K steps within a 90 s budget
    tok = 1
    for w in range(args.warmup):
        _, nx = om.decode_step(kv_host, [tok], [CTX + w], pt[:1], [CTX + w + 1], nthreads=threads)
        tok = int(nx[0])
    done, t0 = 0, time.perf_counter()
    while done < args.steps and time.perf_counter() - t0 < 90.0:
        pos = CTX + (done % CYCLE)
        _, nx = om.decode_step(kv_host, [tok], [pos], pt[:1], [pos + 1], nthreads=threads)
        tok = int(nx[0])
        done += 1
    el = time.perf_counter() - t0
    val = done / el
    sample = (f"{done} of {args.steps} requested decode steps of the dense-2b batch-1 workload "
              f"(90 s budget), plain C fp32 oracle, OpenMP over output rows")
    emit({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": world, "steps": done, "warmup": args.warmup,
        "ms_per_step": 1000.0 * el / max(done, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "dense-2b decoder, batch 1, 8192-token seeded paged KV, greedy decode",
                   "batch": 1, "context": CTX},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }, rank)


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-batch8", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the MoE and 8B lines")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run every workload's shapes with this many layers")
    ap.add_argument("--only", default="", choices=["", "moe_b1", "moe_b8", "dense8b_b1", "dense8b_b4_prefix"],
                    help="profiling only: run just this one of the other workloads (no headline line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank, world, local, dist = init_replicas()

    if args.impl == "reference":
        reference_arm(args, rank, world)
        if dist:
            dist.destroy_process_group()
        return

    import torch
    import synth
    from persistent_megakernel_05_b300 import build as mkbuild
    mkbuild.build()
    import persistent_megakernel_05_b300 as mk
    torch.cuda.set_device(local)
    extra_kw = {"moe_b1": dict(name="moe-64x768", B=1, ctx=4096, steps=128),
                "moe_b8": dict(name="moe-64x768", B=8, ctx=4096, steps=128),
                "dense8b_b1": dict(name="dense-8b", B=1, ctx=32768, steps=128),
                "dense8b_b4_prefix": dict(name="dense-8b", B=4, ctx=0, steps=128,
                                          prefix_pages=1024, private_pages=64)}
    if args.only:  # profiling only: one of the other workloads, --steps timed steps
        kw = dict(extra_kw[args.only], steps=args.steps)
        r = other_config(mk, local, warmup=args.warmup, layers=args.layers, **kw)
        emit({"only": args.only, "layers": args.layers or None, **r}, rank)
        return
    cfg = synth.DENSE_2B
    if args.layers:
        cfg = cfg.with_(name=f"dense-2b-{args.layers}l", n_layers=args.layers)
    W = synth.make_weights(cfg, 1, device=f"cuda:{local}")
    total = args.warmup + args.steps
    S = setup_b1(cfg, W, local, total, mk)
    one, starts, ends = run_device_loop(S, args.steps, args.warmup, cfg)
    with ClockSampler(local) as clk:
        elapsed_ms, wall = timed_region(one, args.warmup, args.steps, dist)
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    code, task = S["model"].status()
    if code != 0:
        raise RuntimeError(f"timed steps failed: status {code} task {task}")
    elapsed_ms = max_over_ranks(elapsed_ms, dist, f"cuda:{local}")
    ms = elapsed_ms / args.steps
    value = whole_job_value(world, 1, args.steps, elapsed_ms)
    lo = [[0] for _ in range(cfg.n_layers)]
    # positions of the timed steps (the decode loop's step t runs at CTX + t mod CYCLE)
    timed_pos = [CTX + (t % CYCLE) for t in range(args.warmup, args.warmup + args.steps)]
    algo = algorithmic_bytes(cfg, 1, lo, [float(np.mean(timed_pos))])
    kern_ms = statistics.mean(per)
    peak, peak_src = measured_peak()
    achieved = algo / (kern_ms / 1000.0) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6400 GB/s", "algorithmic_bytes_per_launch": int(algo),
            "kernel": "mk::decode_step_kernel<128, false>", "kernel_ms_mean": round(kern_ms, 4)}
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) BF16 weights, N(0,1) BF16 KV)",
        "config": {"workload": "dense-2b decoder (25 layers, d 2048, 16/4 heads, hd 128, ffn 8192, "
                               "vocab 128256), batch 1, 8192-token seeded paged KV (random pages), "
                               "greedy decode fed back on device, positions 8192..8447 cycling",
                   "batch": 1, "context": CTX, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "inputs larger than L2 (4.1 GB weights + 0.42 GB KV read per step)"},
        "step_ms": {"median": round(statistics.median(per), 4),
                    "p10": round(float(np.percentile(per, 10)), 4),
                    "p90": round(float(np.percentile(per, 90)), 4)},
        "hbm_gbs": round(achieved, 1), "pct_of_8tbs": round(100 * achieved / NOMINAL_HBM_GBS, 2),
        "roofline": roof, "clocks": clk.summary(), "gpu_launches": args.steps,
    }
    # the same loop with 16 steps per launch (tokens fed back inside the launch)
    ms16 = multi_step_loop(S, max(1, args.steps // 16), 1, 16)
    ach16 = algo / (ms16 / 1000.0) / 1e9
    out["multi_step"] = {"steps_per_launch": 16, "ms_per_step": round(ms16, 4),
                         "tokens_per_s": round(world * 1000.0 / ms16, 2), "hbm_gbs": round(ach16, 1),
                         "frac_of_measured_peak": round(ach16 / peak, 4),
                         "workload": "the headline workload through mk_decode_steps"}
    # batch 8 (secondary workload)
    if not args.no_batch8:
        cfg8 = synth.DENSE_2B_SWA.with_(n_layers=cfg.n_layers)
        # the configuration's 256 decode steps (at least), so that the replacement events
        # (every 64 steps) fall inside the timed window whatever --steps is
        steps8 = min(max(args.steps, 256), 512)
        S8 = setup_b8(cfg8, W, local, args.warmup + steps8, mk)
        one8, st8, en8 = run_device_loop(S8, steps8, args.warmup, cfg8, batch8=True)
        el8, _ = timed_region(one8, args.warmup, steps8, dist)
        el8 = max_over_ranks(el8, dist, f"cuda:{local}")
        code, task = S8["model"].status()
        if code != 0:
            raise RuntimeError(f"batch-8 steps failed: status {code} task {task}")
        per8 = [s.elapsed_time(e) for s, e in zip(st8, en8)]
        bytes8 = 0
        sl = cfg8.layer_is_sliding()
        for i in range(steps8):
            p = S8["pos_host"][args.warmup + i]
            los = [[max(0, int(x) - cfg8.sliding_window + 1) if sl[l] else 0 for x in p]
                   for l in range(cfg8.n_layers)]
            bytes8 += algorithmic_bytes(cfg8, 8, los, [int(x) for x in p])
        ach8 = bytes8 / (sum(per8) / 1000.0) / 1e9
        events = sum(1 for t in range(args.warmup, args.warmup + steps8) if t > 0 and t % 64 == 0)
        out["batch8"] = {"value": round(whole_job_value(world, 8, steps8, el8), 2), "unit": "tokens/s",
                         "steps": steps8, "ms_per_step": round(el8 / steps8, 4),
                         "replacement_events_timed": events,
                         "hbm_gbs": round(ach8, 1), "pct_of_8tbs": round(100 * ach8 / NOMINAL_HBM_GBS, 2),
                         "frac_of_measured_peak": round(ach8 / peak, 4),
                         "workload": "dense-2b, batch 8, lengths U[512, 8192], SWA 4096 on odd layers, "
                                     "2 sequences replaced by fresh 512-token contexts every 64 steps"}
        S8["model"].close()
        del S8
    # the MoE and 8B configs (secondary lines; each on its own seeded weights)
    if not args.no_extra:
        del W
        S["model"].close()
        torch.cuda.empty_cache()
        extra = {}
        for key, kw in extra_kw.items():
            extra[key] = other_config(mk, local, warmup=args.warmup, layers=args.layers, **kw)
            extra[key]["frac_of_measured_peak"] = round(extra[key]["hbm_gbs"] / peak, 4)
        out["other_configs"] = extra
        W = synth.make_weights(cfg, 1, device=f"cuda:{local}")
        S = setup_b1(cfg, W, local, total, mk)
    # end to end through host buffers
    if not args.no_e2e:
        e2e_steps = min(args.steps, 512)
        wall, h2d, d2h = e2e_loop(S, cfg, e2e_steps, args.warmup)
        wall = max_over_ranks(wall, dist, f"cuda:{local}")
        val = whole_job_value(world, S["B"], e2e_steps, 1000.0 * wall)
        out["e2e"] = {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                      "path": "host arrays -> mk_decode_step_host (one H2D copy of the packed inputs, the step, one D2H copy of status + next tokens, synchronous) -> next token fed back"}
    # CPU baseline: the oracle on the host cores (rank 0, N = 1 only)
    if rank == 0 and world == 1 and not args.no_cpu:
        W_cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in W.items() if k != "layers"}
        W_cpu["layers"] = [{k: v.cpu() for k, v in L.items()} for L in W["layers"]]
        kv_host = synth.bf16_bits(S["model"].kv()).copy()
        out["cpu_baseline"] = oracle_sample(cfg, W_cpu, kv_host, S["pt_host"])
    S["model"].close()
    emit(out, rank)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
