#!/usr/bin/env python
"""Decode benchmark of the GGUF decoder token step on GB300.

Workload (default): the llama-3-8B-shaped decoder with Q8_0 weights (32 layers, hidden 4096,
32 Q / 8 KV heads of 128, FFN 14336, vocab 128256), batch size 1, decoding at context 8192: the KV
cache is filled with N(0,1) keys/values (seed 2) for the first 8191 - warmup positions, then
`warmup` untimed and `steps` timed decode steps run, so every timed step reads >= 8192 keys.
Weights are seeded synthetic GGUF bytes (seed 0), token ids uniform (seed 1). One step = one
token through the whole forward (embed, 32 layers, final norm, logits, argmax).

Printed: one JSON line with decode tokens/s (device-resident inputs, CUDA events on the library's
stream), the end-to-end tokens/s through the public Python API (host token in, host logits out,
copies inside the timed region), the roofline of the dominant kernel (the weight-streaming GEMV)
inside the timed step against the measured HBM copy bandwidth (its share of a profiled pass times
the timed ms per step), the whole step's HBM bytes per token, SM clocks sampled during the timed
region, the CPU oracle's tokens/s on the host cores, (key "decode_kv_f16") the same decode with
the optional f16 KV cache, (key "decode_configs") the other decode workloads -- qwen3-0.6B f16 at
128 / 1024 / 4096 keys, gemma3-1B f16 at 8192 keys (window 512 on 5 of 6 layers), qwen2-7B Q4_0
after a 2048-token bulk prefill -- each with its step bytes, in-step GEMV roofline and fraction of
the 70 %-of-8-TB/s target, and (key "prefill") the bulk-prefill tokens/s of the qwen2-7B-shaped Q4_0
decoder on a 2048-token prompt, with resident operand planes and converting them per forward, and
the tensor-core rate of its matmuls against the measured bf16 peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

# DRAM traffic of the GEMV per algorithmic byte, from an ncu --set full capture of a small case of the
# same kernel (profiles/gemv_q8_0_llama3_8b_2layers_ctx1024_full.md: dram__bytes_read.sum +
# dram__bytes_write.sum = 172.59 MB over three launches whose algorithmic bytes total 169.54 MB).
# Traffic grows in proportion to the rows streamed, so the bench scales it to its own launches.
# Keyed by the sha256 prefix of the kernel sources it was measured on (k_gemv.cu + gemv_dev.cuh):
# null once the kernel changes.
GEMV_TRAFFIC_RATIO = {"141c4e285e121f19": 172.591872 / 169.541632}


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b", choices=sorted(synth.CONFIGS))
    ap.add_argument("--ctx", type=int, default=8192, help="decode context length")
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--profile-steps", type=int, default=16)
    ap.add_argument("--cpu-steps", type=int, default=4, help="oracle decode steps for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-workload", default="qwen2_7b", choices=sorted(synth.CONFIGS))
    ap.add_argument("--prefill-tokens", type=int, default=2048)
    ap.add_argument("--prefill-reps", type=int, default=3)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--kv-f16-steps", type=int, default=256, help="timed decode steps with the f16 KV cache (0: skip)")
    ap.add_argument("--no-decode-configs", action="store_true",
                    help="skip the other decode workloads (qwen3-0.6B at 128/1024/4096 keys, gemma3-1B at 8192, "
                         "qwen2-7B after a 2048-token bulk prefill)")
    ap.add_argument("--config-steps", type=int, default=64, help="timed decode steps per extra decode workload")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling cases only; not a bench configuration)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(ms, world, torch, device):
    """The slowest rank's time (ms) of the timed region, then a barrier: the job is done when its
    last replica is. With one rank, ms itself."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t.item())


def job_throughput(steps, world, ms):
    """Whole-job tokens/s of `world` replicas that each ran `steps` decode steps in `ms` (the
    slowest rank's time): weak scaling, every replica decodes its own tokens."""
    return steps * world / (ms / 1000.0)


def kv_fill_all(cfg, n_pos):
    return [synth.kv_fill(cfg, layer, n_pos, seed=2) for layer in range(cfg.n_layer)]


def decode_bytes_per_token(cfg, ctx_mean, kv_elt=4):
    """Algorithmic HBM bytes of one decode step: every weight once (incl. the logits matrix, even
    when tied), the KV cache over the allowed keys (kv_elt bytes per element: 4 for the f32 cache,
    2 for the f16 one), norms, one embedding row."""
    wb = synth.weight_bytes(cfg)
    if cfg.tied:
        wb += synth.tensor_nbytes(synth.DTYPE_IDS[cfg.wtype], cfg.n_vocab * cfg.n_embd)
    # the embedding matrix is not streamed: only one row is read
    emb = synth.tensor_nbytes(synth.DTYPE_IDS[cfg.wtype], cfg.n_vocab * cfg.n_embd)
    wb -= emb
    wb += synth.tensor_nbytes(synth.DTYPE_IDS[cfg.wtype], cfg.n_embd)
    kv = 0.0
    for layer in range(cfg.n_layer):
        glob = cfg.sliding_window == 0 or (cfg.arch == "gemma3" and layer % 6 == 5)
        n = ctx_mean if glob else min(ctx_mean, cfg.sliding_window)
        kv += 2.0 * cfg.n_head_kv * cfg.head_dim * kv_elt * n
    return float(wb + kv), float(wb), float(kv)


# Decode tok/s at 70 % of 8 TB/s for each workload (bytes per token at that context, f32 KV).
TARGET_70 = {("qwen3_0_6b", 128): 4584, ("qwen3_0_6b", 1024): 3924, ("qwen3_0_6b", 4096): 2627,
             ("llama3_8b", 8192): 553, ("qwen2_7b", 2048): 1325, ("gemma3_1b", 8192): 2679}


def in_step_roofline(prof, profile_steps, ms_per_step, peak_gbs, kind="gemv"):
    """HBM roofline of one kernel kind inside the graph-replayed step: its share of the profiled
    device time (eager pass, one event pair per kernel group) times the timed ms per step gives
    its time per step; its algorithmic bytes per step over that time is its achieved rate. The
    per-launch figures divide both by the kind's launches per step."""
    k = prof.get(kind)
    tot = sum(v["ms"] for v in prof.values())
    if not k or not tot or not k["bytes"]:
        return None
    share = k["ms"] / tot
    t_step = share * ms_per_step                                  # ms of the step spent in this kind
    launches = k["launches"] / profile_steps
    bytes_step = k["bytes"] / profile_steps
    gbs = bytes_step / (t_step / 1000.0) / 1e9
    return {"share_of_step": share, "ms_per_step": t_step, "launches_per_step": launches,
            "bytes_per_step": bytes_step, "bytes_per_launch": bytes_step / launches if launches else None,
            "us_per_launch": 1000.0 * t_step / launches if launches else None,
            "achieved": gbs, "frac": gbs / peak_gbs}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def host_cpu() -> str:
    """This host's processor: model name (x86) or implementer/part (Arm) from /proc/cpuinfo, the
    architecture and the logical core count."""
    import platform
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = dict(l.split(":", 1) for l in f.read().splitlines() if ":" in l)
        info = {k.strip(): v.strip() for k, v in info.items()}
        # Arm cores report an implementer and part number; name the common server parts
        arm_parts = {("0x41", "0xd4f"): "Arm Neoverse-V2", ("0x41", "0xd40"): "Arm Neoverse-V1",
                     ("0x41", "0xd0c"): "Arm Neoverse-N1", ("0x41", "0xd49"): "Arm Neoverse-N2"}
        arm = (info.get("CPU implementer"), info.get("CPU part"))
        model = info.get("model name") or arm_parts.get(arm) or " ".join(
            f"{k} {info[k]}" for k in ("CPU implementer", "CPU part") if k in info)
    except (OSError, ValueError):
        pass
    return f"{model or 'unknown'} ({platform.machine()}, {os.cpu_count()} logical cores)"


def cpu_baseline(cfg, W, ctx, n_steps):
    """The oracle as it stands, on this host's cores: n_steps decode steps at the same context."""
    import oracle
    cores = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    P = ctx - 1
    m = oracle.model_from_synth(cfg, W, P + n_steps + 1)
    for layer, (k, v) in enumerate(kv_fill_all(cfg, P)):
        m.write_kv(layer, 0, k, v)
    m.set_kv_len(P)
    toks = synth.tokens(cfg, n_steps, seed=1)
    t0 = time.perf_counter()
    for i in range(n_steps):
        m.forward(toks[i:i + 1], P + i)
    dt = time.perf_counter() - t0
    m.close()
    return {"value": n_steps / dt, "unit": "tok/s", "cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle",
            "host": host_cpu(),
            "sample": f"{n_steps} decode steps of the full {cfg.name} model at context {ctx} (KV injected), "
                      f"f32 values / f64 reductions, OpenMP over matmul rows"}


def run_reference(args):
    """The reference arm: the CPU oracle timed on the host cores, same workload, metric and unit."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    cfg = synth.CONFIGS[args.workload]
    W = synth.make_model(cfg, seed=0)
    cores = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    budget_s = 150.0
    P = args.ctx - 1 - max(1, min(args.warmup, 2))
    m = oracle.model_from_synth(cfg, W, args.ctx + args.steps + 4)
    for layer, (k, v) in enumerate(kv_fill_all(cfg, P)):
        m.write_kv(layer, 0, k, v)
    m.set_kv_len(P)
    toks = synth.tokens(cfg, args.steps + 4, seed=1)
    pos = P
    t0 = time.perf_counter()
    nw = max(1, min(args.warmup, 2))
    for i in range(nw):
        m.forward(toks[i:i + 1], pos)
        pos += 1
    per = (time.perf_counter() - t0) / nw
    steps = max(1, min(args.steps, int(budget_s / max(per, 1e-6))))
    t0 = time.perf_counter()
    for i in range(steps):
        m.forward(toks[nw + i:nw + i + 1], pos)
        pos += 1
    dt = time.perf_counter() - t0
    value = steps / dt
    sample = (f"{steps} of {args.steps} requested decode steps (capped to ~{budget_s:.0f} s), full {cfg.name} model "
              f"at context {args.ctx}, {nw} warm-up step(s)")
    line = {"impl": "reference", "metric": "decode tok/s (bs=1)", "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": steps, "warmup": nw, "ms_per_step": 1000 * dt / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{cfg.name} Q8_0 decode bs=1 at context {args.ctx}", "batch": 1,
                       "context": args.ctx},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
                             "kind": "oracle", "sample": sample, "host": host_cpu()},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_decode_kv_f16(args, syn, torch, cfg, W, ctx, peaks):
    """The same decode workload with the cache stored as f16 (option kv_f16): the attention reads
    half the bytes. Its parity is against the oracle's f16-KV configuration (tests)."""
    K, Wm = args.kv_f16_steps, 8
    P0 = ctx - 1 - Wm
    max_ctx = ctx + K + 8
    stream = torch.cuda.Stream()
    m = syn.Model(syn.read_archdef(cfg.arch), synth.metadata(cfg, max_ctx), max_ctx, arch=cfg.arch,
                  stream=stream.cuda_stream)
    m.set_option("kv_f16", 1)
    m.load_tensors(W)
    m.finalize()
    for layer, (k, v) in enumerate(kv_fill_all(cfg, P0)):
        m.write_kv(layer, 0, k, v)
    toks = synth.tokens(cfg, Wm + K + 2, seed=1)
    dtok = torch.from_numpy(toks.astype(np.int32)).cuda()
    darg = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = syn.TOKENS_ON_DEVICE | syn.ARGMAX_ON_DEVICE
    pos = P0
    for i in range(Wm):
        m.forward_raw(dtok.data_ptr() + 4 * i, 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
    stream.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pos_t0 = pos
    ev0.record(stream)
    for i in range(K):
        m.forward_raw(dtok.data_ptr() + 4 * (Wm + i), 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
    ev1.record(stream)
    ev1.synchronize()
    ms = ev0.elapsed_time(ev1)
    m.close()
    bpt, _, kvb = decode_bytes_per_token(cfg, (pos_t0 + pos_t0 + K) / 2.0, kv_elt=2)
    gbs = bpt * (K / (ms / 1000.0)) / 1e9
    return {"value": K / (ms / 1000.0), "unit": "tok/s", "ms_per_step": ms / K, "steps": K, "kv_cache": "f16",
            "step_hbm": {"bytes_per_token": bpt, "kv_bytes": kvb, "achieved_gbs": gbs,
                         "frac_of_measured": gbs / peaks["hbm_gbs"], "frac_of_8tbs": gbs / 8000.0}}


def oracle_decode_rate(cfg, W, ctx, budget_s=8.0, max_steps=4):
    """The oracle on the host cores: a few decode steps at context ctx (KV injected), at most
    max_steps and about budget_s seconds."""
    import oracle
    cores = os.cpu_count() or 1
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    P = ctx - 1
    m = oracle.model_from_synth(cfg, W, P + max_steps + 1)
    for layer, (k, v) in enumerate(kv_fill_all(cfg, P)):
        m.write_kv(layer, 0, k, v)
    m.set_kv_len(P)
    toks = synth.tokens(cfg, max_steps, seed=1)
    n, t0 = 0, time.perf_counter()
    while n < max_steps and (n == 0 or time.perf_counter() - t0 < budget_s):
        m.forward(toks[n:n + 1], P + n)
        n += 1
    dt = time.perf_counter() - t0
    m.close()
    return {"value": n / dt, "unit": "tok/s", "cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle",
            "sample": f"{n} decode step(s) of the full {cfg.name} model at context {ctx} (KV injected)"}


def bench_decode_configs(args, syn, torch, name, ctxs, peaks, cpu_ctx=None, bulk_prompt=0):
    """bench_decode_config for several contexts of one workload on one loaded model (the KV cache is
    reset between them)."""
    cfg = synth.CONFIGS[name]
    W = synth.make_model(cfg, seed=0)
    stream = torch.cuda.Stream()
    max_ctx = max(ctxs) + args.config_steps + 8 + args.profile_steps + 8
    m = syn.Model(syn.read_archdef(cfg.arch), synth.metadata(cfg, max_ctx), max_ctx, arch=cfg.arch,
                  stream=stream.cuda_stream)
    m.load_tensors(W)
    m.finalize()
    out = []
    for ctx in ctxs:
        m.reset_kv()
        r = bench_decode_config(args, syn, torch, m, stream, cfg, ctx, peaks, bulk_prompt=bulk_prompt)
        if ctx == cpu_ctx and not args.no_cpu_baseline:
            r["cpu_baseline"] = oracle_decode_rate(cfg, W, ctx)
        out.append(r)
    m.close()
    del W
    return out


def bench_decode_config(args, syn, torch, m, stream, cfg, ctx, peaks, bulk_prompt=0):
    """Decode tok/s of one more workload at context ctx on a loaded model with an empty cache: KV
    injected for the first positions (or, with bulk_prompt > 0, a bulk prefill of that many prompt
    tokens), then warm-up and timed steps with device-resident tokens; a profiled pass for the
    in-step GEMV roofline."""
    name = cfg.name
    K, Wm = args.config_steps, 8
    toks = synth.tokens(cfg, ctx + K + Wm + args.profile_steps + 8, seed=1)
    dtok = torch.from_numpy(toks.astype(np.int32)).cuda()
    darg = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = syn.TOKENS_ON_DEVICE | syn.ARGMAX_ON_DEVICE
    if bulk_prompt:
        m.forward_raw(dtok.data_ptr(), bulk_prompt, 0, 0, darg.data_ptr(), flags)
        pos = bulk_prompt
    else:
        pos = ctx - 1 - Wm
        for layer, (k, v) in enumerate(kv_fill_all(cfg, pos)):
            m.write_kv(layer, 0, k, v)
    for _ in range(Wm):
        m.forward_raw(dtok.data_ptr() + 4 * pos, 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
    stream.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pos_t0 = pos
    ev0.record(stream)
    for _ in range(K):
        m.forward_raw(dtok.data_ptr() + 4 * pos, 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
    ev1.record(stream)
    ev1.synchronize()
    ms = ev0.elapsed_time(ev1) / K
    m.set_option("profile", 1)
    for _ in range(args.profile_steps):
        m.forward_raw(dtok.data_ptr() + 4 * pos, 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
    stream.synchronize()
    prof = m.profile(reset=True)
    m.set_option("profile", 0)
    ctx_mean = (pos_t0 + pos_t0 + K) / 2.0
    bpt, wbytes, kvbytes = decode_bytes_per_token(cfg, ctx_mean)
    gbs = bpt / (ms / 1000.0) / 1e9
    value = 1000.0 / ms
    target = TARGET_70.get((name, ctx))
    out = {"workload": f"{name} {cfg.wtype.upper()} decode bs=1 at context {ctx}"
                       + (f" after a {bulk_prompt}-token bulk prefill" if bulk_prompt else ""),
           "value": value, "unit": "tok/s", "ms_per_step": ms, "steps": K, "kv_len_mean_timed": ctx_mean,
           "step_hbm": {"bytes_per_token": bpt, "weight_bytes": wbytes, "kv_bytes": kvbytes, "achieved_gbs": gbs,
                        "frac_of_measured": gbs / peaks["hbm_gbs"], "frac_of_8tbs": gbs / 8000.0},
           "roofline": in_step_roofline(prof, args.profile_steps, ms, peaks["hbm_gbs"]),
           "target_70pct_of_8tbs": target, "frac_of_target": value / target if target else None}
    return out


def bench_prefill(args, syn, torch, peaks, peak_src):
    """Bulk prefill of one random prompt (qwen2-7B Q4_0, 2048 tokens by default) on the tensor-core
    path: mean device time over reps (KV reset before each), then one profiled run for the split of
    time per kernel kind and the tensor-core rate of the bulk matmuls."""
    cfg = synth.CONFIGS[args.prefill_workload]
    if args.layers:
        cfg = synth.scaled(cfg, n_layer=args.layers, name=f"{cfg.name}_{args.layers}layers")
    n = args.prefill_tokens
    W = synth.make_model(cfg, seed=0)
    stream = torch.cuda.Stream()
    m = syn.Model(syn.read_archdef(cfg.arch), synth.metadata(cfg, n + 8), n + 8, arch=cfg.arch,
                  stream=stream.cuda_stream)
    m.load_tensors(W)
    m.finalize()
    del W
    dtok = torch.from_numpy(synth.tokens(cfg, n, seed=1).astype(np.int32)).cuda()
    darg = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = syn.TOKENS_ON_DEVICE | syn.ARGMAX_ON_DEVICE
    m.forward_raw(dtok.data_ptr(), n, 0, 0, darg.data_ptr(), flags)   # warm-up (builds the bulk plan)
    stream.synchronize()
    times = []
    for _ in range(args.prefill_reps):
        m.reset_kv()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        m.forward_raw(dtok.data_ptr(), n, 0, 0, darg.data_ptr(), flags)
        ev1.record(stream)
        ev1.synchronize()
        times.append(ev0.elapsed_time(ev1))
    ms = statistics.mean(times)
    plane_bytes = m.info("tc_plane_bytes")
    # the same prefill converting the f16 hi/lo operand planes inside every forward (no resident planes)
    m.set_option("tc_planes", 0)
    m.reset_kv()
    m.forward_raw(dtok.data_ptr(), n, 0, 0, darg.data_ptr(), flags)
    stream.synchronize()
    times0 = []
    for _ in range(args.prefill_reps):
        m.reset_kv()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        m.forward_raw(dtok.data_ptr(), n, 0, 0, darg.data_ptr(), flags)
        ev1.record(stream)
        ev1.synchronize()
        times0.append(ev0.elapsed_time(ev1))
    ms0 = statistics.mean(times0)
    m.set_option("tc_planes", -1)
    m.reset_kv()
    m.forward_raw(dtok.data_ptr(), n, 0, 0, darg.data_ptr(), flags)   # rebuild the planes for the profile
    stream.synchronize()
    m.reset_kv()
    m.set_option("profile", 1)
    m.forward_raw(dtok.data_ptr(), n, 0, 0, darg.data_ptr(), flags)
    stream.synchronize()
    prof = m.profile(reset=True)
    pool_bytes = m.timings()["pool_bytes"]
    m.close()
    tc = prof.get("gemm_tc", {"ms": 0.0, "flops": 0.0, "launches": 0})
    f32eq = tc["flops"] / (tc["ms"] / 1000.0) / 1e12 if tc["ms"] else None
    at = prof.get("attention_tc", {"ms": 0.0, "flops": 0.0, "launches": 0})
    at_f32eq = at["flops"] / (at["ms"] / 1000.0) / 1e12 if at["ms"] else None
    tot = sum(v["ms"] for v in prof.values())
    return {
        "workload": f"{cfg.name} {cfg.wtype.upper()} bulk prefill of a {n}-token random prompt (one forward, last-row logits)",
        "value": n / (ms / 1000.0), "unit": "tok/s", "ms": ms, "reps": args.prefill_reps,
        "frame_pool_bytes": pool_bytes,
        "resident_plane_bytes": plane_bytes,
        "note": ("value: the f16 hi/lo operand planes of every matmul weight (4 bytes per weight) are resident "
                 "in device memory, built in the untimed warm-up (option tc_planes -1 builds them when they fit "
                 "in half the free memory); planes_per_forward converts them inside every timed forward"),
        "planes_per_forward": {"value": n / (ms0 / 1000.0), "unit": "tok/s", "ms": ms0, "resident_plane_bytes": 0},
        "tensor": {"kernel": "k_gemm_tc (tcgen05 kind::f16, three MMAs of hi/lo f16 splits per product)",
                   "bulk_matmul_tflop": tc["flops"] / 1e12, "ms": tc["ms"],
                   "achieved_tflops_f32_equivalent": f32eq,
                   "mma_tflops": 3 * f32eq if f32eq else None, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": f32eq / peaks["bf16_tflops"] if f32eq else None,
                   "frac_note": "frac: the method's own flops (2 x M x N x K per matmul) over the bf16 peak; "
                                "mma_frac counts the three f16 MMAs issued per product",
                   "mma_frac": 3 * f32eq / peaks["bf16_tflops"] if f32eq else None,
                   "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops burst; dense f16 has the same nominal rate)"},
        "attention_tensor": {"kernel": "k_attn_tc (tcgen05 kind::f16: S = Q K^T and O = P V, three MMAs of hi/lo f16 splits each)",
                             "tflop_f32_equivalent": at["flops"] / 1e12, "ms": at["ms"],
                             "achieved_tflops_f32_equivalent": at_f32eq,
                             "mma_tflops": 3 * at_f32eq if at_f32eq else None, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": at_f32eq / peaks["bf16_tflops"] if at_f32eq else None,
                             "mma_frac": 3 * at_f32eq / peaks["bf16_tflops"] if at_f32eq else None,
                             "note": "ms and flops include the operand-split kernels of the node; causal: only allowed keys count"},
        "kernels": {k: {"launches": v["launches"], "ms": v["ms"], "share": v["ms"] / tot if tot else None}
                    for k, v in sorted(prof.items())},
    }


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from decoder_token_step_gb300 import build as syn_build
    from decoder_token_step_gb300 import syn
    syn_build.build()

    cfg = synth.CONFIGS[args.workload]
    if args.layers:
        cfg = synth.scaled(cfg, n_layer=args.layers, name=f"{cfg.name}_{args.layers}layers")
    K, Wm = args.steps, args.warmup
    ctx = args.ctx
    P0 = ctx - 1 - Wm                      # positions injected before warm-up
    max_ctx = ctx + K + args.e2e_steps + args.profile_steps + 8
    W = synth.make_model(cfg, seed=0)
    stream = torch.cuda.Stream()
    m = syn.Model(syn.read_archdef(cfg.arch), synth.metadata(cfg, max_ctx), max_ctx, arch=cfg.arch,
                  stream=stream.cuda_stream)
    m.load_tensors(W)
    m.finalize()
    kv = kv_fill_all(cfg, P0)
    for layer, (k, v) in enumerate(kv):
        m.write_kv(layer, 0, k, v)
    del kv
    n_tok = Wm + K + args.e2e_steps + args.profile_steps + 4
    toks = synth.tokens(cfg, n_tok, seed=1)
    dtok = torch.from_numpy(toks.astype(np.int32)).cuda()
    darg = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    flags = syn.TOKENS_ON_DEVICE | syn.ARGMAX_ON_DEVICE
    pos = P0
    ti = 0
    for _ in range(Wm):
        m.forward_raw(dtok.data_ptr() + 4 * ti, 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
        ti += 1
    stream.synchronize()

    # ---- timed region: K decode steps, device-resident token ids, CUDA events on the library stream
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local_rank).uuid)
    except Exception:
        gpu_id = str(local_rank)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pos_t0 = pos
    ev0.record(stream)
    for _ in range(K):
        m.forward_raw(dtok.data_ptr() + 4 * ti, 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
        ti += 1
    ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, torch, "cuda")
    ms_per_step = ms / K
    value = job_throughput(K, world, ms)
    launches_per_step = m.info("n_plan_nodes")

    # ---- end to end through the public API: host token in, host logits + argmax out, every step
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        m.forward([int(toks[ti])], pos)
        pos += 1
        ti += 1
    e2e_s = time.perf_counter() - t0
    e2e_value = args.e2e_steps * world / e2e_s  # replicas run concurrently

    # ---- per-kernel-kind device time (eager, one event pair per kernel group)
    m.set_option("profile", 1)
    prof_pos0 = pos
    for _ in range(args.profile_steps):
        m.forward_raw(dtok.data_ptr() + 4 * ti, 1, pos, 0, darg.data_ptr(), flags)
        pos += 1
        ti += 1
    stream.synchronize()
    prof = m.profile(reset=True)
    m.set_option("profile", 0)
    tm = m.timings()
    memory = {"weight_bytes": tm["weight_bytes"], "kv_bytes": tm["kv_bytes"], "frame_pool_bytes": tm["pool_bytes"],
              "note": "device memory the model holds; the frame pool is the activation registers and scratch of the decode plan"}

    peaks, peak_src = measured_peaks()
    g = prof.get("gemv", {"ms": 0.0, "bytes": 0.0, "launches": 0})
    gemv_per_launch_bytes = g["bytes"] / g["launches"] if g["launches"] else None
    gemv_in_step = in_step_roofline(prof, args.profile_steps, ms_per_step, peaks["hbm_gbs"])
    attn_in_step = in_step_roofline(prof, args.profile_steps, ms_per_step, peaks["hbm_gbs"], kind="attention")
    h = hashlib.sha256()
    for src in ("k_gemv.cu", "gemv_dev.cuh"):
        with open(os.path.join(ROOT, "decoder_token_step_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    gemv_src = h.hexdigest()[:16]
    ratio = GEMV_TRAFFIC_RATIO.get(gemv_src)
    traffic = ratio * gemv_per_launch_bytes if (ratio and gemv_per_launch_bytes) else None
    kernels = {k: {"launches_per_step": v["launches"] / args.profile_steps,
                   "eager_us_per_step": 1000.0 * v["ms"] / args.profile_steps,
                   "eager_gbs": (v["bytes"] / (v["ms"] / 1000.0) / 1e9) if v["ms"] and v["bytes"] else None}
               for k, v in sorted(prof.items())}
    tot_prof_ms = sum(v["ms"] for v in prof.values())
    for k in kernels:
        kernels[k]["share"] = prof[k]["ms"] / tot_prof_ms if tot_prof_ms else None
        kernels[k]["in_step_us"] = 1000.0 * ms_per_step * kernels[k]["share"] if tot_prof_ms else None
    kernels["note"] = ("eager_*: a profiled pass without graph replay or PDL, one event pair per kernel group "
                       "(inflated); in_step_us: that kind's share of the profiled time x the graph-replayed ms_per_step")

    ctx_mean = (pos_t0 + pos_t0 + K) / 2.0
    bpt, wbytes, kvbytes = decode_bytes_per_token(cfg, ctx_mean)
    step_gbs = bpt * (K / (ms / 1000.0)) / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, W, ctx, args.cpu_steps)
    m.close()
    kv16 = bench_decode_kv_f16(args, syn, torch, cfg, W, ctx, peaks) if args.kv_f16_steps > 0 else None
    del W

    prefill = None
    if not args.no_prefill:
        prefill = bench_prefill(args, syn, torch, peaks, peak_src)

    decode_configs = None
    if not args.no_decode_configs and rank == 0:
        decode_configs = bench_decode_configs(args, syn, torch, "qwen3_0_6b", (128, 1024, 4096), peaks, cpu_ctx=1024)
        decode_configs += bench_decode_configs(args, syn, torch, "gemma3_1b", (8192,), peaks, cpu_ctx=8192)
        decode_configs += bench_decode_configs(args, syn, torch, "qwen2_7b", (2048,), peaks, cpu_ctx=2048, bulk_prompt=2048)

    if rank == 0:
        line = {
            "metric": "decode tok/s (bs=1)", "value": value, "unit": "tok/s", "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{cfg.name} Q8_0 decode bs=1 at context {ctx}", "batch": 1, "context": ctx,
                       "kv_len_mean_timed": ctx_mean, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (weights + KV per step >> 129 MB)",
                       "weights": f"{cfg.wtype} GGUF blocks, multiplied in f32", "kv_cache": "f32"},
            "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": 4,
                    "d2h_bytes_per_step": 4 * cfg.n_vocab + 4, "steps": args.e2e_steps},
            "roofline": {"bound": "hbm", "kernel": "k_gemv (weight-streaming GEMV, all decode matmuls)",
                         "achieved": gemv_in_step["achieved"] if gemv_in_step else None, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gemv_in_step["frac"] if gemv_in_step else None,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                         "traffic": traffic, "algorithmic_bytes_per_launch": gemv_per_launch_bytes,
                         "method": "algorithmic bytes per launch / in-step launch time; in-step time = the kind's share "
                                   "of the profiled device time x the timed ms_per_step (CUDA events, graph replay)",
                         "in_step": gemv_in_step},
            "attention_in_step": attn_in_step,
            "step_hbm": {"bytes_per_token": bpt, "weight_bytes": wbytes, "kv_bytes": kvbytes,
                         "achieved_gbs": step_gbs, "frac_of_8tbs": step_gbs / 8000.0,
                         "frac_of_measured": step_gbs / peaks["hbm_gbs"]},
            "kernels": kernels,
            "memory": memory,
            "gpu_launches": launches_per_step * K,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "decode_kv_f16": kv16,
            "decode_configs": decode_configs,
            "target_70pct_of_8tbs": TARGET_70.get((args.workload, ctx)),
            "prefill": prefill,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
