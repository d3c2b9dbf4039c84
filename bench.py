#!/usr/bin/env python3
"""Benchmark of the decode-time routed MoE layer stack on GB300 (one JSON line).

Default workload: the DeepSeek-V3-shaped stack, the largest that fits one GPU - 58 MoE
layers, H = 7168, 256 routed experts with F = 2048 plus one always-on shared expert,
sigmoid scores with top-8 selected and normalised, RVQ 3-bit experts (16.55 MB per expert,
58 x 257 experts = 246.7 GB resident in HBM), decode T = 1, x ~ N(0,1) (bf16) fed layer to
layer as x += moe(rmsnorm(x)).  One step = one token through all 58 layers (router,
gate/up, down, combine and the residual RMS norm of every layer), replayed from one CUDA
graph with the inputs resident in HBM.  The per-token expert working set (9 x 58 x
16.55 MB = 8.6 GB) is far larger than the 129 MB L2, so no flush is needed between steps.

Other workloads (``--config``): tiny, mixtral (32 int4 layers), dsv3 with T = 4 or 32
(--tokens-per-step), wide, stream (HBM LRU cache over a pinned host pool), stream-file;
``--top-k`` overrides k (the streamed top-16 vs top-8 comparison).

Reported: tokens/s (value), expert-weight GB/s against the HBM peak, hit %, the dominant
kernel's roofline (CUDA events around each kernel, recorded inside the timed graph), the
end-to-end rate through host buffers, SM clocks sampled during the timed region, and the
fp64 CPU oracle timed on a bounded sample (``cpu_baseline``), which also routes the GPU
run's own normalised inputs of a few tokens and reports the near-ties (oracle gap between
the k-th and (k+1)-th score below 1e-5) and any expert-id mismatch outside them.
``--impl reference`` times that oracle alone on the same workload.  N > 1 GPUs (torchrun)
run independent replicas: the layer does not shard (weak scaling, no collective on the
data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth as S  # noqa: E402

CONFIGS = {
    "tiny": dict(workload="tiny MoE layer: 1 layer, H=256, F=512, 8 experts, top-2 softmax, RVQ-3bit, T=4",
                 layers=1, H=256, F=512, E=8, k=2, router=0, shared=False, wfmt=S.RVQ, T=4,
                 tokens=64, trace="iid", cache=0),
    "mixtral": dict(workload="Mixtral-shaped stack: 32 MoE layers, H=4096, F=14336, 8 experts, top-2 softmax, "
                             "int4 g128 fp16 scales, all 256 experts resident, decode T=1, 512-token sequence",
                    layers=32, H=4096, F=14336, E=8, k=2, router=0, shared=False, wfmt=S.INT4, T=1,
                    tokens=512, trace="iid", cache=0),
    "dsv3": dict(workload="DeepSeek-V3-shaped stack: 58 MoE layers, H=7168, 256 routed experts F=2048 + 1 shared, "
                          "sigmoid top-8 normalised, RVQ-3bit, all resident",
                 layers=58, H=7168, F=2048, E=256, k=8, router=1, shared=True, wfmt=S.RVQ, T=1,
                 tokens=256, trace="iid", cache=0),
    "wide": dict(workload="Wide top-16 stack: 24 MoE layers, H=7168, 384 experts F=1536, top-16 softmax, RVQ-3bit, "
                          "all resident, decode T=1 over a 1024-token domain-local trace",
                 layers=24, H=7168, F=1536, E=384, k=16, router=0, shared=False, wfmt=S.RVQ, T=1,
                 tokens=1024, trace="domain", cache=0),
    "stream": dict(workload="Streaming tier: 48 MoE layers x 256 experts, H=7168, F=1536, top-16, RVQ-3bit, pinned "
                            "host pool, 32 GB HBM LRU cache, side-stream miss copies, 4096-token domain-local trace",
                   layers=48, H=7168, F=1536, E=256, k=16, router=0, shared=False, wfmt=S.RVQ, T=1,
                   tokens=4096, trace="domain", cache=32_000_000_000),
    "stream-file": dict(workload="File tier: 16 MoE layers x 256 experts, H=7168, F=1536, top-16, RVQ-3bit, experts "
                                 "in a local file behind a 16 GB pinned RAM LRU cache behind an 8 GB HBM LRU cache, "
                                 "512-token domain-local trace",
                        layers=16, H=7168, F=1536, E=256, k=16, router=0, shared=False, wfmt=S.RVQ, T=1,
                        tokens=512, trace="domain", cache=8_000_000_000, host_cache=16_000_000_000),
}
# one-layer cuts of the big shapes (a few GB on the device), for profiler captures
for _n, _src in (("mixtral1", "mixtral"), ("dsv3-1", "dsv3"), ("wide1", "wide")):
    CONFIGS[_n] = dict(CONFIGS[_src], layers=1, workload="one layer of the " + CONFIGS[_src]["workload"])
SEED = 0
L2_BYTES = 129e6
FALLBACK_HBM_GBS = 6800.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- peaks, clocks
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in mp:
                return float(mp[key]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (MEASURED_PEAKS.json absent)"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- inputs
def token_inputs(cfg, n):
    """[n, T, H] float32 values (bf16-rounded): the workload's token process."""
    H, T = cfg["H"], cfg["T"]
    if cfg["trace"] == "domain":
        x = S.make_domain_trace(SEED, 0, n * T, H)
    else:
        x = S.make_tokens(SEED, 0, n * T, H)
    return x.reshape(n, T, H)


def build_context(cfg, device, max_tokens):
    """Create the context and register every router and expert (blobs made on the GPU)."""
    import torch
    import routed_expert_ffn_03_gb300 as M
    from synth import device as D
    t0 = time.time()
    ctx = M.Context(cfg["layers"], cfg["H"], cfg["F"], cfg["E"], cfg["k"], cfg["wfmt"], router=cfg["router"],
                    shared_ffn=cfg["F"] if cfg["shared"] else 0, max_tokens=max_tokens,
                    hbm_cache_bytes=cfg["cache"], device=device, pool_file=cfg.get("pool_file"),
                    host_cache_bytes=int(cfg.get("host_cache", 0)))
    nb = S.expert_blob_bytes(cfg["wfmt"], cfg["H"], cfg["F"])
    blob = torch.empty(nb, dtype=torch.uint8, device="cuda:%d" % device)
    experts = list(range(cfg["E"])) + ([-1] if cfg["shared"] else [])
    for l in range(cfg["layers"]):
        ctx.register_router(l, S.make_router(SEED, l, cfg["E"], cfg["H"]))
        for e in experts:
            D.make_expert_blob_device(SEED, l, e, cfg["wfmt"], cfg["H"], cfg["F"], blob,
                                      stream=torch.cuda.current_stream().cuda_stream)
            ctx.register_expert(l, e, blob)
    del blob
    torch.cuda.synchronize()
    log("registered %d layers x %d experts in %.1f s" % (cfg["layers"], len(experts), time.time() - t0))
    return ctx


def measure_link_gbs(device):
    """Host -> device bandwidth of this machine: a pinned 1 GiB cudaMemcpyAsync, best of 10."""
    import torch
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device="cuda:%d" % device)
    best = 0.0
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, n / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del h, d
    return best


def measure_record_copy_gbs(device, rec_bytes, n=48):
    """Host -> device bandwidth of back-to-back copies of one expert record each (pinned
    source), on one stream and spread over four: best of 3.  The link figure at the copy
    size the streamed tier issues."""
    import torch
    h = torch.empty(n * rec_bytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(n * rec_bytes, dtype=torch.uint8, device="cuda:%d" % device)
    out = {}
    for ns in (1, 4):
        streams = [torch.cuda.Stream(device=device) for _ in range(ns)]
        best = 0.0
        for _ in range(3):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(streams[0])
            for st in streams[1:]:
                st.wait_event(e0)
            for i in range(n):
                with torch.cuda.stream(streams[i % ns]):
                    d[i * rec_bytes:(i + 1) * rec_bytes].copy_(h[i * rec_bytes:(i + 1) * rec_bytes], non_blocking=True)
            ends = []
            for st in streams:
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(st)
                ends.append(ev)
            torch.cuda.synchronize()
            ms = max(e0.elapsed_time(ev) for ev in ends)
            best = max(best, n * rec_bytes / (ms / 1e3) / 1e9)
        out["record_copy_gbs_%dstream%s" % (ns, "" if ns == 1 else "s")] = round(best, 2)
    del h, d
    return out


def gateup_bytes_per_expert(cfg):
    H, F = cfg["H"], cfg["F"]
    if cfg["wfmt"] == S.INT4:
        return 2 * (F * H // 2 + F * (H // 128) * 2)
    return 2 * (3 * 256 * 8 * 2 + F * (H // 8) * 3)


def kernel_source_hash(wfmt):
    name = "int4.cu" if wfmt == S.INT4 else "rvq.cu"
    with open(os.path.join(ROOT, "routed_expert_ffn_03_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(cfg_name, wfmt):
    """Per-launch DRAM bytes of the gate/up kernel from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tab = json.load(f)
        ent = tab.get(cfg_name)
        if ent and ent.get("source_sha256_16") == kernel_source_hash(wfmt):
            return float(ent["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# ----------------------------------------------------------------------------- CPU oracle
def oracle_layer_sample(cfg, n_tokens, n_layers, device):
    """Time the fp64 oracle stack on tokens 0..n_tokens-1 through layers 0..n_layers-1.
    Expert blobs are generated on demand; the time spent making them is not counted."""
    import torch
    from oracle import oracle as O
    from synth import device as D
    x0 = token_inputs(cfg, n_tokens)[:, 0, :] if cfg["T"] == 1 else token_inputs(cfg, 1)[0][:n_tokens]
    nb = S.expert_blob_bytes(cfg["wfmt"], cfg["H"], cfg["F"])
    dev = torch.empty(nb, dtype=torch.uint8, device="cuda:%d" % device)
    cache = {}
    gen_time = [0.0]

    def blob(l, e):
        if (l, e) not in cache:
            t = time.perf_counter()
            D.make_expert_blob_device(SEED, l, e, cfg["wfmt"], cfg["H"], cfg["F"], dev)
            cache[(l, e)] = dev.cpu().numpy()
            gen_time[0] += time.perf_counter() - t
        return cache[(l, e)]

    routers = [S.make_router(SEED, l, cfg["E"], cfg["H"]) for l in range(n_layers)]
    layers = []
    for l in range(n_layers):
        def fn(xn, l=l):
            return O.layer(xn, routers[l], cfg["k"], cfg["router"], lambda e: blob(l, e), cfg["wfmt"],
                           cfg["H"], cfg["F"], blob(l, -1) if cfg["shared"] else None,
                           cfg["F"] if cfg["shared"] else 0)
        layers.append(fn)
    t0 = time.perf_counter()
    O.stack(x0, layers)
    dt = time.perf_counter() - t0 - gen_time[0]
    del dev
    return dt, O.threads()


def routing_check(cfg, check):
    """The oracle router (fp64 logits, brute-force top-k) on the normalised inputs the GPU
    run fed each layer (teacher-forced): counts the near-ties (oracle gap between the k-th
    and (k+1)-th score below 1e-5) and the decisions whose expert ids differ outside them."""
    from oracle import oracle as O
    routers = {}
    n = ties = flips = mism = 0
    t0 = time.perf_counter()
    for per_xn, per_idx in check:
        for l, (xnb, idx) in enumerate(zip(per_xn, per_idx)):
            if l not in routers:
                routers[l] = S.make_router(SEED, l, cfg["E"], cfg["H"])
            r = O.router(xnb, routers[l], cfg["k"], cfg["router"])
            for t in range(xnb.shape[0]):
                n += 1
                same = np.array_equal(idx[t], r["idx"][t])
                if r["gap"][t] < 1e-5:
                    ties += 1
                    flips += 0 if same else 1
                elif not same:
                    mism += 1
    return {"decisions": n, "near_ties": ties, "near_tie_flips": flips, "mismatches_outside_near_ties": mism,
            "sample": "the GPU run's bf16 router inputs of %d steps x %d layers x %d tokens per step, routed by the "
                      "fp64 oracle (%.1f s)" % (len(check), cfg["layers"], cfg["T"], time.perf_counter() - t0)}


def cpu_baseline(cfg, device, check=None):
    n_tok, n_lay = (4, min(cfg["layers"], 8)) if cfg["wfmt"] == S.INT4 else (2, min(cfg["layers"], 4))
    if cfg["name"] == "tiny":
        n_tok, n_lay = 4, 1
    dt, cores = oracle_layer_sample(cfg, n_tok, n_lay, device)
    per_token = dt / n_tok * cfg["layers"] / n_lay
    out = {"value": cfg["T"] / per_token if cfg["T"] > 1 and cfg["name"] == "tiny" else 1.0 / per_token,
           "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": "fp64 oracle (router, top-k, explicit dequant, dense SwiGLU, combine, rmsnorm stack) on "
                     "%d tokens x the first %d of %d layers, %.1f s, extrapolated to the full stack"
                     % (n_tok, n_lay, cfg["layers"], dt)}
    if check:
        out["routing_check"] = routing_check(cfg, check)
    return out


# ----------------------------------------------------------------------------- GPU arm
def lru_hit_rate(trace, slots, k_use):
    """Hit rate of a record-granular LRU of `slots` records over a routing trace, cold
    start, lookups of each (token, layer) in ascending expert id, the current layer's
    experts pinned (the engine's rules).  trace: list over (token, layer) of the routed ids
    in rank order; only the first k_use of each are looked up."""
    from collections import OrderedDict
    lru = OrderedDict()
    hits = looks = 0
    for layer, ids in trace:
        cur = sorted(set(int(e) for e in ids[:k_use]))
        pinned = set()
        for e in cur:
            key = (layer, e)
            looks += 1
            if key in lru:
                hits += 1
                lru.move_to_end(key)
            else:
                if len(lru) >= slots:
                    for victim in lru:          # least recent first
                        if victim[0] != layer or victim[1] not in pinned:
                            break
                    del lru[victim]
                lru[key] = True
            pinned.add(e)
    return hits / max(1, looks)


def hit_sweep(ctx, cfg, layers_fn, x, x0_dev, n_tokens, stream):
    """Routing trace of n_tokens through the stack (results do not depend on the cache), then
    the LRU hit rate at several cache budgets for top-k and top-k/2 (the first half of each
    top-k list is the top-(k/2) selection)."""
    import torch
    trace = []
    with torch.cuda.stream(stream):
        for i in range(n_tokens):
            x.copy_(x0_dev[i % x0_dev.shape[0]])
            for l in range(cfg["layers"]):
                layers_fn(l)
                idx, _ = ctx.get_routing(l)
                trace.append((l, idx[0]))
    rec = ctx.stats()["record_bytes"]
    rows = []
    for gb in (8, 16, 32, 64, 96, 128):
        slots = int(gb * 1e9 // rec)
        rows.append({"budget_gb": gb, "slots": slots,
                     "hit_rate_k%d" % cfg["k"]: round(lru_hit_rate(trace, slots, cfg["k"]), 4),
                     "hit_rate_k%d" % (cfg["k"] // 2): round(lru_hit_rate(trace, slots, cfg["k"] // 2), 4)})
    return {"tokens": n_tokens, "method": "routing trace of the stack (T=1, domain-local inputs) replayed through "
            "the engine's LRU rules on the host, cold start", "rows": rows}


def run_gpu(args, cfg, rank, world, device):
    import torch
    torch.cuda.set_device(device)
    import routed_expert_ffn_03_gb300 as M  # noqa: F401
    T = cfg["T"]
    ctx = build_context(cfg, device, max_tokens=T)
    H, L = cfg["H"], cfg["layers"]
    n_inp = cfg["tokens"]
    x0_host = torch.from_numpy(np.ascontiguousarray(token_inputs(cfg, n_inp))).float()   # [n, T, H]
    x0_dev = x0_host.cuda(device)
    x = torch.zeros((T, H), dtype=torch.float32, device=device)
    y = torch.zeros((T, H), dtype=torch.float32, device=device)
    xn = torch.zeros((T, H), dtype=torch.int16, device=device)
    stream = torch.cuda.Stream(device=device)
    streamed = cfg["cache"] != 0
    if streamed:
        ctx.set_readahead(bool(args.readahead))

    def layers():
        # x += y_prev; xn = rmsnorm(x); y = layer(xn)   (fused stack step), then the last add
        for l in range(L):
            ctx.forward_residual(l, x, None if l == 0 else y, xn, y, T)
        ctx.residual_rmsnorm(x, y, xn, T)

    graph = None
    with torch.cuda.stream(stream):
        x.copy_(x0_dev[0])
        layers()
    torch.cuda.synchronize()
    launches_per_step = None
    if not streamed:
        before = ctx.stats()["launches"]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            layers()
        torch.cuda.synchronize()
        launches_per_step = ctx.stats()["launches"] - before   # the kernels of one replay

    def step(i):
        x.copy_(x0_dev[i % n_inp])
        if graph is not None:
            graph.replay()
        else:
            layers()

    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    torch.cuda.synchronize()
    ctx.reset_stats()
    hit_series = []
    clocks = ClockSampler(device)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(K):
            step(W + i)
            if streamed and (i + 1) % 64 == 0:
                st = ctx.stats()
                hit_series.append(round(st["hits"] / max(1, st["lookups"]), 4))
        ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        t = torch.tensor([ms], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    st = ctx.stats()
    secs = ms / 1e3
    tok_s = world * K * T / secs
    expert_gbs = st["bytes_expert_touched"] / secs / 1e9
    peak, peak_src = hbm_peak()

    # e2e: same steps through host (pinned) buffers, copies inside the timed region
    e2e = None
    if graph is not None:
        xh = x0_host.pin_memory()
        outh = torch.empty((min(K, 64), T, H), dtype=torch.float32).pin_memory()
        with torch.cuda.stream(stream):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(K):
                x.copy_(xh[(W + i) % n_inp], non_blocking=True)
                graph.replay()
                outh[i % outh.shape[0]].copy_(x, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        ems = e0.elapsed_time(e1)
        e2e = {"value": round(world * K * T / (ems / 1e3), 3), "unit": "tokens/s",
               "h2d_bytes_per_step": T * H * 4, "d2h_bytes_per_step": T * H * 4}

    # per-kernel durations: CUDA events around every kernel (event nodes of a second graph
    # of the same step, replayed on the same stream); kept out of the headline timing above
    prof = None
    if graph is not None:
        try:
            ctx.profile(True)
            pgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pgraph, stream=stream):
                layers()
            acc4, nacc = [0.0] * 4, 0
            with torch.cuda.stream(stream):
                for i in range(args.prof_steps):
                    x.copy_(x0_dev[(W + K + i) % n_inp])
                    pgraph.replay()
                    ms4_i, nl_i = ctx.profile_read()
                    acc4 = [u + v for u, v in zip(acc4, ms4_i)]
                    nacc += nl_i
            ctx.profile(False)
            prof = (acc4, nacc)
        except Exception as e:  # noqa: BLE001
            log("per-kernel profile failed: %s" % e)
    roofline = None
    if prof is not None:
        ms4, nl = prof
        if nl > 0:
            uniq_per_layer = st["lookups"] / max(1, st["forwards"])
            experts_per_launch = uniq_per_layer + (1 if cfg["shared"] else 0)
            alg = experts_per_launch * gateup_bytes_per_expert(cfg)
            dur = ms4[1] / nl / 1e3
            ach = alg / dur / 1e9
            tr = ncu_traffic(cfg["name"], cfg["wfmt"])
            roofline = {"bound": "hbm", "kernel": "int4_gateup_kernel" if cfg["wfmt"] == S.INT4 else "rvq_kernel<gate/up>",
                        "achieved": round(ach, 1), "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                        "traffic": tr, "peak_source": peak_src,
                        "alg_bytes_per_launch": int(alg), "avg_launch_us": round(dur * 1e6, 2),
                        "timing": "CUDA events around each kernel on its stream, %d replays x %d layers "
                                  "(event nodes in a separate copy of the step graph); an event node between two "
                                  "kernels chained by programmatic dependent launch stops the next kernel's prologue "
                                  "from overlapping the previous one's tail, so this duration is an upper bound and "
                                  "the fraction a lower bound" % (args.prof_steps, cfg["layers"]),
                        "per_kernel_us": {n: round(v / nl * 1e3, 2) for n, v in
                                          zip(("router", "gateup", "down", "combine"), ms4)}}
    out = {
        "metric": "MoE decode tokens/s; expert-weight GB/s vs HBM peak; cache hit % (1 GB300)",
        "value": round(tok_s, 3), "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 x fp16(hi+lo) -> fp32" if cfg["wfmt"] == S.INT4 else "rvq3 (fp16 codebooks) x fp32 LUT -> fp32",
        "data": "synthetic (seeded SplitMix64 weights and inputs, no trained weights)",
        "config": {"workload": cfg["workload"], "layers": L, "hidden": H, "ffn": cfg["F"], "experts": cfg["E"],
                   "top_k": cfg["k"], "tokens_per_step": T, "parallelism": "replicas" if world > 1 else "single GPU",
                   "graph": graph is not None,
                   "l2": "no flush: per-step expert working set %.2f GB > 129 MB L2" % (
                       st["bytes_expert_touched"] / max(1, K) / 1e9)},
        "expert_gbs": round(expert_gbs, 1), "hbm_frac": round(expert_gbs / peak, 4),
        "hit_rate": round(st["hits"] / max(1, st["lookups"]), 4),
        "roofline": roofline, "e2e": e2e,
        "gpu_launches": K * launches_per_step if launches_per_step is not None else st["launches"],
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    if streamed:
        link = measure_link_gbs(device)
        rec_copy = measure_record_copy_gbs(device, st["record_bytes"])
        miss_gbs = st["bytes_h2d"] / max(1e-9, st["h2d_ms"] / 1e3) / 1e9 if st["h2d_ms"] else None
        out["hit_series_per64"] = hit_series
        if args.hit_sweep and T == 1:
            ctx.set_readahead(False)

            def one_layer(l):
                ctx.forward_residual(l, x, None if l == 0 else y, xn, y, T)
            out["hit_rate_vs_cache"] = hit_sweep(ctx, cfg, one_layer, x, x0_dev, args.hit_sweep, stream)
        out["streaming"] = {
            "readahead": bool(args.readahead),
            "misses_per_token": round(st["misses"] / max(1, K), 2), "hits": st["hits"], "misses": st["misses"],
            "prefetches": st["prefetches"], "prefetch_hits": st["prefetch_hits"],
            "prefetch_accuracy": round(st["prefetch_hits"] / st["prefetches"], 4) if st["prefetches"] else None,
            "bytes_h2d": st["bytes_h2d"], "link_busy_ms": round(st["h2d_ms"], 2),
            "link_busy_frac_of_run": round(st["h2d_ms"] / ms, 4),
            "miss_copy_gbs": round(miss_gbs, 2) if miss_gbs else None,
            "link_gbs_measured": round(link, 2),
            "miss_frac_of_link": round(miss_gbs / link, 4) if miss_gbs else None,
            "link_measure": "pinned 1 GiB cudaMemcpyAsync host->device, best of 10, same run; copy GB/s = all "
                            "expert bytes copied (misses and read-ahead) / time the link was busy (union of the "
                            "copy batches)",
            "cache_slots": st["cache_slots"]}
        out["streaming"].update(rec_copy)
        if cfg.get("pool_file"):
            out["streaming"]["file_tier"] = {
                "file_bytes": cfg["file_bytes"], "ram_cache_bytes": int(cfg["host_cache"]),
                "o_direct": bool(st["file_direct"]), "file_reads": st["file_reads"],
                "ram_hits": st["ram_hits"], "ram_misses": st["ram_misses"],
                "file_read_gbs": round(st["file_read_bytes"] / (st["file_read_ms"] / 1e3) / 1e9, 2)
                if st["file_read_ms"] else None,
                "file_read_ms": round(st["file_read_ms"], 2),
                "file_read_frac_of_run": round(st["file_read_ms"] / ms, 4),
                "read_measure": "records read from the file (4096-byte aligned, 8 reader threads) / wall time of "
                                "the read batches, which the forward waits for"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the router inputs (bf16 xn) and expert ids of every layer for a few steps, read back
        # layer by layer, for the oracle's routing check in the CPU-baseline leg
        check = []
        if streamed:
            ctx.set_readahead(False)
        with torch.cuda.stream(stream):
            for i in range(args.check_tokens):
                x.copy_(x0_dev[i % n_inp])
                per_xn, per_idx = [], []
                for l in range(L):
                    ctx.forward_residual(l, x, None if l == 0 else y, xn, y, T)
                    per_xn.append(xn.cpu().numpy().view(np.uint16).copy())
                    per_idx.append(ctx.get_routing(l)[0])
                check.append((per_xn, per_idx))
        torch.cuda.synchronize()
        ctx.close()
        torch.cuda.empty_cache()
        out["cpu_baseline"] = cpu_baseline(cfg, device, check)
        rc = out["cpu_baseline"].get("routing_check")
        if rc:
            out["near_ties"] = {k_: rc[k_] for k_ in ("decisions", "near_ties", "near_tie_flips",
                                                      "mismatches_outside_near_ties")}
    else:
        ctx.close()
    return out


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, cfg, device):
    """The fp64 oracle alone: each step = one token's router + one matrix of one selected
    expert of one layer (layers cycle over the first few), so the whole run stays within
    minutes; the rate is extrapolated to the full stack."""
    from oracle import oracle as O
    nl = min(cfg["layers"], 2)
    xin = token_inputs(cfg, max(1, min(cfg["tokens"], 64)))
    routers = [S.make_router(SEED, l, cfg["E"], cfg["H"]) for l in range(nl)]
    cache = {}

    def blob(l, e):       # host generator: this arm loads no GPU library
        if (l, e) not in cache:
            cache[(l, e)] = S.make_expert_blob(SEED, l, e, cfg["wfmt"], cfg["H"], cfg["F"])
        return cache[(l, e)]

    shapes = S.matrix_shapes(cfg["H"], cfg["F"])
    offs = np.cumsum([0] + [S.matrix_block_bytes(cfg["wfmt"], r, kk) for r, kk in shapes])
    t_router, t_mat = [], [[], [], []]
    for i in range(args.warmup + args.steps):
        l = i % nl
        m = i % 3                      # gate, up, down in rotation
        xb = O.rmsnorm_bf16(xin[i % xin.shape[0]])
        t0 = time.perf_counter()
        r = O.router(xb, routers[l], cfg["k"], cfg["router"])
        t1 = time.perf_counter()
        e = int(r["idx"][0, (i // 3) % cfg["k"]])
        b = blob(l, e)
        rows, K = shapes[m]
        xv = O.bf16_value(xb[:1])
        if K != xv.shape[1]:            # down input: the token's values tiled to F (timing only)
            xv = np.resize(xv, (1, K))
        t2 = time.perf_counter()
        O.matvec(cfg["wfmt"], rows, K, b[offs[m]:offs[m + 1]], xv)
        t3 = time.perf_counter()
        if i >= args.warmup:
            t_router.append(t1 - t0)
            t_mat[m].append(t3 - t2)
    t_expert = [sum(statistics.mean(v) for v in t_mat if v)]
    per_layer_token = statistics.mean(t_router) + (cfg["k"] + (1 if cfg["shared"] else 0)) * statistics.mean(t_expert)
    value = cfg["T"] / (per_layer_token * cfg["T"] * cfg["layers"])
    return {
        "impl": "reference",
        "metric": "MoE decode tokens/s; expert-weight GB/s vs HBM peak; cache hit % (1 GB300)",
        "value": round(value, 6), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * (statistics.mean(t_router) + t_expert[0] / 3), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 weights and inputs)",
        "config": {"workload": cfg["workload"], "layers": cfg["layers"], "hidden": cfg["H"], "ffn": cfg["F"],
                   "experts": cfg["E"], "top_k": cfg["k"], "tokens_per_step": cfg["T"]},
        "cpu_baseline": {"value": round(value, 6), "unit": "tokens/s", "cores": O.threads(), "kind": "oracle",
                         "sample": "each step: fp64 oracle router + one matrix (gate, up, down in rotation) of one "
                                   "selected expert for one token at layer (step mod %d); tokens/s = 1 / (layers x "
                                   "(router + k x (gate + up + down)))" % nl},
        "e2e": {"value": round(value, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="dsv3", choices=sorted(CONFIGS))
    ap.add_argument("--tokens-per-step", type=int, default=0, help="override T (dsv3: 1, 4, 32)")
    ap.add_argument("--top-k", type=int, default=0, help="override k (e.g. 8 on the top-16 stream config)")
    ap.add_argument("--check-tokens", type=int, default=8,
                    help="tokens whose per-layer normalised inputs the CPU-baseline leg routes with the oracle")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prof-steps", type=int, default=16, help="replays of the per-kernel event graph")
    ap.add_argument("--readahead", type=int, default=1, choices=[0, 1],
                    help="streamed configs: predict the next layer's experts and copy them early")
    ap.add_argument("--pool-file", default=None,
                    help="stream-file: where the expert file goes (default: the temp directory)")
    ap.add_argument("--hit-sweep", type=int, default=0, metavar="TOKENS",
                    help="streamed configs: after the timed run, the LRU hit rate vs cache budget over a "
                         "routing trace of this many tokens")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    cfg = dict(CONFIGS[args.config])
    cfg["name"] = args.config
    if args.tokens_per_step:
        cfg["T"] = args.tokens_per_step
        cfg["workload"] += " (T=%d per step)" % cfg["T"]
    if args.top_k:
        if not 1 <= args.top_k <= min(cfg["E"], 32):
            raise SystemExit("--top-k must be in 1..%d" % min(cfg["E"], 32))
        cfg["workload"] += " (top-%d instead of top-%d)" % (args.top_k, cfg["k"])
        cfg["k"] = args.top_k
    if cfg.get("host_cache"):
        # the file tier: the expert file goes to --pool-file's directory (default: the temp
        # directory); fewer layers when that filesystem lacks room for all of them
        import tempfile
        path = args.pool_file or os.path.join(tempfile.gettempdir(), "moe-experts-%d.bin" % os.getpid())
        stride = (S.expert_blob_bytes(cfg["wfmt"], cfg["H"], cfg["F"]) + 4095) // 4096 * 4096
        vfs = os.statvfs(os.path.dirname(os.path.abspath(path)))
        free_b = vfs.f_bavail * vfs.f_frsize
        per_layer = cfg["E"] * stride
        fit = int((free_b * 0.8) // per_layer)
        if fit < 2:
            raise SystemExit("not enough room for the expert file in %s (%.1f GB free)" % (path, free_b / 1e9))
        if fit < cfg["layers"]:
            cfg["workload"] += " (%d of %d layers: %.0f GB free for the file)" % (fit, cfg["layers"], free_b / 1e9)
            cfg["layers"] = fit
        cfg["pool_file"] = path
        cfg["file_bytes"] = cfg["layers"] * per_layer
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        from oracle import oracle as O      # builds and loads oracle/liboracle.so only
        O.build()
        print(json.dumps(run_reference(args, cfg, local)), flush=True)
        return

    import torch
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        import __graft_entry__ as G
        G.build()
    if world > 1:
        torch.distributed.barrier()
    out = run_gpu(args, cfg, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
