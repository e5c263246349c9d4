"""Aggregate decode throughput of the batched W4A16 MoE decode step.

Workload: the full 48-layer 30B-class MoE (hidden 2048, 32/4 heads of 128,
128 experts top-8 with FFN 768, vocab 151936, int4 group 64 with fp16
scales; bf16 embedding and lm_head), synthetic random-init weights drawn on
the device, 32 streams whose prompts (seeded random ids, lengths U[16,512])
are prefilled through decode_step teacher-forced (untimed).  A step is one
decode_step of all B streams: every layer plus the output projection and
greedy argmax, one CUDA graph launch.  Every step reads ~14.6 GB of weights,
far more than L2, so no flush is needed between steps.

Output: one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
on a bounded sample of the same workload instead.
"""

import argparse
import glob
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, os.path.join(ROOT, "tests")):
    if p not in sys.path:
        sys.path.insert(0, p)

METRIC = "aggregate decode tok/s vs B (30B-class int4 MoE, 1 GB300); achieved HBM GB/s"
WORKLOAD = "full_model"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--max-streams", type=int, default=0,
                    help="slots of the engine's KV arena (default: the workload's 32, or --batch if larger; at most 128)")
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--sweep", default="1,2,4,8,16,32", help="B values for the sweep ('' to skip)")
    ap.add_argument("--sweep-steps", type=int, default=10)
    ap.add_argument("--profile-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--policy", type=int, default=0)
    ap.add_argument("--prefill", default="prompt", choices=["prompt", "decode", "kv"],
                    help="prompt: prompts through kv_slot_prefill; decode: through decode_step (teacher-forced); "
                         "kv: seed synthetic K/V of the same lengths (faster start, for profiler runs)")
    ap.add_argument("--prefill-steps", type=int, default=5,
                    help="timed ingestions of one longest-workload prompt (0 to skip)")
    ap.add_argument("--arrivals", type=int, default=64,
                    help="streams of the seeded join/finish run (each ingests its prompt on arrival, decodes "
                         "--gen-tokens greedy tokens and retires; at most max_streams live); 0 to skip")
    ap.add_argument("--gen-tokens", type=int, default=256)
    ap.add_argument("--prefill-path", default="tc", choices=["tc", "decode"],
                    help="kv_slot_prefill on the tcgen05 prompt-length GEMMs (tc) or through the decode kernels "
                         "in blocks of max_streams rows (decode)")
    ap.add_argument("--gemm-sweep", default="16,32,64,128,256,512",
                    help="M values of the prompt-length tcgen05 GEMM timing ('' to skip)")
    ap.add_argument("--tc-probe", action="store_true",
                    help="time the tcgen05 MMA alone (N, A source, operand layout) and the prompt-length GEMM "
                         "against M, without building the model; print one JSON line")
    ap.add_argument("--attention-long", type=int, default=1,
                    help="time the fused attention at the slot-attention workload's lengths (0 to skip)")
    ap.add_argument("--attention-only", action="store_true",
                    help="time only the fused attention at the slot-attention workload's lengths (--steps "
                         "launches after 3 untimed ones), without building the model; print one JSON line")
    ap.add_argument("--kernel-sweep", default="1,4,8,16,32",
                    help="B values of the per-kernel GB/s table ('' to skip)")
    ap.add_argument("--persistent", type=int, default=0,
                    help="1: decode steps of B <= 8 run as the one-launch persistent step (same bytes as the "
                         "multi-kernel step); 0: the multi-kernel step.  Either way the sweep times those B on "
                         "both paths (the solo / batched toggle)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    """Barrier and max-over-ranks of a float; a no-op at world size 1."""

    def __init__(self, world, backend):
        self.world = world
        self.pg = None
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v, device="cpu"):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def timed_region(step, sync, dist, steps, warmup, new_event=None, device="cpu", label="timed"):
    """W untimed steps, then exactly K steps bracketed by barrier + sync on
    both sides; returns the max over ranks of the elapsed seconds.  With
    ``new_event`` (CUDA), the device time between two events is used, inside
    an NVTX range named ``label``."""
    for _ in range(warmup):
        step()
    sync()
    dist.barrier()
    sync()
    if new_event:
        import torch
        t0, t1 = new_event(), new_event()
        torch.cuda.nvtx.range_push(label)
        t0.record()
        for _ in range(steps):
            step()
        t1.record()
        torch.cuda.nvtx.range_pop()
        sync()
        dt = t0.elapsed_time(t1) / 1e3
    else:
        t = time.perf_counter()
        for _ in range(steps):
            step()
        sync()
        dt = time.perf_counter() - t
    dist.barrier()
    return dist.max(dt, device)


class ClockSampler:
    """nvidia-smi samples every 200 ms while running (SM clock, reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu record
    (profiles/dram_traffic.json), or None if there is none or the kernel
    sources changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for path in sorted(glob.glob(os.path.join(ROOT, "bit_moe_decode_w4a16_gb300", "csrc", "*"))):
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("csrc_sha256"):
        return None
    return rec.get("bytes_per_launch", {}).get(kernel)


def int4_bytes(rows, K, g):
    """Bytes of a packed int4 matrix [rows][K] with one fp16 scale per group of g."""
    return rows * K // 2 + rows * (K // g) * 2


def weight_roofline_tok_s(cfg, layers, B, peak_gbs):
    """Decode tok/s if one step only streamed its weights at peak_gbs: per layer
    the dense projections, the fp32 router and the expected number of active
    experts under uniform routing, E (1 - (1 - k/E)^B); once per step the bf16
    output projection."""
    H, F, E, k, g = cfg["hidden"], cfg["ffn"], cfg["experts"], cfg["top_k"], cfg["group"]
    qd, kvd = cfg["q_heads"] * cfg["head_dim"], cfg["kv_heads"] * cfg["head_dim"]
    dense = int4_bytes(qd + 2 * kvd, H, g) + int4_bytes(H, qd, g)
    expert = int4_bytes(2 * F, H, g) + int4_bytes(H, F, g)
    active = E * (1.0 - (1.0 - k / E) ** B)
    step = layers * (dense + E * H * 4 + active * expert) + cfg["vocab"] * H * 2
    return B * peak_gbs * 1e9 / step


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------- our arm

def build_model(bm, cfg, layers, max_streams, policy, prefill_tc=0, persistent_step=0):
    import torch
    from gpu_side import build_engine
    t = time.time()
    e = build_engine(WORKLOAD, cfg, layers, max_streams=max_streams, ctx_cap=cfg["ctx_cap"], policy=policy,
                     gen_device="cuda", prefill_tc=prefill_tc, persistent_step=persistent_step)
    torch.cuda.synchronize()
    return e, time.time() - t


def prefill(bm, e, cfg, B, layers, mode="decode"):
    """Join B streams with empty slots and feed their prompts (kv_slot_prefill,
    or decode_step teacher-forced with mode "decode": the same bytes); returns
    (slots, next device tokens, lengths).  With mode "kv" the slots are
    seeded with synthetic K/V of the same lengths."""
    import torch
    import synth
    lens = synth.prompt_lengths(B, cfg["prompt"][0], cfg["prompt"][1], synth.seed_of(WORKLOAD, "prompt_lens"))
    if mode == "kv":
        slots = []
        for i, L in enumerate(lens):
            k, v = synth.kv_prefix(WORKLOAD, cfg, i, L, layers=layers, device="cuda")
            slots.append(bm.kv_slot_seed(e, k, v, L))
        last = synth.tokens(WORKLOAD, "first", B, cfg["vocab"], device="cuda")
        torch.cuda.synchronize()
        return slots, last, lens
    prompts = [synth.tokens(WORKLOAD, f"prompt{i}", L, cfg["vocab"]).tolist() for i, L in enumerate(lens)]
    empty = torch.empty((layers, cfg["kv_heads"], 0, cfg["head_dim"]), dtype=torch.bfloat16, device="cuda")
    slots = [bm.kv_slot_seed(e, empty, empty, 0) for _ in range(B)]
    last = torch.zeros(B, dtype=torch.int32, device="cuda")
    if mode == "prompt":
        for i, s in enumerate(slots):
            bm.kv_slot_prefill(e, s, torch.tensor(prompts[i], dtype=torch.int32, device="cuda"), last[i:i + 1])
        torch.cuda.synchronize()
        return slots, last, lens
    scratch = torch.empty(B, dtype=torch.int32, device="cuda")
    for t in range(max(lens)):
        idx = [i for i in range(B) if t < lens[i]]
        toks = torch.tensor([prompts[i][t] for i in idx], dtype=torch.int32, device="cuda")
        out = scratch[: len(idx)]
        bm.decode_step(e, [slots[i] for i in idx], toks, out)
        for j, i in enumerate(idx):
            if t == lens[i] - 1:
                last[i] = out[j]
    torch.cuda.synchronize()
    return slots, last, lens


def run_ours(args, dist, world, rank, local):
    import torch
    import bit_moe_decode_w4a16_gb300 as bm
    import synth

    torch.cuda.set_device(local)
    bm.build()
    cfg = dict(synth.CONFIGS[WORKLOAD])
    B = args.batch
    cfg["max_streams"] = max(args.max_streams or cfg["max_streams"], B)
    e, t_build = build_model(bm, cfg, args.layers, cfg["max_streams"], args.policy,
                             prefill_tc=1 if args.prefill_path == "tc" else 0, persistent_step=1)
    bm.bm_engine_set_persistent_step(e, args.persistent)
    slots, last, lens = prefill(bm, e, cfg, B, args.layers, args.prefill)
    stream = torch.cuda.current_stream()
    cur = last.clone()
    nxt = torch.empty_like(cur)

    def step():
        nonlocal cur, nxt
        bm.decode_step(e, slots, cur, nxt, None, stream)
        cur, nxt = nxt, cur

    st0 = bm.bm_engine_stats(e)
    with ClockSampler(local) as clk:
        dt = timed_region(step, torch.cuda.synchronize, dist, args.steps, args.warmup,
                          new_event=lambda: torch.cuda.Event(enable_timing=True), device="cuda")
    st1 = bm.bm_engine_stats(e)
    value = world * B * args.steps / dt
    kernels_per_step = st1["kernels_per_step"]
    launches = (st1["kernel_launches"] - st0["kernel_launches"]) - kernels_per_step * args.warmup

    # end to end through the C ABI with host buffers: H2D of the step's tokens
    # and slots from pinned memory, D2H of the next tokens, every step
    h_in = torch.empty(B, dtype=torch.int32).pin_memory()
    h_out = torch.empty(B, dtype=torch.int32).pin_memory()
    h_in.copy_(cur.cpu())

    def step_e2e():
        bm.decode_step(e, slots, h_in, h_out, None, stream)
        stream.synchronize()
        h_in.copy_(h_out)

    dt_e2e = timed_region(step_e2e, torch.cuda.synchronize, dist, args.steps, 1, device="cuda")
    e2e = {"value": world * B * args.steps / dt_e2e, "unit": "tok/s", "h2d_bytes_per_step": 2 * 4 * B,
           "d2h_bytes_per_step": 4 * B}

    # per-kernel CUDA-event times of eager steps (same stream, same state)
    prof = {}
    for _ in range(args.profile_steps):
        for k in bm.bm_engine_profile_step(e, slots, cur, nxt, stream):
            p = prof.setdefault(k["name"], {"launches": 0, "ms": 0.0, "bytes": 0.0, "flops": 0.0})
            for f in ("launches", "ms", "bytes", "flops"):
                p[f] += k[f]
        cur, nxt = nxt, cur
    peak, peak_kind = peaks()
    kernels = []
    for name, p in sorted(prof.items(), key=lambda kv: -kv[1]["ms"]):
        us = 1e3 * p["ms"] / p["launches"]
        gbs = p["bytes"] / (p["ms"] / 1e3) / 1e9 if p["ms"] > 0 else 0.0
        kernels.append({"name": name, "launches_per_step": p["launches"] // max(1, args.profile_steps),
                        "us_per_launch": round(us, 2), "share": None, "GB_per_s": round(gbs, 1),
                        "frac_hbm": round(gbs / peak, 3)})
    tot = sum(p["ms"] for p in prof.values())
    for k in kernels:
        k["share"] = round(prof[k["name"]]["ms"] / tot, 4) if tot else None
    dom = kernels[0]["name"] if kernels else None
    roof = None
    if dom:
        p = prof[dom]
        achieved = p["bytes"] / (p["ms"] / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": measured_traffic(dom),
                "algorithmic_bytes_per_launch": round(p["bytes"] / p["launches"]),
                "peak_source": f"{peak_kind} hbm_gbs (copy)"}
    step_bytes = sum(p["bytes"] for p in prof.values()) / max(1, args.profile_steps)

    # B sweep (subsets of the joined streams); with the persistent step on,
    # its B also run with it switched off (the multi-kernel step, same bytes)
    sweep, sweep_mk = {}, {}
    if args.sweep:
        def time_b(b):
            sub = slots[:b]
            c1, n1 = cur[:b].clone(), torch.empty(b, dtype=torch.int32, device="cuda")

            def sstep():
                nonlocal c1, n1
                bm.decode_step(e, sub, c1, n1, None, stream)
                c1, n1 = n1, c1

            d = timed_region(sstep, torch.cuda.synchronize, dist, args.sweep_steps, 3,
                             new_event=lambda: torch.cuda.Event(enable_timing=True), device="cuda",
                             label="sweep_timed")
            return round(world * b * args.sweep_steps / d, 1)

        for b in [int(x) for x in args.sweep.split(",") if x]:
            if b > B:
                continue
            sweep[str(b)] = time_b(b)
            if b <= min(8, 64 // cfg["top_k"]):
                bm.bm_engine_set_persistent_step(e, 1 - args.persistent)
                sweep_mk[str(b)] = time_b(b)   # the other path
                bm.bm_engine_set_persistent_step(e, args.persistent)
    # per-kernel GB/s at each B of the kernel sweep (eager steps with events)
    ktab = None
    if args.kernel_sweep:
        try:
            ktab = kernel_table(bm, e, slots, cur, stream, [int(x) for x in args.kernel_sweep.split(",") if x], peak)
        except Exception as ex:   # a reporting extra: never lose the measured line over it
            ktab = {"error": str(ex)}
    # prompt ingestion: one prompt of the workload's longest length into a
    # fresh slot per step (blocks of max_streams rows)
    pf = None
    if args.prefill_steps > 0:
        P = cfg["prompt"][1]
        ptoks = synth.tokens(WORKLOAD, "prefill_bench", P, cfg["vocab"], device="cuda")
        one = torch.empty(1, dtype=torch.int32, device="cuda")
        empty = torch.empty((args.layers, cfg["kv_heads"], 0, cfg["head_dim"]), dtype=torch.bfloat16, device="cuda")
        bm.kv_slot_release(e, slots[0])

        def pstep():
            s = bm.kv_slot_seed(e, empty, empty, 0)
            bm.kv_slot_prefill(e, s, ptoks, one, None, stream)
            bm.kv_slot_release(e, s)

        d = timed_region(pstep, torch.cuda.synchronize, dist, args.prefill_steps, 3,
                         new_event=lambda: torch.cuda.Event(enable_timing=True), device="cuda",
                         label="prefill_timed")
        pf = {"prompt_tokens": P, "path": "tcgen05 prompt-length GEMMs" if args.prefill_path == "tc" else
              f"decode kernels in blocks of {cfg['max_streams']} rows", "steps": args.prefill_steps,
              "ms_per_prompt": round(1e3 * d / args.prefill_steps, 3),
              "tok_s": round(world * P * args.prefill_steps / d, 1)}
    # the prompt-length GEMM on the tensor cores against M
    pg = None
    if args.gemm_sweep:
        try:
            pg = prompt_gemm_sweep(bm, [int(x) for x in args.gemm_sweep.split(",") if x], bf16_peak())
        except Exception as ex:   # a reporting extra: never lose the measured line over it
            pg = {"error": str(ex)}
    att = None
    if args.attention_long:
        try:
            att = attention_long(bm, peak)
        except Exception as ex:   # a reporting extra: never lose the measured line over it
            att = {"error": str(ex)}
    # the configured continuous-batching run: streams join and retire, B varies
    arr = None
    if args.arrivals > 0:
        for s in slots[1:] if args.prefill_steps > 0 else slots:
            bm.kv_slot_release(e, s)
        arr = run_arrivals(bm, e, cfg, args, stream, world)
    # each measured B against the weight-bytes roofline at the measured copy bandwidth
    sweep_roof = {}
    try:
        for b_str, v in sweep.items():
            roof_b = weight_roofline_tok_s(cfg, args.layers, int(b_str), peak) * world
            sweep_roof[b_str] = {"roof_tok_s": round(roof_b, 1), "frac": round(v / roof_b, 4)}
    except Exception:   # a reporting extra: never lose the measured line over it
        sweep_roof = None
    stats = bm.bm_engine_stats(e)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "w4a16 (int4 weights, bf16 activations, fp32 accumulate)",
        "data": "synthetic (random-init N(0,0.02) weights encoded to int4 g64; seeded random prompt ids)",
        "config": {"workload": "full 48-layer 30B-class MoE decode (hidden 2048, 32/4 heads x 128, 128 experts "
                               "top-8, FFN 768, vocab 151936), one decode_step of B streams per step",
                   "global_batch": B, "layers": args.layers, "ctx_cap": cfg["ctx_cap"],
                   "prompt_lens": f"U[{cfg['prompt'][0]},{cfg['prompt'][1]}] ingested before timing ({args.prefill})",
                   "kv_len_mean_at_start": round(sum(lens) / len(lens), 1),
                   "l2": "inputs larger than L2: ~14.6 GB of weights read per step",
                   "parallelism": "replicas" if world > 1 else "1 GPU",
                   "kernel_family": {1: "simt", 2: "tc", 3: "mma"}.get(bm.bm_engine_kernel_family(e), "?")},
        "clocks": clk.summary(), "e2e": e2e, "gpu_launches": int(launches),
        "graph_launches_per_step": (st1["graph_launches"] - st0["graph_launches"]) / (args.steps + args.warmup),
        "roofline": roof,
        "step_algorithmic_GB": round(step_bytes / 1e9, 3),
        "step_GB_per_s": round(step_bytes / (dt / args.steps) / 1e9, 1),
        "kernels": kernels, "sweep_tok_s": sweep, "sweep_weight_roofline": sweep_roof,
        "small_batch_path": {
            "default": "persistent kernel" if args.persistent else "multi-kernel step",
            "rows": min(8, 64 // cfg["top_k"]),
            "persistent_tok_s": sweep_mk if not args.persistent else {b: sweep[b] for b in sweep_mk},
            "multikernel_tok_s": {b: sweep[b] for b in sweep_mk} if not args.persistent else sweep_mk,
            "persistent_over_multikernel": {
                b: round((sweep_mk[b] / sweep[b]) if not args.persistent else (sweep[b] / sweep_mk[b]), 3)
                for b in sweep_mk if sweep_mk[b] and sweep[b]},
            "bytes": "identical on both paths (tests/test_gpu_persist.py)"},
        "kernels_by_B": ktab,
        "arrivals": arr, "prefill": pf, "prompt_gemm": pg, "attention_long": att,
        "weight_GB": round(stats["weight_bytes"] / 1e9, 3), "arena_GB": round(stats["arena_bytes"] / 1e9, 3),
        "setup_s": round(t_build, 1),
    }
    bm.bm_engine_destroy(e)
    return result


def arrival_schedule(n_streams, max_live, gen_tokens, seed):
    """Seeded arrivals of n_streams streams (one per step with probability
    0.35, a burst of up to four with probability 0.05, never more than
    max_live live at once, the first at step 0); each stream decodes
    gen_tokens tokens and retires.  Returns the arrival step of every stream,
    the order in which they may join."""
    import random
    rng = random.Random(seed)
    arrive, live_until, step = [], [], 0
    while len(arrive) < n_streams:
        live_until = [t for t in live_until if t > step]
        want = 1 if (not arrive or rng.random() < 0.35) else 0
        if rng.random() < 0.05:
            want += rng.randint(1, 3)
        for _ in range(want):
            if len(arrive) == n_streams or len(live_until) >= max_live:
                break
            arrive.append(step)
            live_until.append(step + gen_tokens)
        step += 1
    return arrive


def run_arrivals(bm, e, cfg, args, stream, world):
    """The workload's continuous-batching run: streams join on a seeded
    schedule (slot seeded empty, prompt of U[16,512] seeded ids ingested with
    kv_slot_prefill), decode gen_tokens greedy tokens in one decode_step per
    step over every live stream, and retire (slot released, no wipe), so B
    changes as streams come and go.  Decode tok/s = decode tokens / summed
    device time of the decode steps (CUDA events around each step on the
    launching stream); prompt ingestion is timed apart.  Graphs for every B
    are captured in a warm-up pass before the run."""
    import torch
    import synth
    S, n = cfg["max_streams"], args.arrivals
    arrive = arrival_schedule(n, S, args.gen_tokens, synth.seed_of(WORKLOAD, "arrivals"))
    lens = synth.prompt_lengths(n, cfg["prompt"][0], cfg["prompt"][1], synth.seed_of(WORKLOAD, "arrival_lens"))
    empty = torch.empty((args.layers, cfg["kv_heads"], 0, cfg["head_dim"]), dtype=torch.bfloat16, device="cuda")
    # warm-up: one step at every B so that each graph is captured outside the run
    warm = [bm.kv_slot_seed(e, empty, empty, 0) for _ in range(S)]
    toks = torch.zeros(S, dtype=torch.int32, device="cuda")
    outs = torch.empty(S, dtype=torch.int32, device="cuda")
    for b in range(1, S + 1):
        bm.decode_step(e, warm[:b], toks[:b], outs[:b], None, stream)
    torch.cuda.synchronize()
    for s in warm:
        bm.kv_slot_release(e, s)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    live = []          # [slot, remaining tokens, row in cur]
    cur = torch.zeros(n, dtype=torch.int32, device="cuda")   # next input token of each stream
    nxt = torch.empty(S, dtype=torch.int32, device="cuda")
    decode_ev, prefill_ev, bs = [], [], []
    nxt_stream, step, tokens_out = 0, 0, 0
    t_wall = time.perf_counter()
    while nxt_stream < n or live:
        while nxt_stream < n and arrive[nxt_stream] <= step and len(live) < S:
            i = nxt_stream
            prompt = synth.tokens(WORKLOAD, f"arrival_prompt{i}", lens[i], cfg["vocab"], device="cuda")
            s = bm.kv_slot_seed(e, empty, empty, 0)
            a, b = ev(), ev()
            a.record(stream)
            bm.kv_slot_prefill(e, s, prompt, cur[i:i + 1], None, stream)
            b.record(stream)
            prefill_ev.append((a, b, lens[i]))
            live.append([s, args.gen_tokens, i])
            nxt_stream += 1
        if not live:
            step += 1
            continue
        B = len(live)
        idx = torch.tensor([r[2] for r in live], dtype=torch.int64, device="cuda")
        inp = cur.index_select(0, idx).to(torch.int32)
        a, b = ev(), ev()
        a.record(stream)
        bm.decode_step(e, [r[0] for r in live], inp, nxt[:B], None, stream)
        b.record(stream)
        decode_ev.append((a, b, B))
        cur.index_copy_(0, idx, nxt[:B])
        tokens_out += B
        bs.append(B)
        for r in live:
            r[1] -= 1
        for r in [r for r in live if r[1] == 0]:
            bm.kv_slot_release(e, r[0])
        live = [r for r in live if r[1] > 0]
        step += 1
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    t_dec = sum(a.elapsed_time(b) for a, b, _ in decode_ev) / 1e3
    t_pre = sum(a.elapsed_time(b) for a, b, _ in prefill_ev) / 1e3
    hist = {}
    for b in bs:
        hist[b] = hist.get(b, 0) + 1
    return {"streams": n, "gen_tokens": args.gen_tokens, "decode_steps": len(bs), "decode_tokens": tokens_out,
            "decode_tok_s": round(world * tokens_out / t_dec, 1), "decode_s": round(t_dec, 3),
            "B_mean": round(sum(bs) / len(bs), 2), "B_min": min(bs), "B_max": max(bs),
            "prompt_tokens": sum(lens), "prefill_tok_s": round(world * sum(lens) / t_pre, 1),
            "prefill_s": round(t_pre, 3), "wall_s": round(wall, 2),
            "schedule": "seeded arrivals (p=0.35 per step, bursts), prompts U[16,512] ingested on arrival, "
                        f"{args.gen_tokens} greedy tokens each, at most {S} live"}


def kernel_table(bm, e, slots, cur, stream, Bs, peak, steps=2):
    """Per-kernel CUDA-event times of eager steps at each B of Bs, with the
    algorithmic GB/s and their fraction of the measured copy bandwidth."""
    import torch
    out = {}
    for B in Bs:
        if B > len(slots):
            continue
        c, n = cur[:B].clone(), torch.empty(B, dtype=torch.int32, device="cuda")
        acc = {}
        for _ in range(steps):
            for k in bm.bm_engine_profile_step(e, slots[:B], c, n, stream):
                p = acc.setdefault(k["name"], [0, 0.0, 0.0])
                p[0] += k["launches"]
                p[1] += k["ms"]
                p[2] += k["bytes"]
            c, n = n, c
        rows = {}
        for name, (launches, ms, byts) in sorted(acc.items(), key=lambda kv: -kv[1][1]):
            gbs = byts / (ms / 1e3) / 1e9 if ms > 0 else 0.0
            rows[name] = {"us_per_launch": round(1e3 * ms / launches, 2), "GB_per_s": round(gbs, 1),
                          "frac_hbm": round(gbs / peak, 3)}
        out[str(B)] = rows
    return out


def prompt_gemm_sweep(bm, Ms, peak_tflops, reps=20):
    """The prompt-length W4A16 GEMM (w4_gemm_prompt_tc) on the QKV shape
    (N 5120, K 2048, g 64) for each M: CUDA-event time per launch (each launch
    timed alone after warm-up, weights L2-resident after the first), the
    achieved TFLOP/s (2 M N K per launch) and its fraction of the measured
    dense bf16 peak (fp16 runs at the same nominal rate)."""
    import torch
    import synth
    N, K, g = 5120, 2048, 64
    raw = synth.normal((N, K), 0.02, synth.seed_of("bench", "prompt_gemm", N, K), "cuda")
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, K // g), dtype=torch.float16, device="cuda")
    bm.bm_w4_quantize(raw, N, K, g, packed, scales)
    wm = torch.empty_like(packed)
    sm = torch.empty((N * (K // g) // 2,), dtype=torch.int32, device="cuda")
    bm.bm_w4_repack_mma(packed, scales, N, K, g, wm, sm)
    X = synth.normal((max(Ms), K), 1.0, synth.seed_of("bench", "prompt_gemm_x"), "cuda").half()
    out = {}
    for M in Ms:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            bm.w4_gemm_prompt_tc(wm, sm, X[:M], Y, None, M, N, K, g)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record()
        for _ in range(reps):
            bm.w4_gemm_prompt_tc(wm, sm, X[:M], Y, None, M, N, K, g)
        t1.record()
        torch.cuda.synchronize()
        us = 1e3 * t0.elapsed_time(t1) / reps
        tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
        out[str(M)] = {"us": round(us, 2), "TFLOP_s": round(tf, 1), "frac_bf16_peak": round(tf / peak_tflops, 3)}
    return {"shape": f"N {N} x K {K}, g {g}", "peak_tflops": peak_tflops, "by_M": out}


def attention_long(bm, peak_gbs, reps=20):
    """The step's fused attention kernel at the slot-attention workload's
    lengths (16 slots of an 8192-position arena, 32 q / 4 kv heads of 128,
    lengths U[1, 8192]) through bm_engine_attention: CUDA-event time per
    launch (the launch rewrites each slot's position len with the same k, v,
    so repeats are identical) and the K/V bytes attended per second against
    the measured copy bandwidth.  The arena (1.07 GB) is far larger than L2,
    but a launch reads only the attended positions (~97 MB)."""
    import torch
    import synth
    S, cap, qh, kvh, d = 16, 8192, 32, 4, 128
    cfg = {"hidden": 512, "q_heads": qh, "kv_heads": kvh, "head_dim": d, "experts": 8, "top_k": 2, "ffn": 256,
           "group": 32, "vocab": 64, "layers": 1, "rope_base": 1e4, "rms_eps": 1e-6, "max_streams": S,
           "ctx_cap": cap, "renorm_topk": 1, "kernel_policy": 3, "use_graph": 0}
    e = bm.bm_engine_create(cfg)
    try:
        lens = synth.prompt_lengths(S, 1, cap - 1, synth.seed_of("slot_attention", "bench_lens"))
        slots = []
        for i, L in enumerate(lens):
            k = synth.normal_bf16((1, kvh, L, d), 1.0, synth.seed_of("slot_attention", "bk", i, L), "cuda")
            v = synth.normal_bf16((1, kvh, L, d), 1.0, synth.seed_of("slot_attention", "bv", i, L), "cuda")
            slots.append(bm.kv_slot_seed(e, k, v, L))
            del k, v
        qkv = synth.normal_bf16((S, (qh + 2 * kvh) * d), 1.0, synth.seed_of("slot_attention", "bqkv"), "cuda")
        out = torch.empty((S, qh, d), dtype=torch.float16, device="cuda")
        for _ in range(3):
            bm.bm_engine_attention(e, 0, slots, qkv, out)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record()
        for _ in range(reps):
            bm.bm_engine_attention(e, 0, slots, qkv, out)
        t1.record()
        torch.cuda.synchronize()
        bm.bm_engine_sync(e)
        us = 1e3 * t0.elapsed_time(t1) / reps
        byts = sum((L + 1) * kvh * d * 2 * 2 for L in lens)
        gbs = byts / (us * 1e-6) / 1e9
        return {"streams": S, "kv_len_mean": round(sum(lens) / S, 1), "us": round(us, 2),
                "kv_MB": round(byts / 1e6, 1), "GB_per_s": round(gbs, 1), "frac_hbm": round(gbs / peak_gbs, 3)}
    finally:
        bm.bm_engine_destroy(e)


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


# ---------------------------------------------------------------- oracle arm

class OracleSample:
    """The CPU oracle on a bounded sample of the workload: one decoder layer
    of b streams (each with its seeded KV prefix of the workload's length mix)
    plus the output projection of those b rows, projected to the whole model
    as tok/s = b / (layers * t_layer + t_head).  Inputs come from synth;
    encoding the weights is set-up and untimed."""

    def __init__(self, B, layers_total):
        import torch
        import synth
        from oracle_side import bf16_bits, oracle_config, quant
        self.B, self.layers_total = B, layers_total
        cfg = self.cfg = dict(synth.CONFIGS[WORKLOAD])
        g = cfg["group"]
        self.dev = "cuda" if torch.cuda.is_available() else "cpu"
        dev = self.dev
        self.ocfg = oracle_config(cfg, layers=1, max_streams=B, ctx_cap=cfg["ctx_cap"])
        cache = {}

        def expert(e):
            if e not in cache:
                cache[e] = {n: quant(synth.model_tensor(WORKLOAD, cfg, n, 0, e, dev), g) for n in ("wg", "wu", "wd")}
            return cache[e]
        self.lw = {"wqkv": quant(synth.model_tensor(WORKLOAD, cfg, "wqkv", 0, device=dev), g),
                   "wo": quant(synth.model_tensor(WORKLOAD, cfg, "wo", 0, device=dev), g),
                   "wr": synth.model_tensor(WORKLOAD, cfg, "wr", 0, device=dev).cpu().numpy(),
                   "expert": expert}
        self.lens = synth.prompt_lengths(B, cfg["prompt"][0], cfg["prompt"][1],
                                         synth.seed_of(WORKLOAD, "prompt_lens"))
        self.x = synth.activations(WORKLOAD, "oracle_x", (B, cfg["hidden"])).double().numpy()
        self.lm_bits = bf16_bits(synth.model_tensor(WORKLOAD, cfg, "lm_head", device=dev))
        self.prefix = []
        for i, L in enumerate(self.lens):
            k, v = synth.kv_prefix(WORKLOAD, cfg, i, L, layers=1, device=dev)
            self.prefix.append((k.double().cpu().numpy(), v.double().cpu().numpy()))

    def run(self, b=None):
        """Times (t_layer, t_head) of one sample over the first b streams."""
        import oracle
        b = b or self.B
        kv = oracle.OracleKV(self.ocfg, oracle.OracleSlotMap(self.B, self.cfg["ctx_cap"]))
        slots = [kv.seed(*self.prefix[i]) for i in range(b)]
        t = time.perf_counter()
        y = oracle.decoder_layer(self.ocfg, self.lw, self.x[:b], slots, kv, 0)
        t_layer = time.perf_counter() - t
        t = time.perf_counter()
        oracle.model.lm_head_logits(oracle.bf16_round(oracle.rmsnorm(y)), self.lm_bits)
        t_head = time.perf_counter() - t
        return t_layer, t_head

    def tok_s(self, b, t_layer, t_head):
        return b / (self.layers_total * t_layer + t_head)


def oracle_sample(B, layers_total):
    """One warm run (encodes the routed experts), then one timed run."""
    s = OracleSample(B, layers_total)
    s.run()
    tl, th = s.run()
    return s.tok_s(B, tl, th), tl, th


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, world, rank, budget_s=150.0):
    B = args.batch
    s = OracleSample(B, args.layers)
    tl, th = s.run()                          # warm: encodes the routed experts
    # per-step sample size: b of the B streams, so that K steps fit the budget
    b = max(1, min(B, int(B * budget_s / max(1e-9, args.steps * (tl + th)))))
    for _ in range(min(args.warmup, 1)):
        s.run(b)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tl, th = s.run(b)
        vals.append(s.tok_s(b, tl, th))
    wall = time.perf_counter() - t0
    value = sum(vals) / len(vals)
    sample = (f"per step: one decoder layer of {b} of the B={B} streams (their KV prefixes of the workload's "
              f"length mix) + the lm_head of those rows, projected to {args.layers} layers: "
              f"tok/s = b / ({args.layers} * t_layer + t_head)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * B / value, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (numpy oracle)",
            "data": "synthetic", "config": {"workload": "full 48-layer 30B-class MoE decode", "global_batch": B},
            "cpu_baseline": {"value": round(value, 4), "unit": "tok/s", "cores": cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1), "sample_streams": b,
            "projection": (f"value and ms_per_step are projected: each step times ONE decoder layer of {b} streams "
                           f"and the output projection, and scales the layer time to {args.layers} layers; "
                           f"the {args.steps} steps took {wall:.1f} s of wall time")}


def tc_probe():
    """SM cycles per tcgen05 MMA of M 128 x N x K 16 (kind::f16) issued back to
    back by one thread into one accumulator, for N, the A source and the
    shared-memory operand layout (bm_probe_tcgen05_mma)."""
    import torch
    import bit_moe_decode_w4a16_gb300 as bm
    torch.cuda.init()
    bm.build()
    rows = []
    for a_tmem in (1, 0):
        for swz in (0, 1):
            for n in (16, 32, 64, 128, 256):
                bm.bm_probe_tcgen05_mma(n, a_tmem, swz, 64)   # warm
                issue, done = bm.bm_probe_tcgen05_mma(n, a_tmem, swz, 1024)
                macs = 128 * n * 16
                rows.append({"N": n, "A": "tmem" if a_tmem else "smem", "layout": "sw128" if swz else "none",
                             "issue_cycles": round(issue, 1), "complete_cycles": round(done, 1),
                             "MAC_per_cycle": round(macs / done, 1)})
    for n in (16, 128):
        bm.bm_probe_tcgen05_mma(n, 1, 0, 64, 1)
        issue, done = bm.bm_probe_tcgen05_mma(n, 1, 0, 256, 1)
        rows.append({"N": n, "A": "tmem", "layout": "none", "roundtrip": True, "issue_cycles": round(issue, 1),
                     "complete_cycles": round(done, 1), "stage_roundtrip_cycles": round(4 * done, 1)})
    return {"probe": "tcgen05.mma.cta_group::1.kind::f16, M 128 x N x K 16, 1024 stages of 4 MMAs, one accumulator "
                     "(roundtrip rows: 256 stages, each committed and waited for)",
            "rows": rows}


def main():
    args = parse()
    world, rank, local = dist_env()
    if args.tc_probe:
        if rank == 0:
            import bit_moe_decode_w4a16_gb300 as bm
            out = tc_probe()
            out["prompt_gemm"] = prompt_gemm_sweep(bm, [int(x) for x in args.gemm_sweep.split(",") if x], bf16_peak())
            print(json.dumps(out), flush=True)
        return
    if args.attention_only:
        if rank == 0:
            import bit_moe_decode_w4a16_gb300 as bm
            print(json.dumps(attention_long(bm, peaks()[0], reps=args.steps)), flush=True)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    import torch
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist = Dist(world, backend)
    try:
        result = run_ours(args, dist, world, rank, local)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            v, tl, th = oracle_sample(args.batch, args.layers)
            result["cpu_baseline"] = {"value": round(v, 4), "unit": "tok/s", "cores": cores(), "kind": "oracle",
                                      "sample": f"one decoder layer of B={args.batch} streams ({tl:.1f} s) + lm_head "
                                                f"of B rows ({th:.1f} s), projected to {args.layers} layers"}
        if rank == 0:
            print(json.dumps(result), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
