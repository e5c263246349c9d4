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

def build_model(bm, cfg, layers, max_streams, policy):
    import torch
    from gpu_side import build_engine
    t = time.time()
    e = build_engine(WORKLOAD, cfg, layers, max_streams=max_streams, ctx_cap=cfg["ctx_cap"], policy=policy,
                     gen_device="cuda")
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
    e, t_build = build_model(bm, cfg, args.layers, cfg["max_streams"], args.policy)
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

    # B sweep (subsets of the joined streams)
    sweep = {}
    if args.sweep:
        for b in [int(x) for x in args.sweep.split(",") if x]:
            if b > B:
                continue
            sub = slots[:b]
            c1, n1 = cur[:b].clone(), torch.empty(b, dtype=torch.int32, device="cuda")

            def sstep():
                nonlocal c1, n1
                bm.decode_step(e, sub, c1, n1, None, stream)
                c1, n1 = n1, c1

            d = timed_region(sstep, torch.cuda.synchronize, dist, args.sweep_steps, 3,
                             new_event=lambda: torch.cuda.Event(enable_timing=True), device="cuda",
                             label="sweep_timed")
            sweep[str(b)] = round(world * b * args.sweep_steps / d, 1)
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
        pf = {"prompt_tokens": P, "block_rows": cfg["max_streams"], "steps": args.prefill_steps,
              "ms_per_prompt": round(1e3 * d / args.prefill_steps, 3),
              "tok_s": round(world * P * args.prefill_steps / d, 1)}
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
        "kernels": kernels, "sweep_tok_s": sweep, "sweep_weight_roofline": sweep_roof, "prefill": pf,
        "weight_GB": round(stats["weight_bytes"] / 1e9, 3), "arena_GB": round(stats["arena_bytes"] / 1e9, 3),
        "setup_s": round(t_build, 1),
    }
    bm.bm_engine_destroy(e)
    return result


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
            "wall_s": round(wall, 1), "sample_streams": b}


def main():
    args = parse()
    world, rank, local = dist_env()
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
