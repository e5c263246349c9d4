"""Seeded synthetic inputs for the W4A16 MoE decode step.

This module holds none of the decode step's arithmetic: it only draws random
tensors, lengths and join/finish schedules.  Both the CUDA path (through the
tests and the bench) and the CPU oracle take their inputs from here.  Weights
are drawn as raw fp32 values; each side encodes them to int4 with its own
encoder, and the tests check that the two encodings are byte-identical.

Recipes (the workloads of the batched-decode pages, with random-init weights
standing in for the real 30B-class checkpoint, which is not available):

* linear weights: N(0, 0.02) fp32, later quantized to symmetric int4
  (group 32 for the tiny layer, 64 otherwise) with fp16 scales;
* router weights: N(0, 0.02) fp32;
* activations and the KV arena: bf16 N(0, 1);
* embedding and lm_head: bf16 N(0, 0.02);
* slot lengths: uniform integers; prompts: uniform random token ids;
* join/finish schedules: seeded arrivals and departures (``schedule``).

Seeds are derived from a name with SHA-256 so every tensor is reproducible
on its own; ``torch.Generator`` on the requested device draws the values.
"""

import hashlib
import random

import torch

__all__ = ["seed_of", "normal", "normal_bf16", "randint", "CONFIGS",
           "schedule", "prompt_lengths", "model_tensor", "kv_prefix",
           "activations", "tokens"]


def seed_of(*parts):
    """A 63-bit seed from any printable parts (config, tensor name, layer...)."""
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std, seed, device="cpu"):
    """fp32 N(0, std²) tensor."""
    t = torch.randn(shape, generator=_gen(seed, device), device=device,
                    dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def normal_bf16(shape, std, seed, device="cpu"):
    """bf16 tensor of N(0, std²) draws (drawn in fp32, rounded once)."""
    return normal(shape, std, seed, device).to(torch.bfloat16)


def randint(low, high, shape, seed, device="cpu"):
    """int32 uniform integers in [low, high)."""
    return torch.randint(low, high, shape, generator=_gen(seed, device),
                         device=device, dtype=torch.int64).to(torch.int32)


def prompt_lengths(n, low, high, seed):
    """n prompt lengths uniform in [low, high] (inclusive)."""
    rng = random.Random(seed)
    return [rng.randint(low, high) for _ in range(n)]


# Shapes of the five workloads (the tiny single layer, the dense GEMM micro,
# the grouped expert op, slot attention, and the full 48-layer model).
CONFIGS = {
    "tiny_layer": dict(hidden=512, q_heads=8, kv_heads=2, head_dim=64,
                       experts=8, top_k=2, ffn=256, group=32, layers=1,
                       vocab=4096, rope_base=1e4, streams=2, lens=(17, 40)),
    "dense_micro": dict(shapes=((5120, 2048), (2048, 4096)),
                        rows=(1, 2, 4, 8, 16, 32, 64), group=64),
    "expert_op": dict(experts=128, top_k=8, hidden=2048, ffn=768, group=64,
                      batches=(1, 4, 8, 16, 32)),
    "slot_attention": dict(max_streams=16, ctx_cap=8192, q_heads=32,
                           kv_heads=4, head_dim=128, steps=200),
    "full_model": dict(hidden=2048, q_heads=32, kv_heads=4, head_dim=128,
                       experts=128, top_k=8, ffn=768, group=64, layers=48,
                       vocab=151936, rope_base=1e4, max_streams=32,
                       ctx_cap=4096, prompt=(16, 512), gen_tokens=256),
}


WEIGHT_STD = 0.02


def model_tensor(cfg_name, cfg, name, layer=0, expert=0, device="cpu"):
    """One raw weight tensor of a decoder model with shape ``cfg``.

    Linear weights and the router are fp32 N(0, 0.02) (the int4 encoding is
    applied by the consumer); the embedding and lm_head are bf16 N(0, 0.02).
    Row layout of "wqkv": q heads, then k heads, then v heads, head-major.
    """
    H, qh, kvh, d = cfg["hidden"], cfg["q_heads"], cfg["kv_heads"], cfg["head_dim"]
    E, F, V = cfg["experts"], cfg["ffn"], cfg["vocab"]
    shapes = {
        "wqkv": ((qh + 2 * kvh) * d, H), "wo": (H, qh * d), "wr": (E, H),
        "wg": (F, H), "wu": (F, H), "wd": (H, F),
        "embed": (V, H), "lm_head": (V, H),
    }
    shape = shapes[name]
    seed = seed_of(cfg_name, name, layer, expert if name in ("wg", "wu", "wd") else 0)
    if name in ("embed", "lm_head"):
        return normal_bf16(shape, WEIGHT_STD, seed, device)
    return normal(shape, WEIGHT_STD, seed, device)


def kv_prefix(cfg_name, cfg, stream, length, layers=None, device="cpu"):
    """bf16 N(0, 1) K and V prefixes [layers][kvh][length][d] of one stream."""
    L = layers if layers is not None else cfg["layers"]
    shape = (L, cfg["kv_heads"], length, cfg["head_dim"])
    k = normal_bf16(shape, 1.0, seed_of(cfg_name, "kv_prefix_k", stream, length), device)
    v = normal_bf16(shape, 1.0, seed_of(cfg_name, "kv_prefix_v", stream, length), device)
    return k, v


def activations(cfg_name, name, shape, device="cpu"):
    """bf16 N(0, 1) activations."""
    return normal_bf16(shape, 1.0, seed_of(cfg_name, "act", name, *shape), device)


def tokens(cfg_name, name, n, vocab, device="cpu"):
    """n uniform random token ids in [0, vocab)."""
    return randint(0, vocab, (n,), seed_of(cfg_name, "tokens", name, n), device)


def schedule(seed, steps, max_streams, ctx_cap, min_len=1, join_p=0.35,
             finish_p=0.2, max_batch=None):
    """A seeded join/finish schedule.

    Returns a list of per-step event dicts: {"join": [prefix lengths of
    streams joining before this step], "finish": [indices (into the list of
    live streams, oldest first) of streams retiring after this step]}.  At
    least one stream is live at every step; at most ``max_batch`` (default
    ``max_streams``) are live at once; a stream retires no later than one
    step before its length would reach the context cap.
    """
    rng = random.Random(seed)
    cap_b = max_batch or max_streams
    live = []   # remaining steps allowed per live stream
    events = []
    for _ in range(steps):
        joins = []
        want = 1 if not live else (1 if rng.random() < join_p else 0)
        if rng.random() < 0.1 and len(live) + 3 <= cap_b:
            want += 2
        for _ in range(want):
            if len(live) + len(joins) >= cap_b:
                break
            length = rng.randint(min_len, ctx_cap - 2)
            joins.append(length)
        for length in joins:
            live.append(ctx_cap - 1 - length)
        finish = []
        for i in range(len(live)):
            live[i] -= 1
            if live[i] <= 0 or (len(live) - len(finish) > 1 and rng.random() < finish_p):
                finish.append(i)
        if len(finish) == len(live):
            finish = finish[:-1] if live[finish[-1]] > 0 else finish
        events.append({"join": joins, "finish": finish})
        live = [r for i, r in enumerate(live) if i not in set(finish)]
    return events
