"""Decoder layer, full decode step and the slot lifecycle, in plain fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

One decode step ([Batched serving, §1 Contribution]): B streams each bring
one token; all layers run over the B rows; then the per-stream output
projection and greedy selection.  The layer is the pre-norm MoE decoder:

    xn = R(rmsnorm(x))
    q, k, v = R(xn · Wqkvᵀ)                     (q: qh heads, k/v: kvh heads)
    q, k = R(rope(q, pos)), R(rope(k, pos))     pos = the slot's length
    K/V of the slot at position pos <- k, v     (appended before attention)
    o = R(attention(q, K[0..pos], V[0..pos]))
    h = R(x + o · Woᵀ)
    hn = R(rmsnorm(h))
    ids, w = top-k routing of hn
    a_r = R(SiLU(W_g[e_r] hn) ⊙ (W_u[e_r] hn));  out_r = W_d[e_r] a_r
    y = R(h + Σ_r w_r out_r)                    (rank order)

R is rounding to bf16: the path's activations are 16-bit ("W4A16"), so every
activation tensor handed from one op to the next is a bf16 tensor; inside an
op the arithmetic is exact (fp64 here).  After the last layer:
logits = R(rmsnorm(y)) · W_lmᵀ (bf16 head, unrounded logits), next token =
argmax with ties to the lowest id.

Readings where the pages are silent: no biases, no QK-norm, no shared expert,
untied bf16 embedding and head; RMSNorm eps 1e-6 with unit weights unless
given; RoPE rotate-half, base 1e4; a new stream's slot is the lowest-numbered
free slot; a slot's length advances once per step, after all layers.

The slot lifecycle ([KV-slot isolation, §1 Contribution];
[Crash root cause, §3 Results]): a stream's KV prefix is written once when it
joins (seed), each step appends one position, the slot is released when the
stream retires (a logical reset, no wipe), and a change in batch composition
never touches a continuing stream's KV.
"""

from dataclasses import dataclass, field

import numpy as np

from .numerics import bf16_round, dequant_w4, from_bf16_bits
from .ops import rmsnorm, rope_rotate_half, slot_attention, causal_block_attention, route_topk, silu, rowwise


@dataclass
class OracleConfig:
    hidden: int = 2048
    q_heads: int = 32
    kv_heads: int = 4
    head_dim: int = 128
    experts: int = 128
    top_k: int = 8
    ffn: int = 768
    group: int = 64
    vocab: int = 151936
    layers: int = 48
    rope_base: float = 1e4
    eps: float = 1e-6
    ctx_cap: int = 4096
    max_streams: int = 32
    renorm_topk: bool = True

    @property
    def qkv_rows(self):
        return (self.q_heads + 2 * self.kv_heads) * self.head_dim


class OracleSlotMap:
    """Host model of the slot lifecycle: seed at join, release at retire."""

    def __init__(self, max_streams, ctx_cap):
        self.max_streams = max_streams
        self.ctx_cap = ctx_cap
        self.active = [False] * max_streams
        self.length = [0] * max_streams

    def seed(self, length):
        """Admit a stream with a prefix of ``length`` positions; return its slot.

        Rejected (ValueError) when the prefix leaves no room for a decode
        token, or when every slot is taken.
        """
        if length < 0 or length >= self.ctx_cap:
            raise ValueError("context cap")
        for s in range(self.max_streams):
            if not self.active[s]:
                self.active[s] = True
                self.length[s] = length
                return s
        raise ValueError("no free slot")

    def release(self, slot):
        if not self.active[slot]:
            raise ValueError("slot is free")
        self.active[slot] = False
        self.length[slot] = 0

    def check_batch(self, slots):
        if len(set(slots)) != len(slots):
            raise ValueError("duplicate slot")
        for s in slots:
            if not self.active[s]:
                raise ValueError("slot is free")
            if self.length[s] >= self.ctx_cap:
                raise ValueError("context cap")

    def advance(self, slots):
        for s in slots:
            self.length[s] += 1


class OracleKV:
    """K/V contents of every slot and layer, as float64 arrays [kvh][len][d]."""

    def __init__(self, cfg, slot_map):
        self.cfg = cfg
        self.map = slot_map
        self.K = {}
        self.V = {}

    def seed(self, K, V):
        """K, V: [layers][kvh][len][d] (bf16 values).  Returns the slot."""
        K = np.asarray(K, dtype=np.float64)
        V = np.asarray(V, dtype=np.float64)
        length = K.shape[2]
        slot = self.map.seed(length)
        self.K[slot] = [K[l].copy() for l in range(self.cfg.layers)]
        self.V[slot] = [V[l].copy() for l in range(self.cfg.layers)]
        return slot

    def release(self, slot):
        self.map.release(slot)
        del self.K[slot]
        del self.V[slot]

    def write_pending(self, layer, slot, k, v):
        """Place this step's k, v ([kvh][d]) at position = the slot's length."""
        pos = self.map.length[slot]
        Kl, Vl = self.K[slot][layer], self.V[slot][layer]
        assert Kl.shape[1] in (pos, pos + 1)
        Kl = np.concatenate([Kl[:, :pos], np.asarray(k, np.float64)[:, None]], axis=1)
        Vl = np.concatenate([Vl[:, :pos], np.asarray(v, np.float64)[:, None]], axis=1)
        self.K[slot][layer], self.V[slot][layer] = Kl, Vl

    def write_block(self, layer, slot, k, v):
        """Place a prompt's k, v ([P][kvh][d]) at positions length .. length+P-1."""
        pos = self.map.length[slot]
        k = np.asarray(k, np.float64).transpose(1, 0, 2)
        v = np.asarray(v, np.float64).transpose(1, 0, 2)
        Kl, Vl = self.K[slot][layer], self.V[slot][layer]
        assert Kl.shape[1] in (pos, pos + k.shape[1])
        self.K[slot][layer] = np.concatenate([Kl[:, :pos], k], axis=1)
        self.V[slot][layer] = np.concatenate([Vl[:, :pos], v], axis=1)

    def view(self, layer, slot, count):
        return self.K[slot][layer][:, :count], self.V[slot][layer][:, :count]


def _round(x):
    return bf16_round(x)


def decoder_layer(cfg, lw, x, slots, kv, layer, trace=None):
    """One decoder layer over the B rows of ``x`` (bf16 values, [B][H]).

    ``lw`` holds the layer's weights: "attn_norm"/"ffn_norm" ([H] or None),
    "wqkv" and "wo" as (packed, scales), "wr" (fp32 [E][H]) and "expert"
    (a callable e -> dict with "wg", "wu", "wd" as (packed, scales)).
    Returns the layer output (bf16 values, float64 [B][H]).
    """
    H, qh, kvh, d, g = cfg.hidden, cfg.q_heads, cfg.kv_heads, cfg.head_dim, cfg.group
    x = np.asarray(x, dtype=np.float64)
    B = x.shape[0]
    xn = _round(rmsnorm(x, lw.get("attn_norm"), cfg.eps))
    Wqkv = dequant_w4(lw["wqkv"][0], lw["wqkv"][1], H, g)
    qkv = _round(rowwise(Wqkv, xn))
    q = qkv[:, : qh * d].reshape(B, qh, d)
    k = qkv[:, qh * d: (qh + kvh) * d].reshape(B, kvh, d)
    v = qkv[:, (qh + kvh) * d:].reshape(B, kvh, d)
    o = np.empty((B, qh * d), dtype=np.float64)
    q_rot = np.empty_like(q)
    for b in range(B):
        slot = slots[b]
        pos = kv.map.length[slot]
        q_rot[b] = _round(rope_rotate_half(q[b], pos, cfg.rope_base))
        k_rot = _round(rope_rotate_half(k[b], pos, cfg.rope_base))
        kv.write_pending(layer, slot, k_rot, v[b])
        Kc, Vc = kv.view(layer, slot, pos + 1)
        o[b] = _round(slot_attention(q_rot[b], Kc, Vc)).reshape(-1)
    y = _after_attention(cfg, lw, x, o, trace)
    if trace is not None:
        trace.update(dict(xn=xn, qkv=qkv, q_rot=q_rot, attn=o))
    return y


def _after_attention(cfg, lw, x, o, trace=None):
    """The rest of a decoder layer, row by row: output projection with the
    residual, RMSNorm, top-k routing, the selected experts, and the weighted
    combine with the residual (x, o: bf16 values [B][H], [B][qh*d])."""
    H, qh, d, g = cfg.hidden, cfg.q_heads, cfg.head_dim, cfg.group
    Wo = dequant_w4(lw["wo"][0], lw["wo"][1], qh * d, g)
    h = _round(x + rowwise(Wo, o))
    return moe_block(cfg, lw, h, trace)


def moe_block(cfg, lw, h, trace=None):
    """The mixture-of-experts half of a decoder layer on the residual rows h
    (bf16 values [B][H]): RMSNorm with the ffn norm, top-k routing, the
    selected experts' FFNs, and the combine with the residual, row by row
    ([Batched serving, §1 Contribution]: the experts the router selects for
    each stream run against the resident int4 bank)."""
    H, g = cfg.hidden, cfg.group
    h = np.asarray(h, dtype=np.float64)
    B = h.shape[0]
    hn = _round(rmsnorm(h, lw.get("ffn_norm"), cfg.eps))
    ids, w = route_topk(hn, lw["wr"], cfg.top_k, cfg.renorm_topk)
    F = cfg.ffn
    cache = {}

    def expert_mats(e):
        if e not in cache:
            ew = lw["expert"](e)
            cache[e] = (dequant_w4(ew["wg"][0], ew["wg"][1], H, g),
                        dequant_w4(ew["wu"][0], ew["wu"][1], H, g),
                        dequant_w4(ew["wd"][0], ew["wd"][1], F, g))
        return cache[e]

    y = np.empty_like(h)
    outs_all = np.empty((B, cfg.top_k, H), dtype=np.float64)
    for b in range(B):
        acc = np.zeros(H, dtype=np.float64)
        for r in range(cfg.top_k):
            Wg, Wu, Wd = expert_mats(int(ids[b, r]))
            a = _round(silu(Wg @ hn[b]) * (Wu @ hn[b]))
            out = Wd @ a
            outs_all[b, r] = out
            acc = acc + w[b, r] * out
        y[b] = _round(h[b] + acc)
    if trace is not None:
        trace.update(dict(h=h, hn=hn, ids=ids, w=w, expert_out=outs_all, y=y))
    return y


def prefill_layer(cfg, lw, x, slot, kv, layer, trace=None):
    """One decoder layer over the P prompt rows of one stream (bf16 values
    [P][H]); row i sits at position start + i, start = the slot's length.
    Same arithmetic as ``decoder_layer`` for every row; the attention is the
    causal block form over the slot."""
    H, qh, kvh, d, g = cfg.hidden, cfg.q_heads, cfg.kv_heads, cfg.head_dim, cfg.group
    x = np.asarray(x, dtype=np.float64)
    P = x.shape[0]
    start = kv.map.length[slot]
    xn = _round(rmsnorm(x, lw.get("attn_norm"), cfg.eps))
    Wqkv = dequant_w4(lw["wqkv"][0], lw["wqkv"][1], H, g)
    qkv = _round(rowwise(Wqkv, xn))
    q = qkv[:, : qh * d].reshape(P, qh, d)
    k = qkv[:, qh * d: (qh + kvh) * d].reshape(P, kvh, d)
    v = qkv[:, (qh + kvh) * d:].reshape(P, kvh, d)
    pos = start + np.arange(P)
    q_rot = _round(rope_rotate_half(q, pos, cfg.rope_base))
    k_rot = _round(rope_rotate_half(k, pos, cfg.rope_base))
    kv.write_block(layer, slot, k_rot, v)
    Kc, Vc = kv.view(layer, slot, start + P)
    o = _round(causal_block_attention(q_rot, Kc, Vc, start)).reshape(P, qh * d)
    y = _after_attention(cfg, lw, x, o, trace)
    if trace is not None:
        trace.update(dict(xn=xn, qkv=qkv, q_rot=q_rot, attn=o))
    return y


def lm_head_logits(xf, lm_head_bits, chunk=16384):
    """logits = xf · W_lmᵀ with W_lm given as bf16 bit patterns [V][H]."""
    xf = np.asarray(xf, dtype=np.float64)
    V = lm_head_bits.shape[0]
    out = np.empty((xf.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, chunk):
        W = from_bf16_bits(lm_head_bits[v0: v0 + chunk])
        out[:, v0: v0 + chunk] = rowwise(W, xf)
    return out


def model_step(cfg, weights, kv, slots, tokens, traces=None):
    """One decode step of B streams; returns (logits [B][V], next ids [B]).

    ``weights``: "embed_row" (callable id -> bf16 values [H]), "layers"
    (list of per-layer dicts as in ``decoder_layer``), "final_norm" ([H] or
    None) and "lm_head_bits" (uint16 [V][H]).  Each stream's token sits at
    position = its slot's current length; the lengths advance after the step.
    """
    kv.map.check_batch(list(slots))
    x = np.stack([np.asarray(weights["embed_row"](int(t)), np.float64) for t in tokens])
    for layer, lw in enumerate(weights["layers"]):
        tr = {} if traces is not None else None
        x = decoder_layer(cfg, lw, x, slots, kv, layer, tr)
        if traces is not None:
            traces.append(tr)
    xf = _round(rmsnorm(x, weights.get("final_norm"), cfg.eps))
    logits = lm_head_logits(xf, weights["lm_head_bits"])
    nxt = np.argmax(logits, axis=1).astype(np.int32)
    kv.map.advance(list(slots))
    return logits, nxt


def model_prefill(cfg, weights, kv, slot, tokens, traces=None):
    """Prompt ingestion for one active stream; returns (logits [V], next id)
    of the position after the prompt.

    The P tokens take positions start .. start+P-1 (start = the slot's
    length); every layer writes their K/V into the slot
    ([KV-slot isolation, §1 Contribution]: the stream's K/V is written once,
    at join, then extended by decode), and the length advances by P.  Only
    the last row reaches the output projection.  Rejected (ValueError) when
    the slot is free or the prompt does not fit the context cap.
    """
    P = len(tokens)
    if P < 1:
        raise ValueError("empty prompt")
    if not kv.map.active[slot]:
        raise ValueError("slot is free")
    if kv.map.length[slot] + P > kv.map.ctx_cap:
        raise ValueError("context cap")
    x = np.stack([np.asarray(weights["embed_row"](int(t)), np.float64) for t in tokens])
    for layer, lw in enumerate(weights["layers"]):
        tr = {} if traces is not None else None
        x = prefill_layer(cfg, lw, x, slot, kv, layer, tr)
        if traces is not None:
            traces.append(tr)
    xf = _round(rmsnorm(x[-1:], weights.get("final_norm"), cfg.eps))
    logits = lm_head_logits(xf, weights["lm_head_bits"])[0]
    kv.map.length[slot] += P
    return logits, int(np.argmax(logits))
