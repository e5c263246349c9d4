"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of an oracle function (on the CPU, in
this process only) and checks that at least one pin of that function fails.
"""

import math

import numpy as np
import pytest

import oracle
import oracle.numerics as onum
import oracle.ops as oops
import test_oracle_numerics as tn
import test_oracle_ops as to


def _dequant_offset7(packed, scales, K, g):
    u = onum.unpack_int4(packed, K).astype(np.float64)
    s = np.asarray(scales, np.float16).astype(np.float64)
    N = u.shape[0]
    return ((u - 7.0).reshape(N, K // g, g) * s[:, :, None]).reshape(N, K)


def _unpack_swapped(packed, K):
    packed = np.asarray(packed, np.uint8)
    u = np.empty((packed.shape[0], K), np.uint8)
    u[:, 0::2] = packed >> 4
    u[:, 1::2] = packed & 0x0F
    return u


def _dequant_scale_by_row_block(packed, scales, K, g):
    u = onum.unpack_int4(packed, K).astype(np.float64)
    s = np.asarray(scales, np.float16).astype(np.float64)
    N = u.shape[0]
    # wrong index: scale chosen by k % (K/g) instead of k // g
    idx = np.arange(K) % (K // g)
    return (u - 8.0) * s[:, idx]


def _rope_sign(x, pos, base):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    h = d // 2
    th = base ** (-2.0 * np.arange(h) / d)
    a = pos * th
    c, s = np.cos(a), np.sin(a)
    return np.concatenate([x[..., :h] * c + x[..., h:] * s, x[..., h:] * c - x[..., :h] * s], -1)


def _rope_adjacent_pairs(x, pos, base):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    th = base ** (-2.0 * np.arange(d // 2) / d)
    a = pos * th
    c, s = np.cos(a), np.sin(a)
    y = x.copy()
    y[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    y[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return y


def _attn_no_scale(q, K, V):
    q, K, V = (np.asarray(a, np.float64) for a in (q, K, V))
    qh, d = q.shape
    grp = qh // K.shape[0]
    out = np.empty_like(q)
    for h in range(qh):
        s = K[h // grp] @ q[h]
        p = np.exp(s - s.max())
        out[h] = (p / p.sum()) @ V[h // grp]
    return out


def _attn_gqa_modulo(q, K, V):
    q, K, V = (np.asarray(a, np.float64) for a in (q, K, V))
    qh, d = q.shape
    out = np.empty_like(q)
    for h in range(qh):
        kv = h % K.shape[0]
        s = K[kv] @ q[h] / math.sqrt(d)
        p = np.exp(s - s.max())
        out[h] = (p / p.sum()) @ V[kv]
    return out


def _causal_strict(Q, K, V, start):
    # wrong mask: a row does not see its own position
    Q, K, V = (np.asarray(a, np.float64) for a in (Q, K, V))
    P, qh, d = Q.shape
    L = K.shape[1]
    vis = np.arange(L)[None, :] < (start + np.arange(P))[:, None]
    out = np.zeros((P, qh, d))
    for h in range(qh):
        kv = h // (qh // K.shape[0])
        S = np.where(vis, Q[:, h] @ K[kv].T / math.sqrt(d), -np.inf)
        E = np.nan_to_num(np.exp(S - S.max(1, keepdims=True)))
        out[:, h] = E / np.maximum(E.sum(1, keepdims=True), 1e-300) @ V[kv]
    return out


def _causal_no_offset(Q, K, V, start):
    # wrong mask: row i sees positions 0..i, ignoring the prefix length
    Q, K, V = (np.asarray(a, np.float64) for a in (Q, K, V))
    P, qh, d = Q.shape
    L = K.shape[1]
    vis = np.arange(L)[None, :] <= np.arange(P)[:, None]
    out = np.zeros((P, qh, d))
    for h in range(qh):
        kv = h // (qh // K.shape[0])
        S = np.where(vis, Q[:, h] @ K[kv].T / math.sqrt(d), -np.inf)
        E = np.exp(S - S.max(1, keepdims=True))
        out[:, h] = E / E.sum(1, keepdims=True) @ V[kv]
    return out


def _route_ties_high(xn, Wr, k, renorm=True):
    logits = np.asarray(xn, np.float64) @ np.asarray(Wr, np.float64).T
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    E = p.shape[1]
    ids = np.array([(E - 1 - np.argsort(-p[b][::-1], kind="stable"))[:k] for b in range(len(p))])
    w = np.take_along_axis(p, ids, 1)
    return ids.astype(np.int32), w / w.sum(1, keepdims=True)


def _route_no_renorm(xn, Wr, k, renorm=True):
    ids, _ = oops.route_topk(xn, Wr, k, renorm)
    logits = np.asarray(xn, np.float64) @ np.asarray(Wr, np.float64).T
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    return ids, np.take_along_axis(p, ids, 1)


def _rmsnorm_sum(x, weight=None, eps=1e-6):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps)


def _combine_no_residual(h, outs, weights):
    return sum(w * np.asarray(o, np.float64) for w, o in zip(weights, outs))


def _silu_wrong(x):
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(x))


def _gemm_transposed_scale(X, packed, scales, K, g):
    W = _dequant_scale_by_row_block(packed, scales, K, g)
    return np.asarray(X, np.float64) @ W.T


MUTANTS = [
    ("dequant offset 7", [(oracle, "dequant_w4"), (oops, "dequant_w4")], _dequant_offset7,
     [tn.test_int4_dequant_hand_values, tn.test_int4_dequant_exhaustive_codes, to.test_gemm_hand_value]),
    ("nibble order swapped", [(oracle, "unpack_int4"), (onum, "unpack_int4")], _unpack_swapped,
     [tn.test_int4_dequant_hand_values, tn.test_quantize_hand_values, to.test_gemm_closed_forms_and_row_independence]),
    ("scale index", [(oracle, "dequant_w4"), (oops, "dequant_w4")], _dequant_scale_by_row_block,
     [tn.test_int4_group_scale_indexing]),
    ("gemm scale index", [(oracle, "w4_gemm")], _gemm_transposed_scale,
     [to.test_gemm_brute_force_tiny]),
    ("rope sign", [(oracle, "rope_rotate_half")], _rope_sign,
     [to.test_rope_hand_value]),
    ("rope pairing", [(oracle, "rope_rotate_half")], _rope_adjacent_pairs,
     [to.test_rope_hand_value]),
    ("attention scale", [(oracle, "slot_attention")], _attn_no_scale,
     [to.test_attention_hand_value, to.test_attention_brute_force_and_gqa_map]),
    ("gqa map", [(oracle, "slot_attention")], _attn_gqa_modulo,
     [to.test_attention_special_cases, to.test_attention_brute_force_and_gqa_map]),
    ("causal mask strict", [(oracle, "causal_block_attention")], _causal_strict,
     [to.test_causal_block_attention_brute_force_and_causality]),
    ("causal mask offset", [(oracle, "causal_block_attention")], _causal_no_offset,
     [to.test_causal_block_attention_brute_force_and_causality]),
    ("router ties", [(oracle, "route_topk")], _route_ties_high,
     [to.test_router_hand_values]),
    ("router renorm", [(oracle, "route_topk")], _route_no_renorm,
     [to.test_router_hand_values, to.test_router_invariants]),
    ("rmsnorm sum", [(oracle, "rmsnorm")], _rmsnorm_sum,
     [to.test_rmsnorm_hand_and_invariants]),
    ("combine residual", [(oracle, "moe_combine")], _combine_no_residual,
     [to.test_expert_ffn_special_cases]),
    ("silu sign", [(oracle, "silu")], _silu_wrong,
     [to.test_silu_values]),
]


@pytest.mark.parametrize("name,targets,mutant,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, name, targets, mutant, pins):
    for mod, attr in targets:
        monkeypatch.setattr(mod, attr, mutant)
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught the planted mistake: {name}"


# ---------------------------------------------------------------- prompt ingestion (model level)

def _prefill_layer_positions_from_zero(cfg, lw, x, slot, kv, layer, trace=None):
    # wrong: the prompt's rows are rotated at 0..P-1, ignoring the slot's prefix
    import oracle.model as om
    H, qh, kvh, d, g = cfg.hidden, cfg.q_heads, cfg.kv_heads, cfg.head_dim, cfg.group
    x = np.asarray(x, dtype=np.float64)
    P = x.shape[0]
    start = kv.map.length[slot]
    xn = om._round(om.rmsnorm(x, lw.get("attn_norm"), cfg.eps))
    qkv = om._round(om.rowwise(om.dequant_w4(lw["wqkv"][0], lw["wqkv"][1], H, g), xn))
    q = qkv[:, : qh * d].reshape(P, qh, d)
    k = qkv[:, qh * d: (qh + kvh) * d].reshape(P, kvh, d)
    v = qkv[:, (qh + kvh) * d:].reshape(P, kvh, d)
    pos = np.arange(P)
    q_rot = om._round(om.rope_rotate_half(q, pos, cfg.rope_base))
    k_rot = om._round(om.rope_rotate_half(k, pos, cfg.rope_base))
    kv.write_block(layer, slot, k_rot, v)
    Kc, Vc = kv.view(layer, slot, start + P)
    o = om._round(om.causal_block_attention(q_rot, Kc, Vc, start)).reshape(P, qh * d)
    return om._after_attention(cfg, lw, x, o, trace)


def _block_attention_unmasked(Q, K, V, start):
    # wrong: every row of the prompt sees the whole block (no causal mask)
    Q, K, V = (np.asarray(a, np.float64) for a in (Q, K, V))
    P, qh, d = Q.shape
    out = np.empty((P, qh, d))
    for h in range(qh):
        kv = h // (qh // K.shape[0])
        S = Q[:, h] @ K[kv].T / math.sqrt(d)
        E = np.exp(S - S.max(1, keepdims=True))
        out[:, h] = E / E.sum(1, keepdims=True) @ V[kv]
    return out


PREFILL_MUTANTS = [
    ("prompt positions from zero", "prefill_layer", _prefill_layer_positions_from_zero),
    ("prompt attention unmasked", "causal_block_attention", _block_attention_unmasked),
]


@pytest.mark.parametrize("name,attr,mutant", PREFILL_MUTANTS, ids=[m[0] for m in PREFILL_MUTANTS])
def test_decode_equivalence_catches_prefill_mutant(monkeypatch, name, attr, mutant):
    import oracle.model as om
    import test_oracle_model as tmod
    cfg = tmod.oracle_config(tmod.CFG, layers=tmod.LAYERS, max_streams=6, ctx_cap=128)
    w = tmod.oracle_weights(tmod.NAME, tmod.CFG, tmod.LAYERS)
    tmod.test_prefill_equals_token_by_token_decode((cfg, w))   # the pin holds on the oracle as written
    monkeypatch.setattr(om, attr, mutant)
    with pytest.raises(AssertionError):
        tmod.test_prefill_equals_token_by_token_decode((cfg, w))


# ---------------------------------------------------------------- decoder-layer composition

def _layer_mutant(mistake):
    """A copy of the oracle's decoder layer with one composition mistake."""
    import oracle.model as om

    def after_attention(cfg, lw, x, o, trace=None):
        H, qh, d, g = cfg.hidden, cfg.q_heads, cfg.head_dim, cfg.group
        B = x.shape[0]
        Wo = om.dequant_w4(lw["wo"][0], lw["wo"][1], qh * d, g)
        h = om._round(x + om.rowwise(Wo, o))
        norm_w = None if mistake == "ffn norm weight dropped" else lw.get("ffn_norm")
        hn = om.rmsnorm(h, norm_w, cfg.eps)
        if mistake != "hn not rounded":
            hn = om._round(hn)
        ids, w = om.route_topk(h if mistake == "router reads h" else hn, lw["wr"], cfg.top_k, cfg.renorm_topk)
        xin = h if mistake == "experts read h" else hn
        y = np.empty_like(h)
        outs = np.empty((B, cfg.top_k, H))
        for b in range(B):
            acc = np.zeros(H)
            for r in range(cfg.top_k):
                ew = lw["expert"](int(ids[b, r]))
                Wg = om.dequant_w4(ew["wg"][0], ew["wg"][1], H, g)
                Wu = om.dequant_w4(ew["wu"][0], ew["wu"][1], H, g)
                Wd = om.dequant_w4(ew["wd"][0], ew["wd"][1], cfg.ffn, g)
                a = om._round(om.silu(Wg @ xin[b]) * (Wu @ xin[b]))
                outs[b, r] = Wd @ a
                acc = acc + w[b, r] * outs[b, r]
            y[b] = om._round((hn[b] if mistake == "combine residual from hn" else h[b]) + acc)
        if trace is not None:
            trace.update(dict(h=h, hn=hn, ids=ids, w=w, expert_out=outs, y=y))
        return y

    def decoder_layer(cfg, lw, x, slots, kv, layer, trace=None):
        H, qh, kvh, d, g = cfg.hidden, cfg.q_heads, cfg.kv_heads, cfg.head_dim, cfg.group
        x = np.asarray(x, dtype=np.float64)
        B = x.shape[0]
        xn = om._round(om.rmsnorm(x, lw.get("attn_norm"), cfg.eps))
        qkv = om._round(om.rowwise(om.dequant_w4(lw["wqkv"][0], lw["wqkv"][1], H, g), xn))
        q = qkv[:, : qh * d].reshape(B, qh, d)
        k = qkv[:, qh * d: (qh + kvh) * d].reshape(B, kvh, d)
        v = qkv[:, (qh + kvh) * d:].reshape(B, kvh, d)
        if mistake == "v taken from the k rows":
            v = k
        o = np.empty((B, qh * d))
        q_rot = np.empty_like(q)
        for b in range(B):
            pos = kv.map.length[slots[b]]
            q_rot[b] = om._round(om.rope_rotate_half(q[b], pos, cfg.rope_base))
            k_rot = om._round(om.rope_rotate_half(k[b], pos, cfg.rope_base))
            if mistake == "attention before the append":
                Kc, Vc = kv.view(layer, slots[b], pos)
                kv.write_pending(layer, slots[b], k_rot, v[b])
            else:
                kv.write_pending(layer, slots[b], k_rot, v[b])
                Kc, Vc = kv.view(layer, slots[b], pos + 1)
            o[b] = om._round(om.slot_attention(q_rot[b], Kc, Vc)).reshape(-1)
        y = after_attention(cfg, lw, xn if mistake == "attention residual from xn" else x, o, trace)
        if trace is not None:
            trace.update(dict(xn=xn, qkv=qkv, q_rot=q_rot, attn=o))
        return y

    return decoder_layer


LAYER_MUTANTS = ["attention residual from xn", "combine residual from hn", "router reads h", "experts read h",
                 "ffn norm weight dropped", "hn not rounded", "attention before the append",
                 "v taken from the k rows"]


def test_layer_golden_holds_on_the_oracle_and_its_copy():
    import test_oracle_layer_golden as tl
    tl.check_layer()
    orig = None
    import oracle.model as om
    orig, om.decoder_layer = om.decoder_layer, _layer_mutant("none")
    try:
        tl.check_layer()   # the copy without a mistake passes: the mutants differ by their mistake only
    finally:
        om.decoder_layer = orig


@pytest.mark.parametrize("mistake", LAYER_MUTANTS)
def test_layer_golden_catches_composition_mutant(monkeypatch, mistake):
    import oracle.model as om
    import test_oracle_layer_golden as tl
    monkeypatch.setattr(om, "decoder_layer", _layer_mutant(mistake))
    with pytest.raises(AssertionError):
        tl.check_layer()
