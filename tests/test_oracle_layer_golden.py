"""Pin of the oracle's decoder-layer composition: one whole layer at toy size
against the hand-worked values of ``tests/golden/decoder_layer.txt`` (norm
placement and weights, residual sources, the bf16 rounding points, the q/k/v
split, the append before attention, the router's input, the expert FFN and
the combine).  Every expected value is exactly representable, so the trace
is compared exactly."""

import numpy as np

import oracle
import oracle.model as omodel
from golden_io import lines

GOLD = "decoder_layer.txt"


def golden():
    out = {}
    for tok in lines(GOLD):
        key, vals = tok[0], tok[1:]
        rows = [[]]
        for v in vals:
            if v == "|":
                rows.append([])
            else:
                rows[-1].append(float(v))
        out[key] = np.array(rows if len(rows) > 1 else rows[0], dtype=np.float64)
    return out


def _packed(codes, g=2):
    q = np.asarray(codes, dtype=np.int64)
    packed = oracle.pack_int4((q + 8).astype(np.uint8))
    scales = np.ones((q.shape[0], q.shape[1] // g), dtype=np.float16)
    return packed, scales


def toy_layer():
    """Config, layer weights, KV store with the seeded slot, and the input row."""
    G = golden()
    cfg = oracle.OracleConfig(hidden=4, q_heads=1, kv_heads=1, head_dim=2, experts=2, top_k=1, ffn=2, group=2,
                              vocab=4, layers=1, rope_base=1e4, eps=1e-6, ctx_cap=8, max_streams=2)
    experts = {e: {n: _packed(G[f"e{e}_{n}"]) for n in ("wg", "wu", "wd")} for e in (0, 1)}
    lw = {"wqkv": _packed(G["wqkv"]), "wo": _packed(G["wo"]), "wr": G["wr"].astype(np.float32),
          "expert": lambda e: experts[e], "attn_norm": None, "ffn_norm": G["ffn_norm"]}
    kv = oracle.OracleKV(cfg, oracle.OracleSlotMap(cfg.max_streams, cfg.ctx_cap))
    slot = kv.seed(G["seed_k"].reshape(1, 1, 1, 2), G["seed_v"].reshape(1, 1, 1, 2))
    return G, cfg, lw, kv, slot


def run_layer():
    G, cfg, lw, kv, slot = toy_layer()
    tr = {}
    y = omodel.decoder_layer(cfg, lw, G["x"][None, :], [slot], kv, 0, tr)
    return G, y, tr, kv, slot


def check_layer():
    """The layer's trace and output equal the hand-worked values exactly."""
    G, y, tr, kv, slot = run_layer()
    np.testing.assert_array_equal(tr["xn"][0], G["xn"])
    np.testing.assert_array_equal(tr["qkv"][0], G["qkv"])
    np.testing.assert_array_equal(tr["q_rot"][0].reshape(-1), G["q_rot"])
    np.testing.assert_array_equal(tr["attn"][0], G["attn"])
    np.testing.assert_array_equal(tr["h"][0], G["h"])
    np.testing.assert_array_equal(tr["hn"][0], G["hn"])
    np.testing.assert_array_equal(tr["ids"][0], G["ids"].astype(np.int32))
    np.testing.assert_array_equal(tr["w"][0], G["weights"])
    np.testing.assert_array_equal(tr["expert_out"][0, 0], G["expert_out"])
    np.testing.assert_array_equal(y[0], G["y"])
    K, V = kv.view(0, slot, 2)
    np.testing.assert_array_equal(K[0, 1], G["k_appended"])
    np.testing.assert_array_equal(V[0, 1], G["v_appended"])
    np.testing.assert_array_equal(K[0, 0], G["seed_k"])


def test_decoder_layer_matches_hand_worked_values():
    check_layer()
