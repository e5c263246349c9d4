"""GPU parity of the grouped int4 expert op: 128 experts top-8, hidden 2048,
FFN 768, group 64, B in {1, 4, 8, 16, 32}, natural routing and a forced
overlap where every stream picks experts 0..7; plus the tiny layer's expert
shape (8 experts top-2, hidden 512, FFN 256, group 32)."""

import functools

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_rows, topk_near_tie

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bm():
    import bit_moe_decode_w4a16_gb300 as m
    m.build()
    return m


def _bank(bm, name, cfg, layer=0):
    """GPU bank (product encoder) and an oracle-side lazy accessor (oracle
    encoder) of the same raw weights (drawn on the CPU)."""
    E, H, F, g = cfg["experts"], cfg["hidden"], cfg["ffn"], cfg["group"]
    shapes = {"wg": (F, H), "wu": (F, H), "wd": (H, F)}
    dev = {}
    for kind, (rows, K) in shapes.items():
        packed = torch.empty((E, rows, K // 2), dtype=torch.uint8, device="cuda")
        scales = torch.empty((E, rows, K // g), dtype=torch.float16, device="cuda")
        for e in range(E):
            raw = synth.model_tensor(name, cfg, kind, layer, e)
            bm.bm_w4_quantize(raw.cuda(), rows, K, g, packed[e], scales[e])
        dev[kind] = (packed, scales)
    torch.cuda.synchronize()

    @functools.lru_cache(maxsize=None)
    def ora(e):
        return {kind: oracle.quantize_w4(synth.model_tensor(name, cfg, kind, layer, e).numpy(), g)
                for kind in shapes}
    return dev, ora


def _run(bm, cfg, dev, wr, X, R):
    B, H, k = X.shape[0], cfg["hidden"], cfg["top_k"]
    w = {"experts": cfg["experts"], "top_k": k, "hidden": H, "ffn": cfg["ffn"], "group": cfg["group"],
         "renorm_topk": 1, "wr": wr, "wg": dev["wg"][0], "wg_s": dev["wg"][1], "wu": dev["wu"][0],
         "wu_s": dev["wu"][1], "wd": dev["wd"][0], "wd_s": dev["wd"][1]}
    nbytes = bm.bm_moe_workspace_bytes(B, cfg["experts"], k, H, cfg["ffn"])
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    Y = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((B, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((B, k), dtype=torch.float32, device="cuda")
    bm.moe_grouped_w4(w, X, R, Y, ids, tw, B, ws, nbytes)
    torch.cuda.synchronize()
    return Y, ids.cpu().numpy(), tw.cpu().numpy()


def _oracle(cfg, ora, wr, X, R):
    H, F, g, k = cfg["hidden"], cfg["ffn"], cfg["group"], cfg["top_k"]
    x = X.double().numpy()
    r = R.double().numpy()
    logits = x @ wr.double().numpy().T
    ids, w = oracle.route_topk(x, wr.numpy(), k)
    Y = np.empty_like(x)
    for b in range(x.shape[0]):
        outs = [oracle.expert_ffn(x[b], ora(int(e))["wg"], ora(int(e))["wu"], ora(int(e))["wd"], H, F, g,
                                  oracle.bf16_round) for e in ids[b]]
        Y[b] = oracle.bf16_round(oracle.moe_combine(r[b], outs, w[b]))
    return Y, ids, w, logits


EXPERTS = synth.CONFIGS["expert_op"]
CFG3 = dict(experts=EXPERTS["experts"], top_k=EXPERTS["top_k"], hidden=EXPERTS["hidden"], ffn=EXPERTS["ffn"],
            group=EXPERTS["group"], q_heads=1, kv_heads=1, head_dim=1, vocab=1)


@pytest.fixture(scope="module")
def bank3(bm):
    return _bank(bm, "expert_op", CFG3)


def _inputs(case, B, cfg):
    H, E = cfg["hidden"], cfg["experts"]
    wr = synth.model_tensor("expert_op", cfg, "wr", 0)
    X = synth.activations("expert_op", f"x_{case}", (B, H))
    if case == "forced":
        # every stream picks experts 0..7: their router rows lean positive and
        # the inputs are non-negative, so their logits dominate
        wr = wr.clone()
        wr[:8] += 0.05
        X = X.abs()
    R = synth.activations("expert_op", f"res_{case}", (B, H))
    return wr, X, R


@pytest.mark.parametrize("case", ["natural", "forced"])
@pytest.mark.parametrize("B", EXPERTS["batches"])
def test_grouped_experts_match_oracle(bm, bank3, case, B):
    dev, ora = bank3
    wr, X, R = _inputs(case, B, CFG3)
    Y, ids, tw = _run(bm, CFG3, dev, wr.cuda(), X.cuda(), R.cuda())
    Yr, ids_r, w_r, logits = _oracle(CFG3, ora, wr, X, R)
    ok = []
    for b in range(B):
        if topk_near_tie(logits[b], ids_r[b], 1e-4):
            continue   # either order of a near-tie is correct
        np.testing.assert_array_equal(ids[b], ids_r[b])
        ok.append(b)
    assert len(ok) >= max(1, B - 1)
    np.testing.assert_allclose(tw[ok], w_r[ok], rtol=1e-4, atol=1e-6)
    assert_close_rows(Y[ok], Yr[ok], what=f"moe {case} B={B}")
    if case == "forced":
        assert all(set(r) == set(range(8)) for r in ids)


def test_grouped_experts_solo_equals_batched(bm, bank3):
    dev, _ = bank3
    wr, X, R = _inputs("natural", 32, CFG3)
    wr, X, R = wr.cuda(), X.cuda(), R.cuda()
    Yb, _, _ = _run(bm, CFG3, dev, wr, X, R)
    for b in (0, 5, 31):
        Ys, _, _ = _run(bm, CFG3, dev, wr, X[b:b + 1].contiguous(), R[b:b + 1].contiguous())
        assert torch.equal(Ys.view(torch.int16), Yb[b:b + 1].view(torch.int16))
    # and inside another batch composition
    idx = [31, 2, 17, 5]
    Yp, _, _ = _run(bm, CFG3, dev, wr, X[idx].contiguous(), R[idx].contiguous())
    assert torch.equal(Yp.view(torch.int16), Yb[idx].view(torch.int16))


def test_tiny_layer_experts(bm):
    cfg = synth.CONFIGS["tiny_layer"]
    dev, ora = _bank(bm, "tiny_layer", cfg)
    wr = synth.model_tensor("tiny_layer", cfg, "wr", 0)
    X = synth.activations("tiny_layer", "moe_x", (5, cfg["hidden"]))
    R = synth.activations("tiny_layer", "moe_r", (5, cfg["hidden"]))
    Y, ids, tw = _run(bm, cfg, dev, wr.cuda(), X.cuda(), R.cuda())
    Yr, ids_r, w_r, logits = _oracle(cfg, ora, wr, X, R)
    np.testing.assert_array_equal(ids, ids_r)
    assert_close_rows(Y, Yr, what="tiny experts")
