"""moe_grouped_w4_noalloc, the grouped expert op for callers that cannot
allocate device memory (for example a plugin whose host engine owns the whole
device memory pool, or a latency-critical path where cudaMalloc is not
allowed): called through the C ABI, its output must match moe_grouped_w4 with
a caller-owned workspace, on two calls in a row (the second call runs on the
first call's leftover workspace contents).

The file is named to be collected last, so a run that stops at the first
failure has already run every other test."""

import numpy as np
import pytest
import torch

import synth
from parity import assert_close_rows

pytestmark = pytest.mark.gpu

CFG = dict(experts=32, top_k=8, hidden=2048, ffn=768, group=64, q_heads=1, kv_heads=1, head_dim=1, vocab=1)


@pytest.fixture(scope="module")
def setup():
    import bit_moe_decode_w4a16_gb300 as bm
    bm.build()
    E, H, F, g = CFG["experts"], CFG["hidden"], CFG["ffn"], CFG["group"]
    w = {"experts": E, "top_k": CFG["top_k"], "hidden": H, "ffn": F, "group": g, "renorm_topk": 1,
         "wr": synth.model_tensor("no_alloc", CFG, "wr", 0).cuda()}
    keep = [w["wr"]]
    for kind, (rows, K) in {"wg": (F, H), "wu": (F, H), "wd": (H, F)}.items():
        packed = torch.empty((E, rows, K // 2), dtype=torch.uint8, device="cuda")
        scales = torch.empty((E, rows, K // g), dtype=torch.float16, device="cuda")
        for e in range(E):
            bm.bm_w4_quantize(synth.model_tensor("no_alloc", CFG, kind, 0, e).cuda(), rows, K, g, packed[e], scales[e])
        w[kind], w[kind + "_s"] = packed, scales
        keep += [packed, scales]
    torch.cuda.synchronize()
    return bm, w


def _reference(bm, w, X, R, B):
    k = CFG["top_k"]
    nbytes = bm.bm_moe_workspace_bytes(B, CFG["experts"], k, CFG["hidden"], CFG["ffn"])
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    Y = torch.empty((B, CFG["hidden"]), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((B, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((B, k), dtype=torch.float32, device="cuda")
    bm.moe_grouped_w4(w, X, R, Y, ids, tw, B, ws, nbytes)
    torch.cuda.synchronize()
    return Y, ids, tw


def _no_alloc(bm, w, X, R, B):
    k = CFG["top_k"]
    Y = torch.empty((B, CFG["hidden"]), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((B, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((B, k), dtype=torch.float32, device="cuda")
    bm.moe_grouped_w4_noalloc(w, X, R, Y, ids, tw, B)
    torch.cuda.synchronize()
    return Y, ids, tw


@pytest.mark.parametrize("B", [1, 8, 32])
def test_no_alloc_matches_workspace_entry_point_twice(setup, B):
    bm, w = setup
    X = synth.activations("no_alloc", "x", (B, CFG["hidden"])).cuda()
    R = synth.activations("no_alloc", "r", (B, CFG["hidden"])).cuda()
    Y0, ids0, tw0 = _reference(bm, w, X, R, B)
    for call in range(2):
        Y, ids, tw = _no_alloc(bm, w, X, R, B)
        # the same kernels on the same inputs: the same bytes
        assert torch.equal(ids, ids0), f"call {call}: expert ids differ"
        assert torch.equal(tw, tw0), f"call {call}: expert weights differ"
        assert torch.equal(Y.view(torch.int16), Y0.view(torch.int16)), f"call {call}, B={B}: outputs differ"
        assert_close_rows(Y, Y0, what=f"no-alloc call {call}, B={B}")


def test_no_alloc_rejects_sizes_beyond_its_workspace(setup):
    bm, w = setup
    big = dict(w, experts=CFG["experts"])
    need = bm.bm_moe_workspace_bytes(128, CFG["experts"], CFG["top_k"], CFG["hidden"], CFG["ffn"])
    assert need > bm.bm_moe_noalloc_max_bytes()
    X = torch.zeros((128, CFG["hidden"]), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bm.BitMoeError) as ei:
        bm.moe_grouped_w4_noalloc(big, X, None, X, None, None, 128)
    assert ei.value.status == 1 and "workspace" in ei.value.message
