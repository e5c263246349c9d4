"""GPU parity of prompt ingestion (kv_slot_prefill).

A prompt runs through the decode kernels in blocks of max_streams rows of
one slot.  Checked here: the last-position logits, the greedy id and the K/V
written at every prompt position against the oracle's causal block prefill;
byte identity (arena, logits, next id, length) with feeding the same prompt
through single-stream decode steps; blocks with a ragged tail, a prompt that
crosses a 128-position attention chunk, an empty prefix, the graph path
against the eager path with its launch count, a decode step after the
prompt, a bystander slot left byte-identical, and the argument checks."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_side import build_engine, seed_stream
from oracle_side import oracle_config, oracle_weights
from parity import assert_close_rows, check_greedy

pytestmark = pytest.mark.gpu

NAME = "tiny_layer"
CFG = synth.CONFIGS[NAME]
MMA = 3


@pytest.fixture(scope="module")
def bm():
    import bit_moe_decode_w4a16_gb300 as m
    m.build()
    return m


def logit_bound(layers):
    """The specified 2e-2 max-abs bound at every depth these tests run (their
    measured logit errors stay below 0.008 at two layers)."""
    return 2e-2


def _prefill(bm, e, slot, toks, V):
    nxt = torch.empty(1, dtype=torch.int32)
    logits = torch.empty(V, dtype=torch.float32, device="cuda")
    bm.kv_slot_prefill(e, slot, torch.tensor(toks, dtype=torch.int32), nxt, logits)
    bm.bm_engine_sync(e)
    return int(nxt[0]), logits


def _decode_prompt(bm, e, slot, toks, V):
    """The prompt fed one single-stream decode step at a time."""
    nxt = torch.empty(1, dtype=torch.int32)
    logits = torch.empty((1, V), dtype=torch.float32, device="cuda")
    for t in toks:
        bm.decode_step(e, [slot], torch.tensor([t], dtype=torch.int32), nxt, logits)
    bm.bm_engine_sync(e)
    return int(nxt[0]), logits[0]


def _read(bm, e, cfg, layer, slot, n):
    K = torch.empty((cfg["kv_heads"], n, cfg["head_dim"]), dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    bm.kv_slot_read(e, layer, slot, n, K, V)
    bm.bm_engine_sync(e)
    return K, V


def _seed(bm, e, name, cfg, stream, L0, layers):
    k, v = synth.kv_prefix(name, cfg, stream, L0, layers=layers)
    return bm.kv_slot_seed(e, k.cuda().contiguous(), v.cuda().contiguous(), L0)


def _oracle_prefill(name, cfg, layers, cap, stream, L0, toks, max_streams=4):
    ocfg = oracle_config(cfg, layers=layers, max_streams=max_streams, ctx_cap=cap)
    ow = oracle_weights(name, cfg, layers)
    kv = oracle.OracleKV(ocfg, oracle.OracleSlotMap(ocfg.max_streams, ocfg.ctx_cap))
    k, v = synth.kv_prefix(name, cfg, stream, L0, layers=layers)
    s = kv.seed(k.double().numpy(), v.double().numpy())
    logits, nxt = oracle.model_prefill(ocfg, ow, kv, s, toks)
    return logits, nxt, kv, s


def _check_against_decode_and_oracle(bm, e, name, cfg, layers, cap, L0, toks, what):
    V = cfg["vocab"]
    P = len(toks)
    # a bystander stream whose slot neither the prompt nor the decode steps may touch
    L_by = 23
    s_by = _seed(bm, e, name, cfg, 3, L_by, layers)
    by_before = [_read(bm, e, cfg, l, s_by, L_by) for l in range(layers)]
    sa = _seed(bm, e, name, cfg, 0, L0, layers)
    sb = _seed(bm, e, name, cfg, 0, L0, layers)
    nxt_a, logits_a = _prefill(bm, e, sa, toks, V)
    nxt_b, logits_b = _decode_prompt(bm, e, sb, toks, V)
    assert bm.kv_slot_length(e, sa) == bm.kv_slot_length(e, sb) == L0 + P
    assert bm.kv_slot_length(e, s_by) == L_by
    for l in range(layers):
        Kx, Vx = _read(bm, e, cfg, l, s_by, L_by)
        assert torch.equal(Kx, by_before[l][0]) and torch.equal(Vx, by_before[l][1]), f"{what}: bystander slot changed"
    bm.kv_slot_release(e, s_by)
    # byte identity with teacher-forced decode
    assert torch.equal(logits_a, logits_b), f"{what}: prompt logits differ from decode bytes"
    assert nxt_a == nxt_b
    for l in range(layers):
        Ka, Va = _read(bm, e, cfg, l, sa, L0 + P)
        Kb, Vb = _read(bm, e, cfg, l, sb, L0 + P)
        assert torch.equal(Ka, Kb) and torch.equal(Va, Vb), f"{what}: layer {l} K/V differ from decode bytes"
    # the oracle's causal block prefill
    ref, ref_id, kv, so = _oracle_prefill(name, cfg, layers, cap, 0, L0, toks)
    err, _ = assert_close_rows(logits_a[None], ref[None], max_abs=logit_bound(layers), what=f"{what}: logits",
                               bf16_out=False)
    check_greedy([nxt_a], ref[None], err)
    for l in range(layers):
        Ka, Va = _read(bm, e, cfg, l, sa, L0 + P)
        assert_close_rows(Ka[:, L0:], kv.K[so][l][:, L0:], what=f"{what}: layer {l} prompt k (rotated)")
        assert_close_rows(Va[:, L0:], kv.V[so][l][:, L0:], what=f"{what}: layer {l} prompt v")
        if L0:
            k0, v0 = synth.kv_prefix(name, cfg, 0, L0, layers=layers)
            assert torch.equal(Ka[:, :L0].cpu(), k0[l]) and torch.equal(Va[:, :L0].cpu(), v0[l])
    return sa, sb, nxt_a


@pytest.mark.parametrize("L0,P", [(17, 9), (120, 13), (0, 6), (40, 1)],
                         ids=["ragged_tail", "crosses_chunk", "empty_prefix", "one_token"])
def test_tiny_prefill_matches_oracle_and_decode_bytes(bm, L0, P):
    layers = 2
    toks = [int(t) for t in synth.tokens(NAME, f"prompt_{L0}", P, CFG["vocab"])]
    e = build_engine(NAME, CFG, layers, max_streams=4, ctx_cap=256, policy=MMA, gen_device="cpu")
    try:
        sa, sb, nxt = _check_against_decode_and_oracle(bm, e, NAME, CFG, layers, 256, L0, toks,
                                                       f"tiny prefill {L0}+{P}")
        # decoding on from the prompt: both slots give the same bytes
        out = []
        for s in (sa, sb):
            n1 = torch.empty(1, dtype=torch.int32)
            l1 = torch.empty((1, CFG["vocab"]), dtype=torch.float32, device="cuda")
            bm.decode_step(e, [s], torch.tensor([nxt], dtype=torch.int32), n1, l1)
            bm.bm_engine_sync(e)
            out.append((int(n1[0]), l1))
        assert out[0][0] == out[1][0] and torch.equal(out[0][1], out[1][1])
    finally:
        bm.bm_engine_destroy(e)


def test_prefill_graph_eager_and_launch_count(bm):
    layers = 1
    toks = [int(t) for t in synth.tokens(NAME, "prompt_graph", 9, CFG["vocab"])]
    eg = build_engine(NAME, CFG, layers, max_streams=4, ctx_cap=128, policy=MMA, gen_device="cpu")
    ee = build_engine(NAME, CFG, layers, max_streams=4, ctx_cap=128, policy=MMA, use_graph=0, gen_device="cpu")
    try:
        s_g = _seed(bm, eg, NAME, CFG, 1, 10, layers)
        s_e = _seed(bm, ee, NAME, CFG, 1, 10, layers)
        st0 = bm.bm_engine_stats(eg)
        n_g, l_g = _prefill(bm, eg, s_g, toks, CFG["vocab"])
        n_e, l_e = _prefill(bm, ee, s_e, toks, CFG["vocab"])
        assert torch.equal(l_g, l_e) and n_g == n_e
        Kg, Vg = _read(bm, eg, CFG, 0, s_g, 19)
        Ke, Ve = _read(bm, ee, CFG, 0, s_e, 19)
        assert torch.equal(Kg, Ke) and torch.equal(Vg, Ve)
        st1 = bm.bm_engine_stats(eg)
        # blocks of 4, 4, 1: one graph launch each, two shapes captured
        assert st1["graph_launches"] - st0["graph_launches"] == 3
        assert st1["graph_captures"] - st0["graph_captures"] == 2
        # per block: embed, 8 per layer (append, attention, qkv, o_proj, routing,
        # gate/up, down, combine), then the length advance or the output projection
        assert st1["kernel_launches"] - st0["kernel_launches"] == 3 * (1 + 8 * layers + 1)
        # a second prompt of the same shape reuses the graphs
        s2 = _seed(bm, eg, NAME, CFG, 2, 3, layers)
        _prefill(bm, eg, s2, toks, CFG["vocab"])
        assert bm.bm_engine_stats(eg)["graph_captures"] == st1["graph_captures"]
        # device-resident tokens and output take the same path
        s3 = _seed(bm, eg, NAME, CFG, 1, 10, layers)
        nd = torch.empty(1, dtype=torch.int32, device="cuda")
        bm.kv_slot_prefill(eg, s3, torch.tensor(toks, dtype=torch.int32, device="cuda"), nd)
        bm.bm_engine_sync(eg)
        assert int(nd.cpu()[0]) == n_g
    finally:
        bm.bm_engine_destroy(eg)
        bm.bm_engine_destroy(ee)


def test_prefill_rejections_leave_the_slot_alone(bm):
    layers = 1
    e = build_engine(NAME, CFG, layers, max_streams=4, ctx_cap=64, policy=MMA, gen_device="cpu")
    try:
        s = _seed(bm, e, NAME, CFG, 0, 60, layers)
        K0, V0 = _read(bm, e, CFG, 0, s, 60)
        nxt = torch.empty(1, dtype=torch.int32)
        with pytest.raises(bm.BitMoeError) as ei:      # 60 + 5 > 64
            bm.kv_slot_prefill(e, s, torch.arange(5, dtype=torch.int32), nxt)
        assert ei.value.status == 2
        with pytest.raises(bm.BitMoeError) as ei:
            bm.kv_slot_prefill(e, s, torch.zeros(0, dtype=torch.int32), nxt)
        assert ei.value.status == 1
        with pytest.raises(bm.BitMoeError) as ei:
            bm.kv_slot_prefill(e, 3, torch.arange(2, dtype=torch.int32), nxt)
        assert ei.value.status == 4                      # slot 3 is free
        with pytest.raises(bm.BitMoeError) as ei:
            bm.kv_slot_prefill(e, 7, torch.arange(2, dtype=torch.int32), nxt)
        assert ei.value.status == 1                      # out of range
        assert bm.kv_slot_length(e, s) == 60
        K1, V1 = _read(bm, e, CFG, 0, s, 60)
        assert torch.equal(K0, K1) and torch.equal(V0, V1)
        # exactly up to the cap is accepted
        bm.kv_slot_prefill(e, s, torch.arange(4, dtype=torch.int32), nxt)
        bm.bm_engine_sync(e)
        assert bm.kv_slot_length(e, s) == 64
    finally:
        bm.bm_engine_destroy(e)
    # other kernel families do not take prompts
    e = build_engine(NAME, CFG, 1, max_streams=4, ctx_cap=64, policy=2, gen_device="cpu")
    try:
        s = _seed(bm, e, NAME, CFG, 0, 5, 1)
        with pytest.raises(bm.BitMoeError) as ei:
            bm.kv_slot_prefill(e, s, torch.arange(3, dtype=torch.int32), torch.empty(1, dtype=torch.int32))
        assert ei.value.status == 9
    finally:
        bm.bm_engine_destroy(e)


def test_prefill_at_full_width(bm):
    # One layer of the 30B-class shape, blocks of 32 rows: a 40-token prompt
    # (32 + a ragged 8) from a 100-position prefix, across the 128-position
    # chunk boundary; bf16 head of vocab 4096.
    cfg = dict(synth.CONFIGS["full_model"])
    cfg["vocab"] = 4096
    layers, cap = 1, 256
    toks = [int(t) for t in synth.tokens("full_width", "prompt", 40, cfg["vocab"])]
    e = build_engine("full_width", cfg, layers, max_streams=32, ctx_cap=cap, policy=MMA, gen_device="cpu")
    try:
        _check_against_decode_and_oracle(bm, e, "full_width", cfg, layers, cap, 100, toks, "full-width prefill")
    finally:
        bm.bm_engine_destroy(e)
