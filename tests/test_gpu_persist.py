"""GPU checks of the persistent small-batch decode step (engines created with
persistent_step = 1: every layer of a step of B <= 8 rows in one cooperative
kernel).  It computes every value with the multi-kernel step's arithmetic,
so the checks are byte equality against a multi-kernel engine holding the
same weights and streams: logits, greedy ids, the residual rows after the
last layer and every slot's K/V, over a join/finish schedule whose batch
changes from step to step (the multi-kernel step itself is compared with
the oracle in test_gpu_step.py).  Also: a direct oracle comparison on the
tiny model, the launch count, the eager (no graph) form, and the bounded
waits: a weight unit that never arrives makes the step give up with device
check code 6, and the engine then decodes correctly again."""

import pytest
import torch

import oracle
import synth
from gpu_side import build_engine, seed_stream
from oracle_side import oracle_config, oracle_weights
from parity import assert_close_rows, check_greedy

pytestmark = pytest.mark.gpu

MMA = 3


@pytest.fixture(scope="module")
def bm():
    import bit_moe_decode_w4a16_gb300 as m
    m.build()
    return m


def _step(bm, e, slots, toks, V):
    B = len(slots)
    nxt = torch.empty(B, dtype=torch.int32)
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda")
    bm.decode_step(e, slots, torch.tensor(toks, dtype=torch.int32), nxt, logits)
    bm.bm_engine_sync(e)
    return nxt.numpy().copy(), logits


def _hidden(bm, e, B, H):
    out = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    bm.bm_engine_read_hidden(e, B, out)
    bm.bm_engine_sync(e)
    return out


def _slot_bytes(bm, e, layers, slot, cfg):
    n = bm.kv_slot_length(e, slot)
    out = []
    for l in range(layers):
        K = torch.empty((cfg["kv_heads"], n, cfg["head_dim"]), dtype=torch.bfloat16, device="cuda")
        V = torch.empty_like(K)
        bm.kv_slot_read(e, l, slot, n, K, V)
        out += [K, V]
    bm.bm_engine_sync(e)
    return out


def _schedule(name, cfg, layers, lens, batches, bm, ref, per, gen_device):
    """Seed the same streams on both engines, then run `batches` (lists of
    stream indices) as decode steps, feeding each stream its greedy token;
    every step's outputs must be equal byte for byte."""
    V, H = cfg["vocab"], cfg["hidden"]
    sr = [seed_stream(ref, name, cfg, i, L, layers, gen_device=gen_device) for i, L in enumerate(lens)]
    sp = [seed_stream(per, name, cfg, i, L, layers, gen_device=gen_device) for i, L in enumerate(lens)]
    tok = [int(t) for t in synth.tokens(name, "persist", len(lens), V)]
    for n, batch in enumerate(batches):
        toks = [tok[i] for i in batch]
        nr, lr = _step(bm, ref, [sr[i] for i in batch], toks, V)
        npz, lp = _step(bm, per, [sp[i] for i in batch], toks, V)
        where = f"step {n} (B={len(batch)}, streams {batch})"
        assert (nr == npz).all(), f"greedy ids differ at {where}: {nr} vs {npz}"
        assert torch.equal(lr, lp), f"logits differ at {where}: max |d| {(lr - lp).abs().max().item()}"
        assert torch.equal(_hidden(bm, ref, len(batch), H), _hidden(bm, per, len(batch), H)), f"hidden at {where}"
        for j, i in enumerate(batch):
            tok[i] = int(nr[j])
    for i in range(len(lens)):
        a, b = _slot_bytes(bm, ref, layers, sr[i], cfg), _slot_bytes(bm, per, layers, sp[i], cfg)
        assert all(torch.equal(x, y) for x, y in zip(a, b)), f"K/V bytes of stream {i} differ"
    for s in sr:
        bm.kv_slot_release(ref, s)
    for s in sp:
        bm.kv_slot_release(per, s)


TINY = "tiny_layer"
TCFG = synth.CONFIGS[TINY]


@pytest.mark.parametrize("use_graph", [1, 0], ids=["graph", "eager"])
def test_tiny_persistent_step_same_bytes_as_multikernel(bm, use_graph):
    layers = 2
    ref = build_engine(TINY, TCFG, layers, 8, 256, policy=MMA, gen_device="cpu")
    per = build_engine(TINY, TCFG, layers, 8, 256, policy=MMA, use_graph=use_graph, gen_device="cpu",
                       persistent_step=1)
    try:
        lens = [17, 40, 1, 127, 128, 129, 200, 63]
        batches = [[0], [1, 0], [2, 3, 4], list(range(8)), [7, 5], [6], list(range(8)), [3, 1, 4, 0, 7]]
        _schedule(TINY, TCFG, layers, lens, batches, bm, ref, per, "cpu")
        st = bm.bm_engine_stats(per)
        assert st["kernels_per_step"] == 3, st   # embedding, the persistent step, the output projection
        # the toggle: switched off, the same engine runs the multi-kernel step, switched on again the
        # persistent one, and the streams stay byte-equal throughout
        bm.bm_engine_set_persistent_step(per, 0)
        _schedule(TINY, TCFG, layers, [5, 90], [[0, 1], [1]], bm, ref, per, "cpu")
        assert bm.bm_engine_stats(per)["kernels_per_step"] > 3
        bm.bm_engine_set_persistent_step(per, 1)
        _schedule(TINY, TCFG, layers, [33, 2], [[1, 0], [0]], bm, ref, per, "cpu")
        assert bm.bm_engine_stats(per)["kernels_per_step"] == 3
        with pytest.raises(bm.BitMoeError):
            bm.bm_engine_set_persistent_step(ref, 1)   # created without it
    finally:
        bm.bm_engine_destroy(ref)
        bm.bm_engine_destroy(per)


def test_tiny_persistent_step_matches_oracle(bm):
    layers = 2
    lens = TCFG["lens"]
    toks = [int(t) for t in synth.tokens(TINY, "step", 2, TCFG["vocab"])]
    e = build_engine(TINY, TCFG, layers, 4, 128, policy=MMA, gen_device="cpu", persistent_step=1)
    try:
        slots = [seed_stream(e, TINY, TCFG, i, L, layers, gen_device="cpu") for i, L in enumerate(lens)]
        nxt, logits = _step(bm, e, slots, toks, TCFG["vocab"])
        ocfg = oracle_config(TCFG, layers=layers, max_streams=4, ctx_cap=128)
        ow = oracle_weights(TINY, TCFG, layers)
        kv = oracle.OracleKV(ocfg, oracle.OracleSlotMap(ocfg.max_streams, ocfg.ctx_cap))
        oslots = []
        for i, L in enumerate(lens):
            k, v = synth.kv_prefix(TINY, TCFG, i, L, layers=layers)
            oslots.append(kv.seed(k.double().numpy(), v.double().numpy()))
        ref_logits, _ = oracle.model_step(ocfg, ow, kv, oslots, toks)
        err, _ = assert_close_rows(logits, ref_logits, max_abs=2e-2, what="persistent tiny step logits",
                                   bf16_out=False)
        check_greedy(nxt, ref_logits, err)
    finally:
        bm.bm_engine_destroy(e)


FULL = "full_model"
FCFG = synth.CONFIGS[FULL]


def test_full_width_persistent_step_same_bytes_as_multikernel(bm):
    """Full width (hidden 2048, 128 experts top-8, 32/4 heads of 128), two
    layers: prefixes that end inside, at and past 128-position chunk
    boundaries, batches of 1 to 8 that change every step."""
    layers = 2
    ref = build_engine(FULL, FCFG, layers, 8, 1024, policy=MMA)
    per = build_engine(FULL, FCFG, layers, 8, 1024, policy=MMA, persistent_step=1)
    try:
        lens = [300, 17, 513, 128, 1, 700, 64, 255]
        batches = [[0], [0, 1], [2, 3, 4, 5], list(range(8)), [6], [7, 2, 0], list(range(8)), [5]]
        _schedule(FULL, FCFG, layers, lens, batches, bm, ref, per, "cuda")
    finally:
        bm.bm_engine_destroy(ref)
        bm.bm_engine_destroy(per)


def test_persistent_step_bounded_wait_gives_up_and_recovers(bm):
    layers = 2
    ref = build_engine(TINY, TCFG, layers, 4, 128, policy=MMA, gen_device="cpu")
    per = build_engine(TINY, TCFG, layers, 4, 128, policy=MMA, gen_device="cpu", persistent_step=1)
    try:
        lens = [17, 40]
        sp = [seed_stream(per, TINY, TCFG, i, L, layers, gen_device="cpu") for i, L in enumerate(lens)]
        toks = [int(t) for t in synth.tokens(TINY, "step", 2, TCFG["vocab"])]
        _step(bm, per, sp, toks, TCFG["vocab"])                     # a good step first
        bm.bm_engine_test_drop_persist_unit(per, 3)
        nxt = torch.empty(2, dtype=torch.int32)
        bm.decode_step(per, sp, torch.tensor(toks, dtype=torch.int32), nxt)
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_engine_sync(per)
        assert "code 6" in str(ei.value), str(ei.value)
        bm.bm_engine_test_drop_persist_unit(per, -1)
        for s in sp:
            bm.kv_slot_release(per, s)
        # fresh streams on both engines: the persistent engine is usable and exact again
        _schedule(TINY, TCFG, layers, lens, [[0, 1], [1], [0, 1]], bm, ref, per, "cpu")
    finally:
        bm.bm_engine_destroy(ref)
        bm.bm_engine_destroy(per)


def test_persistent_step_needs_the_mma_family(bm):
    from gpu_side import engine_config
    with pytest.raises(bm.BitMoeError):
        bm.bm_engine_create(engine_config(TCFG, 1, 4, 128, policy=1, persistent_step=1))
