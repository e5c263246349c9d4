"""GPU parity of prompt ingestion on the tcgen05 tensor cores (prefill_tc):
the dense projections and the experts of every layer run as prompt-length
GEMMs (M = 128 weight rows x N = up to 128 prompt rows per CTA) over blocks
of up to 512 prompt rows.

Checked against the oracle's causal block prefill: the logits and greedy id
after the prompt and every prompt position's K/V, for prompts of 1, 13, 300
and 700 rows (one row; fewer rows than one MMA column group; several
attention launches and N tiles; two blocks), with and without a seeded
prefix, on the tiny layer (2 layers) and at full width (hidden 2048, 128
experts top-8).  Also: a prompt split over two calls leaves the same bytes
as the whole prompt in one (a row's result does not depend on the other rows
of its block), decode steps continue from the ingested prompt, and a
bystander slot keeps its bytes."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_side import build_engine
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


def _prefill(bm, e, slot, toks, V):
    nxt = torch.empty(1, dtype=torch.int32)
    logits = torch.empty(V, dtype=torch.float32, device="cuda")
    bm.kv_slot_prefill(e, slot, torch.tensor(toks, dtype=torch.int32), nxt, logits)
    bm.bm_engine_sync(e)
    return int(nxt[0]), logits


def _read(bm, e, cfg, layer, slot, n):
    K = torch.empty((cfg["kv_heads"], n, cfg["head_dim"]), dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    bm.kv_slot_read(e, layer, slot, n, K, V)
    bm.bm_engine_sync(e)
    return K, V


def _seed(bm, e, name, cfg, stream, L0, layers):
    k, v = synth.kv_prefix(name, cfg, stream, L0, layers=layers)
    return bm.kv_slot_seed(e, k.cuda().contiguous(), v.cuda().contiguous(), L0)


# Router logit gap below which the two sides may pick different experts
# (reading C-G: near-ties are reported, not failed).  The prompt GEMMs round
# each weight once (q x s in fp16), which moves a row's hidden state by about
# 1e-3 relative; the row's RMSNorm output then lands on the other side of up
# to a quarter of its bf16 rounding points, each moving a router logit by
# ~1.6e-4.  Measured: a 700-row prompt flipped the second expert of rows whose
# oracle gaps were 7e-5, 3.6e-4 and 2.6e-3; the band is twice the largest.
ROUTER_TIE = 5e-3


def _oracle(name, cfg, layers, cap, stream, L0, toks):
    ocfg = oracle_config(cfg, layers=layers, max_streams=4, ctx_cap=cap)
    ow = oracle_weights(name, cfg, layers)
    kv = oracle.OracleKV(ocfg, oracle.OracleSlotMap(ocfg.max_streams, ocfg.ctx_cap))
    k, v = synth.kv_prefix(name, cfg, stream, L0, layers=layers)
    s = kv.seed(k.double().numpy(), v.double().numpy())
    traces = []
    logits, nxt = oracle.model_prefill(ocfg, ow, kv, s, toks, traces=traces)
    # rows whose routing had a near-tie at layer l or before: their later
    # layers' values may legitimately differ (another expert)
    tied, acc = [], np.zeros(len(toks), dtype=bool)
    for l, tr in enumerate(traces):
        lg = tr["hn"] @ ow["layers"][l]["wr"].astype(np.float64).T
        top = np.sort(lg, axis=1)[:, ::-1][:, : ocfg.top_k + 1]
        acc = acc | (np.abs(np.diff(top, axis=1)) < ROUTER_TIE).any(axis=1)
        tied.append(acc.copy())
    return logits, ocfg, ow, kv, s, tied


def _check(bm, e, name, cfg, layers, cap, L0, toks, what):
    V = cfg["vocab"]
    s = _seed(bm, e, name, cfg, 0, L0, layers)
    nxt, logits = _prefill(bm, e, s, toks, V)
    # the same prompt into a second slot: the same bytes
    s2 = _seed(bm, e, name, cfg, 0, L0, layers)
    nxt2, logits2 = _prefill(bm, e, s2, toks, V)
    assert torch.equal(logits, logits2) and nxt == nxt2, f"{what}: a second ingestion differs"
    for l in range(layers):
        K1, V1 = _read(bm, e, cfg, l, s, L0 + len(toks))
        K2, V2 = _read(bm, e, cfg, l, s2, L0 + len(toks))
        assert torch.equal(K1, K2) and torch.equal(V1, V2), f"{what}: layer {l} second ingestion differs"
    bm.kv_slot_release(e, s2)
    assert bm.kv_slot_length(e, s) == L0 + len(toks)
    ref, ocfg, ow, kv, so, tied = _oracle(name, cfg, layers, cap, 0, L0, toks)
    if not tied[-1][-1]:
        err, _ = assert_close_rows(logits[None], ref[None], what=f"{what}: logits", bf16_out=False)
        check_greedy([nxt], ref[None], err)
    for l in range(layers):
        K, Vv = _read(bm, e, cfg, l, s, L0 + len(toks))
        # rows tied in an earlier layer's routing are left out from this layer on
        keep = np.nonzero(~tied[l - 1])[0] if l else np.arange(len(toks))
        assert len(toks) - len(keep) <= max(2, 0.05 * len(toks)), \
            f"{what}: {len(toks) - len(keep)} rows with router near-ties"
        # one row per prompt position: [P][kv heads x d]
        rows = lambda t: t.transpose(0, 1).reshape(t.shape[1], -1)
        Kg, Vg = K[:, L0:].float().cpu()[:, keep], Vv[:, L0:].float().cpu()[:, keep]
        Kr = torch.from_numpy(np.ascontiguousarray(kv.K[so][l][:, L0:][:, keep]))
        Vr = torch.from_numpy(np.ascontiguousarray(kv.V[so][l][:, L0:][:, keep]))
        for label, g_, r_ in (("k (rotated)", Kg, Kr), ("v", Vg, Vr)):
            d = (rows(g_).double() - rows(r_).double()).abs().amax(dim=1).numpy()
            far = keep[np.nonzero(d > 2e-2)[0]][:8].tolist()   # positions of rows past 2e-2 (a bf16 flip may pass)
            assert_close_rows(rows(g_), rows(r_), what=f"{what}: layer {l} prompt {label} (positions past 2e-2: {far})")
        if L0:
            k0, v0 = synth.kv_prefix(name, cfg, 0, L0, layers=layers)
            assert torch.equal(K[:, :L0].cpu(), k0[l]) and torch.equal(Vv[:, :L0].cpu(), v0[l])
    return s, nxt, ocfg, ow, kv, so


@pytest.fixture(scope="module")
def tiny(bm):
    e = build_engine(NAME, CFG, 2, max_streams=4, ctx_cap=1024, policy=MMA, gen_device="cpu", prefill_tc=1)
    yield e
    bm.bm_engine_destroy(e)


@pytest.mark.parametrize("L0,P", [(0, 1), (5, 13), (0, 300), (17, 700)])
def test_prefill_tc_tiny_matches_oracle(bm, tiny, L0, P):
    toks = [int(t) for t in synth.tokens(NAME, f"pftc{L0}_{P}", P, CFG["vocab"])]
    # a bystander slot that the prompt may not touch
    s_by = _seed(bm, tiny, NAME, CFG, 3, 23, 2)
    try:
        before = [_read(bm, tiny, CFG, l, s_by, 23) for l in range(2)]
        s, *_ = _check(bm, tiny, NAME, CFG, 2, 1024, L0, toks, f"tc prefill {L0}+{P}")
        for l in range(2):
            K, Vv = _read(bm, tiny, CFG, l, s_by, 23)
            assert torch.equal(K, before[l][0]) and torch.equal(Vv, before[l][1])
        assert bm.kv_slot_length(tiny, s_by) == 23
    finally:
        for slot in range(4):
            try:
                bm.kv_slot_release(tiny, slot)
            except bm.BitMoeError:
                pass


def test_prefill_tc_split_equals_whole_and_decode_continues(bm, tiny):
    P = 300
    toks = [int(t) for t in synth.tokens(NAME, "pftc_split", P, CFG["vocab"])]
    V = CFG["vocab"]
    sa = _seed(bm, tiny, NAME, CFG, 0, 9, 2)
    sb = _seed(bm, tiny, NAME, CFG, 0, 9, 2)
    try:
        _split_and_continue(bm, tiny, toks, V, P, sa, sb)
    finally:
        for slot in (sa, sb):
            try:
                bm.kv_slot_release(tiny, slot)
            except bm.BitMoeError:
                pass


def _split_and_continue(bm, tiny, toks, V, P, sa, sb):
    na, la = _prefill(bm, tiny, sa, toks, V)
    _prefill(bm, tiny, sb, toks[:170], V)
    nb, lb = _prefill(bm, tiny, sb, toks[170:], V)
    assert torch.equal(la, lb) and na == nb
    for l in range(2):
        Ka, Va = _read(bm, tiny, CFG, l, sa, 9 + P)
        Kb, Vb = _read(bm, tiny, CFG, l, sb, 9 + P)
        assert torch.equal(Ka, Kb) and torch.equal(Va, Vb), f"layer {l}: split prompt bytes differ"
    # decode steps after the prompt against the oracle continuing from its own prefill
    ref, ocfg, ow, kv, so, _ = _oracle(NAME, CFG, 2, 1024, 0, 9, toks)
    t = na
    nxt = torch.empty(1, dtype=torch.int32)
    logits = torch.empty((1, V), dtype=torch.float32, device="cuda")
    for k in range(3):
        bm.decode_step(tiny, [sa], torch.tensor([t], dtype=torch.int32), nxt, logits)
        bm.bm_engine_sync(tiny)
        r, _ = oracle.model_step(ocfg, ow, kv, [so], [t])
        err, _ = assert_close_rows(logits, r, what=f"decode step {k} after a tc prefill", bf16_out=False)
        check_greedy(nxt.numpy(), r, err)
        t = int(nxt[0])


def test_prefill_tc_full_width(bm):
    cfg = dict(synth.CONFIGS["full_model"])
    cfg["vocab"] = 4096
    e = build_engine("full_width", cfg, 1, max_streams=4, ctx_cap=1024, policy=MMA, gen_device="cpu", prefill_tc=1)
    try:
        toks = [int(t) for t in synth.tokens("full_width", "pftc", 300, cfg["vocab"])]
        _check(bm, e, "full_width", cfg, 1, 1024, 40, toks, "full-width tc prefill 40+300")
    finally:
        bm.bm_engine_destroy(e)


def test_prefill_tc_rejects_other_families(bm):
    cfg = dict(CFG)
    from gpu_side import engine_config
    with pytest.raises(bm.BitMoeError) as ei:
        bm.bm_engine_create(engine_config(cfg, 1, 4, 128, policy=1, prefill_tc=1))
    assert ei.value.status == 9
