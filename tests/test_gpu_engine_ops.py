"""GPU parity of the decode step's own hot kernels, one layer at a time,
through the engine-bound layer ops of the C ABI:

* the grouped expert op at 128 experts top-8, hidden 2048, FFN 768, group 64,
  B in {1, 4, 8, 16, 32}, natural routing and a forced overlap where every
  stream picks experts 0..7 (so each of those experts runs four jobs of eight
  rows and the staged kernels' stage ring wraps), through the step's routing
  kernel (router, top-k and grouping in one launch), the staged gate/up and
  down kernels and the combine; routed ids compared exactly, weights and
  outputs elementwise, solo against batched bytes;
* the step's fused attention (RoPE, append, chunked attention and merge) on a
  16-slot x 8192-position arena, 32 q / 4 kv heads of 128, ragged lengths,
  over a seeded 200-step join/finish schedule with B between 1 and 16: the
  output against the oracle, the appended k and v, and every continuing
  slot's bytes after every step;
* failure detection: a staged expert work item whose copies are never issued
  makes its consumers' bounded wait run out; the engine reports code 5 and
  stays usable.
"""

import functools

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_side import expert_bank, quantize_dev
from parity import assert_close_rows

pytestmark = pytest.mark.gpu

MMA = 3
NAME = "expert_op"
EX = synth.CONFIGS[NAME]
# the expert op's shapes inside the 30B-class layer geometry
CFG = dict(hidden=EX["hidden"], q_heads=32, kv_heads=4, head_dim=128, experts=EX["experts"], top_k=EX["top_k"],
           ffn=EX["ffn"], group=EX["group"], vocab=256, rope_base=1e4)
TIE_EPS = 1e-3   # router logit gap below which either order of two experts is correct


@pytest.fixture(scope="module")
def bm():
    import bit_moe_decode_w4a16_gb300 as m
    m.build()
    return m


def _wr(case):
    wr = synth.model_tensor(NAME, CFG, "wr", 0)
    if case == "forced":
        # every stream picks experts 0..7: their router rows lean positive and
        # the inputs are non-negative, so their logits dominate
        wr = wr.clone()
        wr[:8] += 0.05
    return wr


@pytest.fixture(scope="module")
def moe_engine(bm):
    """Layer 0 routes naturally, layer 1 is forced onto experts 0..7; both
    share one expert bank (the product encoder) and small dense weights."""
    cfg = {"hidden": CFG["hidden"], "q_heads": CFG["q_heads"], "kv_heads": CFG["kv_heads"],
           "head_dim": CFG["head_dim"], "experts": CFG["experts"], "top_k": CFG["top_k"], "ffn": CFG["ffn"],
           "group": CFG["group"], "vocab": CFG["vocab"], "layers": 2, "rope_base": 1e4, "rms_eps": 1e-6,
           "max_streams": 32, "ctx_cap": 256, "renorm_topk": 1, "kernel_policy": MMA, "use_graph": 0}
    e = bm.bm_engine_create(cfg)
    g = CFG["group"]
    wqkv = quantize_dev(synth.model_tensor(NAME, CFG, "wqkv", 0), g)
    wo = quantize_dev(synth.model_tensor(NAME, CFG, "wo", 0), g)
    wg, wu, wd = (expert_bank(NAME, CFG, 0, n, gen_device="cpu") for n in ("wg", "wu", "wd"))
    for layer, case in enumerate(("natural", "forced")):
        w = {"wqkv": wqkv[0], "wqkv_s": wqkv[1], "wo": wo[0], "wo_s": wo[1], "wr": _wr(case).cuda().contiguous(),
             "wg": wg[0], "wg_s": wg[1], "wu": wu[0], "wu_s": wu[1], "wd": wd[0], "wd_s": wd[1],
             "attn_norm": None, "ffn_norm": None}
        bm.bm_engine_set_layer(e, layer, w)
    torch.cuda.synchronize()
    assert bm.bm_engine_kernel_family(e) == MMA
    yield e
    bm.bm_engine_destroy(e)


@functools.lru_cache(maxsize=None)
def _oracle_expert(e):
    return {n: oracle.quantize_w4(synth.model_tensor(NAME, CFG, n, 0, e).numpy(), CFG["group"])
            for n in ("wg", "wu", "wd")}


def _oracle_moe(case, h):
    ocfg = oracle.OracleConfig(hidden=CFG["hidden"], experts=CFG["experts"], top_k=CFG["top_k"], ffn=CFG["ffn"],
                               group=CFG["group"], layers=1)
    lw = {"wr": _wr(case).numpy(), "expert": _oracle_expert, "ffn_norm": None}
    tr = {}
    y = oracle.moe_block(ocfg, lw, h.double().numpy(), tr)
    logits = tr["hn"] @ lw["wr"].astype(np.float64).T
    return y, tr["ids"], tr["w"], logits


def _inputs(case, B):
    h = synth.activations(NAME, f"h_{case}", (B, CFG["hidden"]))
    return h.abs() if case == "forced" else h


def _run(bm, e, layer, h):
    B, k = h.shape[0], CFG["top_k"]
    y = torch.empty_like(h)
    ids = torch.empty((B, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((B, k), dtype=torch.float32, device="cuda")
    bm.bm_engine_moe(e, layer, h, y, ids, tw)
    bm.bm_engine_sync(e)
    return y, ids.cpu().numpy(), tw.cpu().numpy()


def _check_ids(ids, ids_r, logits):
    """Routed ids equal the oracle's exactly, except that two experts whose
    oracle logits are within TIE_EPS may trade ranks; returns the rows whose
    ranking had no such near-tie."""
    exact = []
    for b in range(ids.shape[0]):
        assert len(set(ids[b].tolist())) == ids.shape[1] and ids[b].min() >= 0 and ids[b].max() < CFG["experts"]
        s = np.sort(logits[b])[::-1][: ids.shape[1] + 1]
        if np.all(np.abs(np.diff(s)) >= TIE_EPS):
            np.testing.assert_array_equal(ids[b], ids_r[b], err_msg=f"row {b}")
            exact.append(b)
        else:
            # a near-tie: every rank's expert scores within TIE_EPS of the oracle's
            np.testing.assert_allclose(logits[b][ids[b]], logits[b][ids_r[b]], atol=TIE_EPS)
    return exact


@pytest.mark.parametrize("case", ["natural", "forced"])
@pytest.mark.parametrize("B", EX["batches"])
def test_step_moe_kernels_match_oracle(bm, moe_engine, case, B):
    layer = 0 if case == "natural" else 1
    h = _inputs(case, B)
    y, ids, tw = _run(bm, moe_engine, layer, h.cuda())
    y_r, ids_r, w_r, logits = _oracle_moe(case, h)
    exact = _check_ids(ids, ids_r, logits)
    assert len(exact) >= max(1, (9 * B) // 10), f"only {len(exact)} of {B} rows without a near-tie"
    np.testing.assert_allclose(tw[exact], w_r[exact], rtol=1e-4, atol=1e-6)
    assert_close_rows(y[exact], y_r[exact], what=f"step moe kernels {case} B={B}")
    if case == "forced":
        assert all(set(r.tolist()) == set(range(8)) for r in ids)


def test_step_moe_kernels_solo_equals_batched(bm, moe_engine):
    for layer, case in enumerate(("natural", "forced")):
        h = _inputs(case, 32).cuda()
        yb, ib, wb = _run(bm, moe_engine, layer, h)
        for b in (0, 7, 31):
            ys, is_, ws = _run(bm, moe_engine, layer, h[b:b + 1].contiguous())
            assert torch.equal(ys.view(torch.int16), yb[b:b + 1].view(torch.int16)), (case, b)
            assert np.array_equal(is_[0], ib[b]) and np.array_equal(ws[0], wb[b])
        idx = [31, 2, 17, 5, 9]
        yp, ip, _ = _run(bm, moe_engine, layer, h[idx].contiguous())
        assert torch.equal(yp.view(torch.int16), yb[idx].view(torch.int16)), case
        assert np.array_equal(ip, ib[idx])


def test_expert_pipeline_timeout_is_reported_and_engine_recovers(bm, moe_engine):
    # No copy is issued for the first work item of the gate/up kernel: the
    # stage's full barrier never completes, the consumers' bounded wait runs
    # out, the CTA waits for the copies it did issue and stops, and the host
    # reads code 5.  Nothing faults, and the next call computes normally.
    h = _inputs("natural", 8).cuda()
    y0, i0, w0 = _run(bm, moe_engine, 0, h)
    bm.bm_engine_test_drop_expert_item(moe_engine, 0)
    try:
        y = torch.empty_like(h)
        bm.bm_engine_moe(moe_engine, 0, h, y)
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_engine_sync(moe_engine)
        assert ei.value.status == 8 and "code 5" in ei.value.message, ei.value.message
    finally:
        bm.bm_engine_test_drop_expert_item(moe_engine, -1)
    bm.bm_engine_sync(moe_engine)   # the flag was cleared by the report
    y1, i1, w1 = _run(bm, moe_engine, 0, h)
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))
    assert np.array_equal(i1, i0) and np.array_equal(w1, w0)


# ---------------------------------------------------------------- attention

A = synth.CONFIGS["slot_attention"]
S, CAP, QH, KVH, D = A["max_streams"], A["ctx_cap"], A["q_heads"], A["kv_heads"], A["head_dim"]
QKV = (QH + 2 * KVH) * D


def _attn_engine(bm):
    cfg = {"hidden": 512, "q_heads": QH, "kv_heads": KVH, "head_dim": D, "experts": 8, "top_k": 2, "ffn": 256,
           "group": 32, "vocab": 64, "layers": 1, "rope_base": 1e4, "rms_eps": 1e-6, "max_streams": S,
           "ctx_cap": CAP, "renorm_topk": 1, "kernel_policy": MMA, "use_graph": 0}
    e = bm.bm_engine_create(cfg)
    assert bm.bm_engine_kernel_family(e) == MMA
    return e


def _prefix(stream, length):
    shape = (1, KVH, length, D)
    k = synth.normal_bf16(shape, 1.0, synth.seed_of("slot_attention", "k", stream, length), "cuda")
    v = synth.normal_bf16(shape, 1.0, synth.seed_of("slot_attention", "v", stream, length), "cuda")
    return k, v


def _oracle_attend(qkv_row, p, Ko, Vo):
    """Oracle attention of one decode row at position p over its slot's K/V
    (oracle copies, [kvh][p][d], the new position not yet included)."""
    q = qkv_row[: QH * D].reshape(QH, D)
    k = qkv_row[QH * D: (QH + KVH) * D].reshape(KVH, D)
    v = qkv_row[(QH + KVH) * D:].reshape(KVH, D)
    q_rot = oracle.bf16_round(oracle.rope_rotate_half(q, p, 1e4))
    k_rot = oracle.bf16_round(oracle.rope_rotate_half(k, p, 1e4))
    Kf = np.concatenate([Ko, k_rot[:, None]], axis=1)
    Vf = np.concatenate([Vo, v[:, None]], axis=1)
    return oracle.bf16_round(oracle.slot_attention(q_rot, Kf, Vf)), k_rot, v


def _live_counts(events):
    live, out = 0, []
    for ev in events:
        live += len(ev["join"])
        out.append(live)
        live -= len(ev["finish"])
    return out


def test_step_attention_kernel_schedule(bm):
    # arrivals outpace departures, so the batch spans 1..16 streams (mean ~12)
    events = synth.schedule(seed=2025, steps=A["steps"], max_streams=S, ctx_cap=CAP, max_batch=S, join_p=0.6,
                            finish_p=0.05)
    assert max(_live_counts(events)) == S and min(_live_counts(events)) == 1
    e = _attn_engine(bm)
    try:
        # per slot: the bytes it must hold (seeded prefix, then the kernel's own
        # appended k and the given v) and the oracle's copy of K (its own
        # rotated keys); V is the same on both sides
        exp_K = torch.empty((S, KVH, CAP, D), dtype=torch.bfloat16, device="cuda")
        exp_V = torch.empty_like(exp_K)
        ora_K = torch.empty_like(exp_K)
        length = {}
        live = []       # slots, oldest first
        sid = 0
        checked = 0
        for step, ev in enumerate(events):
            for L in ev["join"]:
                k, v = _prefix(5000 + sid, L)
                slot = bm.kv_slot_seed(e, k, v, L)
                live.append(slot)
                exp_K[slot, :, :L] = k[0]
                exp_V[slot, :, :L] = v[0]
                ora_K[slot, :, :L] = k[0]
                length[slot] = L
                sid += 1
            B = len(live)
            assert 1 <= B <= S
            qkv = synth.normal_bf16((B, QKV), 1.0, synth.seed_of("slot_attention", "qkv", step, B), "cuda")
            out = torch.empty((B, QH, D), dtype=torch.float16, device="cuda")
            bm.bm_engine_attention(e, 0, live, qkv, out)
            bm.kv_slot_advance(e, live)
            bm.bm_engine_sync(e)
            rows = qkv.double().cpu().numpy()
            for i, s in enumerate(live):
                p = length[s]
                n = p + 1
                Kr = torch.empty((KVH, n, D), dtype=torch.bfloat16, device="cuda")
                Vr = torch.empty_like(Kr)
                bm.kv_slot_read(e, 0, s, n, Kr, Vr)
                torch.cuda.synchronize()
                # every earlier position of the slot is as it was: no write of this
                # or any earlier step touched it; v lands byte for byte
                assert torch.equal(Kr[:, :p], exp_K[s, :, :p]) and torch.equal(Vr[:, :p], exp_V[s, :, :p]), \
                    f"step {step}: slot {s} disturbed"
                v_new = qkv[i, (QH + KVH) * D:].view(KVH, D)
                assert torch.equal(Vr[:, p], v_new), f"step {step}: slot {s} appended v"
                k_row = rows[i][QH * D: (QH + KVH) * D].reshape(KVH, D)
                k_rot = oracle.bf16_round(oracle.rope_rotate_half(k_row, p, 1e4))
                if step % 25 == 0 or i == step % B:
                    Ko = ora_K[s, :, :p].double().cpu().numpy()
                    Vo = exp_V[s, :, :p].double().cpu().numpy()
                    ref, _, _ = _oracle_attend(rows[i], p, Ko, Vo)
                    assert_close_rows(out[i:i + 1].float(), ref[None], what=f"step attention kernel, len {n}")
                    assert_close_rows(Kr[:, p][None].float(), k_rot[None], what="step attention appended k (rotated)")
                    checked += 1
                exp_K[s, :, p] = Kr[:, p]
                exp_V[s, :, p] = v_new
                ora_K[s, :, p] = torch.from_numpy(k_rot).to(torch.bfloat16).cuda()
                length[s] = n
            fin = set(ev["finish"])
            for j, s in enumerate(live):
                if j in fin:
                    bm.kv_slot_release(e, s)
            live = [s for j, s in enumerate(live) if j not in fin]
        assert checked >= A["steps"]
    finally:
        bm.bm_engine_destroy(e)


def test_step_attention_merge_levels(bm):
    # chunk counts on both sides of the two-level merge (blocks of 8 chunks of
    # 128 positions): 1, 8 (one level), 9 (a block and one chunk), 16, 17 and
    # 64 (eight blocks, the cap) in one launch, each row against the oracle;
    # a two-level stream alone gives its batched bytes
    e = _attn_engine(bm)
    try:
        lens = [5, 1023, 1024, 2047, 2048, CAP - 1]
        slots, pre = [], {}
        for i, L in enumerate(lens):
            k, v = _prefix(7000 + i, L)
            slots.append(bm.kv_slot_seed(e, k, v, L))
            pre[slots[-1]] = (k[0].double().cpu().numpy(), v[0].double().cpu().numpy())
        B = len(slots)
        qkv = synth.normal_bf16((B, QKV), 1.0, synth.seed_of("slot_attention", "qkv_levels", B), "cuda")
        out = torch.empty((B, QH, D), dtype=torch.float16, device="cuda")
        bm.bm_engine_attention(e, 0, slots, qkv, out)
        bm.bm_engine_sync(e)
        rows = qkv.double().cpu().numpy()
        for i, s in enumerate(slots):
            Ko, Vo = pre[s]
            ref, _, _ = _oracle_attend(rows[i], lens[i], Ko, Vo)
            assert_close_rows(out[i:i + 1].float(), ref[None], what=f"attention merge levels, len {lens[i] + 1}")
        # the same rows again, the 17-chunk stream alone: identical bytes (its
        # position's k and v are rewritten with the same values)
        one = torch.empty((1, QH, D), dtype=torch.float16, device="cuda")
        bm.bm_engine_attention(e, 0, [slots[4]], qkv[4:5].contiguous(), one)
        bm.bm_engine_sync(e)
        assert torch.equal(one.view(torch.int16), out[4:5].view(torch.int16))
    finally:
        bm.bm_engine_destroy(e)
