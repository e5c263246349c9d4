"""GPU parity of slot attention over the fixed arena (16 slots x 8192
positions, 32 q / 4 kv heads, head_dim 128, bf16 N(0,1) K/V, ragged lengths
in [1, 8192]) and slot isolation under a seeded 200-step join/finish
schedule with B between 1 and 16."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_rows

pytestmark = pytest.mark.gpu

A = synth.CONFIGS["slot_attention"]
S, CAP, QH, KVH, D = A["max_streams"], A["ctx_cap"], A["q_heads"], A["kv_heads"], A["head_dim"]


@pytest.fixture(scope="module")
def bm():
    import bit_moe_decode_w4a16_gb300 as m
    m.build()
    return m


def _engine(bm, cap=CAP, streams=S):
    cfg = {"hidden": 512, "q_heads": QH, "kv_heads": KVH, "head_dim": D, "experts": 8, "top_k": 2, "ffn": 256,
           "group": 32, "vocab": 16, "layers": 1, "rope_base": 1e4, "rms_eps": 1e-6, "max_streams": streams,
           "ctx_cap": cap, "renorm_topk": 1, "kernel_policy": 1, "use_graph": 0}
    return bm.bm_engine_create(cfg)


def _prefix(stream, length):
    shape = (1, KVH, length, D)
    k = synth.normal_bf16(shape, 1.0, synth.seed_of("slot_attention", "k", stream, length), "cuda")
    v = synth.normal_bf16(shape, 1.0, synth.seed_of("slot_attention", "v", stream, length), "cuda")
    return k, v


def _new(step, B):
    q = synth.normal_bf16((B, QH, D), 1.0, synth.seed_of("slot_attention", "q", step, B), "cuda")
    k = synth.normal_bf16((B, KVH, D), 1.0, synth.seed_of("slot_attention", "kn", step, B), "cuda")
    v = synth.normal_bf16((B, KVH, D), 1.0, synth.seed_of("slot_attention", "vn", step, B), "cuda")
    return q, k, v


def _oracle_attend(q, Kfull, Vfull):
    return oracle.bf16_round(oracle.slot_attention(q, Kfull, Vfull))


def test_attention_ragged_full_arena(bm):
    e = _engine(bm)
    try:
        lens = synth.prompt_lengths(S, 1, CAP - 1, synth.seed_of("slot_attention", "lens"))
        lens[0], lens[1], lens[2] = 1, CAP - 1, 127        # edge lengths: 1 position, full cap, chunk edge
        kv = {}
        slots = []
        for i, L in enumerate(lens):
            k, v = _prefix(i, L)
            slots.append(bm.kv_slot_seed(e, k, v, L))
            kv[slots[-1]] = (k, v)
        torch.cuda.synchronize()
        q, kn, vn = _new(0, S)
        bm.kv_slot_append(e, 0, slots, kn, vn)
        O = torch.empty((S, QH, D), dtype=torch.bfloat16, device="cuda")
        bm.kv_slot_attend(e, 0, slots, q, O)
        bm.bm_engine_sync(e)
        for i, s in enumerate(slots):
            k, v = kv[s]
            Kf = torch.cat([k[0], kn[i][:, None]], dim=1).double().cpu().numpy()
            Vf = torch.cat([v[0], vn[i][:, None]], dim=1).double().cpu().numpy()
            ref = _oracle_attend(q[i].double().cpu().numpy(), Kf, Vf)
            assert_close_rows(O[i:i + 1], ref[None], what=f"attention slot {s} len {lens[i] + 1}")
        # solo == batched bytes: attend one stream alone
        O1 = torch.empty((1, QH, D), dtype=torch.bfloat16, device="cuda")
        bm.kv_slot_attend(e, 0, [slots[5]], q[5:6].contiguous(), O1)
        bm.bm_engine_sync(e)
        assert torch.equal(O1.view(torch.int16), O[5:6].view(torch.int16))
        # the appended position is committed by advance, then reads back
        bm.kv_slot_advance(e, slots)
        assert bm.kv_slot_length(e, slots[0]) == 2
        Kr = torch.empty((KVH, 2, D), dtype=torch.bfloat16, device="cuda")
        Vr = torch.empty_like(Kr)
        bm.kv_slot_read(e, 0, slots[0], 2, Kr, Vr)
        bm.bm_engine_sync(e)
        assert torch.equal(Kr[:, 1], kn[0]) and torch.equal(Vr[:, 0], kv[slots[0]][1][0, :, 0])
        # a full slot is rejected, not truncated
        with pytest.raises(bm.BitMoeError) as ei:
            bm.kv_slot_append(e, 0, [slots[1]], kn[:1].contiguous(), vn[:1].contiguous())
        assert ei.value.status == 2
        with pytest.raises(bm.BitMoeError) as ei:
            bm.kv_slot_seed(e, kn, vn, CAP)
        assert ei.value.status in (2, 3)
    finally:
        bm.bm_engine_destroy(e)


def test_join_finish_schedule_isolation(bm):
    events = synth.schedule(seed=2024, steps=A["steps"], max_streams=S, ctx_cap=CAP, max_batch=S)
    e = _engine(bm)
    try:
        live = []                  # (stream id, slot)
        expect = {}                # slot -> (K [kvh][n][d], V) expected device contents
        sid = 0
        checked = 0
        for step, ev in enumerate(events):
            before = {s: (expect[s][0].clone(), expect[s][1].clone()) for _, s in live}
            for L in ev["join"]:
                k, v = _prefix(1000 + sid, L)
                slot = bm.kv_slot_seed(e, k, v, L)
                live.append((sid, slot))
                expect[slot] = (k[0].clone(), v[0].clone())
                sid += 1
            slots = [s for _, s in live]
            B = len(slots)
            assert 1 <= B <= S
            q, kn, vn = _new(step, B)
            bm.kv_slot_append(e, 0, slots, kn, vn)
            O = torch.empty((B, QH, D), dtype=torch.bfloat16, device="cuda")
            bm.kv_slot_attend(e, 0, slots, q, O)
            bm.kv_slot_advance(e, slots)
            for i, s in enumerate(slots):
                expect[s] = (torch.cat([expect[s][0], kn[i][:, None]], 1), torch.cat([expect[s][1], vn[i][:, None]], 1))
            bm.bm_engine_sync(e)
            # continuing streams' K/V untouched by this step's joins and appends of others
            for s, (Kb, Vb) in before.items():
                n = Kb.shape[1]
                Kr = torch.empty((KVH, n, D), dtype=torch.bfloat16, device="cuda")
                Vr = torch.empty_like(Kr)
                bm.kv_slot_read(e, 0, s, n, Kr, Vr)
                torch.cuda.synchronize()
                assert torch.equal(Kr, Kb) and torch.equal(Vr, Vb), f"step {step}: slot {s} disturbed"
            if step % 20 == 0 or ev["join"]:
                i = step % B
                s = slots[i]
                ref = _oracle_attend(q[i].double().cpu().numpy(), expect[s][0].double().cpu().numpy(),
                                     expect[s][1].double().cpu().numpy())
                assert_close_rows(O[i:i + 1], ref[None], what=f"schedule step {step} slot {s}")
                checked += 1
            fin = set(ev["finish"])
            for j, (_, s) in enumerate(live):
                if j in fin:
                    bm.kv_slot_release(e, s)
                    del expect[s]
            live = [x for j, x in enumerate(live) if j not in fin]
        assert checked >= 10
    finally:
        bm.bm_engine_destroy(e)
