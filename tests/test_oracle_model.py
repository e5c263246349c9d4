"""Pins of the oracle's decode step: row independence, the slot lifecycle,
slot isolation under ragged join/finish, and the wipe-on-batch-change bug."""

import copy

import numpy as np
import pytest

import oracle
import synth
from oracle_side import oracle_config, oracle_weights

NAME = "tiny_layer"
CFG = synth.CONFIGS[NAME]
LAYERS = 2   # the tiny layer stacked twice, with a bf16 head of vocab 4096


@pytest.fixture(scope="module")
def model():
    cfg = oracle_config(CFG, layers=LAYERS, max_streams=6, ctx_cap=128)
    return cfg, oracle_weights(NAME, CFG, LAYERS)


def _kv(cfg):
    return oracle.OracleKV(cfg, oracle.OracleSlotMap(cfg.max_streams, cfg.ctx_cap))


def _prefix(stream, length):
    k, v = synth.kv_prefix(NAME, CFG, stream, length, layers=LAYERS)
    return k.double().numpy(), v.double().numpy()


def test_row_independence(model):
    cfg, w = model
    lens = [5, 17, 40]
    toks = [11, 4000, 257]
    kv = _kv(cfg)
    slots = [kv.seed(*_prefix(i, L)) for i, L in enumerate(lens)]
    logits_b, ids_b = oracle.model_step(cfg, w, kv, slots, toks)
    for i, L in enumerate(lens):
        solo = _kv(cfg)
        s = solo.seed(*_prefix(i, L))
        logits_s, ids_s = oracle.model_step(cfg, w, solo, [s], [toks[i]])
        np.testing.assert_array_equal(logits_s[0], logits_b[i])
        assert ids_s[0] == ids_b[i]
    # order of rows in the batch does not matter either
    kv2 = _kv(cfg)
    slots2 = [kv2.seed(*_prefix(i, L)) for i, L in enumerate(lens)]
    perm = [2, 0, 1]
    logits_p, _ = oracle.model_step(cfg, w, kv2, [slots2[p] for p in perm], [toks[p] for p in perm])
    for j, p in enumerate(perm):
        np.testing.assert_array_equal(logits_p[j], logits_b[p])


def test_seeded_prefix_equals_decoded_prefix(model):
    # Decoding tokens t0..t5 from an empty slot, or seeding a slot with the
    # K/V that t0..t4 left behind and decoding t5, gives the same step-5 output.
    cfg, w = model
    toks = [3, 99, 1024, 7, 3000, 42]
    kv = _kv(cfg)
    s = kv.seed(np.zeros((LAYERS, cfg.kv_heads, 0, cfg.head_dim)),
                np.zeros((LAYERS, cfg.kv_heads, 0, cfg.head_dim)))
    for t in toks[:-1]:
        oracle.model_step(cfg, w, kv, [s], [t])
    K = np.stack([kv.K[s][l][:, :5] for l in range(LAYERS)])
    V = np.stack([kv.V[s][l][:, :5] for l in range(LAYERS)])
    last_a, _ = oracle.model_step(cfg, w, kv, [s], [toks[-1]])
    kv2 = _kv(cfg)
    s2 = kv2.seed(K, V)
    last_b, _ = oracle.model_step(cfg, w, kv2, [s2], [toks[-1]])
    np.testing.assert_array_equal(last_a, last_b)


def test_prefill_equals_token_by_token_decode(model):
    # Ingesting a prompt in one block (causal block attention over the slot)
    # leaves the same K/V, length and last-position logits as feeding the
    # prompt one decode step at a time: the definition a prompt has.
    cfg, w = model
    toks = [3, 99, 1024, 7, 3000, 42, 5, 4095, 17]
    L0 = 17
    kv_a = _kv(cfg)
    sa = kv_a.seed(*_prefix(0, L0))
    logits_a, nxt_a = oracle.model_prefill(cfg, w, kv_a, sa, toks)
    kv_b = _kv(cfg)
    sb = kv_b.seed(*_prefix(0, L0))
    for t in toks:
        logits_b, ids_b = oracle.model_step(cfg, w, kv_b, [sb], [t])
    np.testing.assert_allclose(logits_a, logits_b[0], rtol=0, atol=1e-9)
    assert nxt_a == int(ids_b[0])
    assert kv_a.map.length[sa] == kv_b.map.length[sb] == L0 + len(toks)
    for l in range(LAYERS):
        np.testing.assert_allclose(kv_a.K[sa][l], kv_b.K[sb][l], rtol=0, atol=1e-12)
        np.testing.assert_allclose(kv_a.V[sa][l], kv_b.V[sb][l], rtol=0, atol=1e-12)
    # the prefix seeded at join is untouched
    K0, V0 = _prefix(0, L0)
    np.testing.assert_array_equal(kv_a.K[sa][1][:, :L0], K0[1])


def test_prefill_from_empty_slot_and_rejections(model):
    cfg, w = model
    kv = _kv(cfg)
    empty = np.zeros((LAYERS, cfg.kv_heads, 0, cfg.head_dim))
    s = kv.seed(empty, empty)
    logits, nxt = oracle.model_prefill(cfg, w, kv, s, [11])
    kv2 = _kv(cfg)
    s2 = kv2.seed(empty, empty)
    ref, ids = oracle.model_step(cfg, w, kv2, [s2], [11])
    np.testing.assert_allclose(logits, ref[0], rtol=0, atol=1e-9)
    with pytest.raises(ValueError):
        oracle.model_prefill(cfg, w, kv, s, [])
    with pytest.raises(ValueError):
        oracle.model_prefill(cfg, w, kv, s, [1] * cfg.ctx_cap)     # 1 + cap > cap
    kv.release(s)
    with pytest.raises(ValueError):
        oracle.model_prefill(cfg, w, kv, s, [1])


def test_slot_map_lifecycle_errors():
    m = oracle.OracleSlotMap(2, 16)
    with pytest.raises(ValueError):
        m.seed(16)                      # no room for a decode token
    a = m.seed(15)
    b = m.seed(0)
    assert (a, b) == (0, 1)
    with pytest.raises(ValueError):
        m.seed(1)                       # all slots taken
    with pytest.raises(ValueError):
        m.check_batch([0, 0])           # duplicate slot
    m.advance([0])
    with pytest.raises(ValueError):
        m.check_batch([0])              # slot 0 reached the cap
    m.release(0)
    with pytest.raises(ValueError):
        m.release(0)                    # double release
    with pytest.raises(ValueError):
        m.check_batch([0])              # free slot in a batch
    assert m.seed(3) == 0               # lowest free slot is reused


class WipeOnBatchChange(oracle.OracleKV):
    """The failure the slot design rules out ([Crash root cause, §3 Results]):
    pools keyed by batch size are wiped when the batch size changes, and the
    re-seed only has the prompt prefix, not the decode-appended K/V."""

    def __init__(self, cfg, slot_map):
        super().__init__(cfg, slot_map)
        self.last_b = None
        self.prompt = {}

    def seed(self, K, V):
        s = super().seed(K, V)
        self.prompt[s] = (np.asarray(K, np.float64), np.asarray(V, np.float64))
        return s

    def on_batch(self, slots):
        if self.last_b is not None and len(slots) != self.last_b:
            for s in slots:   # re-seed from what the host still has
                K, V = self.prompt[s]
                L = K.shape[2]
                self.K[s] = [K[l].copy() for l in range(self.cfg.layers)]
                self.V[s] = [V[l].copy() for l in range(self.cfg.layers)]
                self.map.length[s] = L
        self.last_b = len(slots)


def run_schedule(cfg, w, events, kv_cls, check_isolation=True):
    """Greedy-decode a join/finish schedule; return each stream's tokens.

    Before and after every step, the K/V of every continuing stream at its
    committed positions must be unchanged by other streams' joins and
    finishes (checked when ``check_isolation``).
    """
    kv = kv_cls(cfg, oracle.OracleSlotMap(cfg.max_streams, cfg.ctx_cap))
    live = []          # (stream id, slot)
    next_tok = {}
    out = {}
    sid = 0
    for ev in events:
        snap = {s: [kv.K[s][l][:, :kv.map.length[s]].copy() for l in range(cfg.layers)]
                for _, s in live}
        for length in ev["join"]:
            K, V = _prefix(100 + sid, length)
            slot = kv.seed(K, V)
            live.append((sid, slot))
            next_tok[sid] = (sid * 977 + 13) % cfg.vocab
            out[sid] = []
            sid += 1
        if hasattr(kv, "on_batch"):
            kv.on_batch([s for _, s in live])
        if check_isolation:
            for s, Ks in snap.items():
                for l in range(cfg.layers):
                    np.testing.assert_array_equal(kv.K[s][l][:, :Ks[l].shape[1]], Ks[l])
        slots = [s for _, s in live]
        _, ids = oracle.model_step(cfg, w, kv, slots, [next_tok[i] for i, _ in live])
        for (i, _), t in zip(live, ids):
            out[i].append(int(t))
            next_tok[i] = int(t)
        fin = set(ev["finish"])
        for j, (i, s) in enumerate(live):
            if j in fin:
                kv.release(s)
        live = [x for j, x in enumerate(live) if j not in fin]
    return out


def solo_tokens(cfg, w, events):
    """Each stream of the schedule decoded alone, for its own number of steps."""
    lens, steps, sid, live = {}, {}, 0, []
    for ev in events:
        for length in ev["join"]:
            lens[sid] = length
            steps[sid] = 0
            live.append(sid)
            sid += 1
        for i in live:
            steps[i] += 1
        fin = set(ev["finish"])
        live = [i for j, i in enumerate(live) if j not in fin]
    out = {}
    for i in lens:
        kv = _kv(cfg)
        s = kv.seed(*_prefix(100 + i, lens[i]))
        tok = (i * 977 + 13) % cfg.vocab
        out[i] = []
        for _ in range(steps[i]):
            _, ids = oracle.model_step(cfg, w, kv, [s], [tok])
            tok = int(ids[0])
            out[i].append(tok)
    return out


def test_ragged_join_finish_isolation_and_solo_parity(model):
    cfg, w = model
    events = synth.schedule(seed=7, steps=14, max_streams=cfg.max_streams,
                            ctx_cap=48, min_len=1, max_batch=4)
    assert len({sum(len(e["join"]) for e in events[:i + 1]) for i in range(len(events))}) > 2
    batched = run_schedule(cfg, w, events, oracle.OracleKV)
    solo = solo_tokens(cfg, w, events)
    assert batched == solo


def test_wipe_on_batch_change_is_caught(model):
    # Negative control: the pre-fix pool design breaks solo parity (and the
    # continuing streams' K/V) on the same schedule.
    cfg, w = model
    events = synth.schedule(seed=7, steps=14, max_streams=cfg.max_streams,
                            ctx_cap=48, min_len=1, max_batch=4)
    with pytest.raises(AssertionError):
        run_schedule(cfg, w, events, WipeOnBatchChange)
    mutant = run_schedule(cfg, w, events, WipeOnBatchChange, check_isolation=False)
    assert mutant != solo_tokens(cfg, w, events)
