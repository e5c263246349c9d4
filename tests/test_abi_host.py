"""The C-ABI library without a GPU: exported symbols, argument checks, and the
host slot map under ragged join/finish schedules."""

import ctypes
import os
import re
import subprocess

import pytest

import bit_moe_decode_w4a16_gb300 as bm
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitmoe.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    bm.build()
    return bm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted({n for n in names if n not in ("if", "return", "sizeof")})


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "decode_step" in names and "w4_gemm_batched" in names and len(names) >= 25
    out = subprocess.run(["nm", "-D", "--defined-only", bm.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(bm.lib(), n)


def test_no_vendor_blas_linked():
    # The device path makes no BLAS calls: nothing of cuBLAS is linked.
    out = subprocess.run(["ldd", bm.LIB_PATH], capture_output=True, text=True).stdout
    assert "cublas" not in out.lower()
    syms = subprocess.run(["nm", "-D", bm.LIB_PATH], capture_output=True, text=True).stdout
    assert "cublas" not in syms.lower()


def test_argument_checks_without_gpu():
    cfg = {"hidden": 512, "q_heads": 8, "kv_heads": 3, "head_dim": 64, "experts": 8, "top_k": 2, "ffn": 256,
           "group": 32, "vocab": 100, "layers": 1, "rope_base": 1e4, "rms_eps": 1e-6, "max_streams": 2,
           "ctx_cap": 64, "renorm_topk": 1, "kernel_policy": 0, "use_graph": 1}
    with pytest.raises(bm.BitMoeError) as ei:
        bm.bm_engine_create(cfg)
    assert ei.value.status == 1 and "kv_heads" in ei.value.message
    cfg.update(kv_heads=2, group=48)
    with pytest.raises(bm.BitMoeError) as ei:
        bm.bm_engine_create(cfg)
    assert ei.value.status == 1
    cfg.update(group=32, top_k=9)
    with pytest.raises(bm.BitMoeError):
        bm.bm_engine_create(cfg)
    cfg.update(top_k=2, max_streams=129)
    with pytest.raises(bm.BitMoeError) as ei:
        bm.bm_engine_create(cfg)
    assert ei.value.status == 1 and "max_streams" in ei.value.message
    cfg.update(max_streams=100, kernel_policy=1)      # above 64 only on the warp-MMA family
    with pytest.raises(bm.BitMoeError) as ei:
        bm.bm_engine_create(cfg)
    assert ei.value.status == 1 and "warp-MMA" in ei.value.message
    cfg.update(max_streams=2, kernel_policy=0)
    # the dense op rejects bad shapes before touching the device
    for (M, N, K, g) in [(0, 8, 64, 32), (1, 8, 48, 32), (1, 8, 64, 48), (1, 0, 64, 32)]:
        with pytest.raises(bm.BitMoeError) as ei:
            bm.w4_gemm_batched(1, 1, 1, 1, None, M, N, K, g)
        assert ei.value.status == 1
    with pytest.raises(bm.BitMoeError):
        bm.w4_gemm_batched(None, 1, 1, 1, None, 1, 8, 64, 32)
    with pytest.raises(bm.BitMoeError):
        bm.bm_w4_quantize(1, 4, 60, 32, 1, 1)
    w = {"experts": 8, "top_k": 2, "hidden": 512, "ffn": 256, "group": 32, "renorm_topk": 1,
         "wr": 1, "wg": 1, "wg_s": 1, "wu": 1, "wu_s": 1, "wd": 1, "wd_s": 1}
    need = bm.bm_moe_workspace_bytes(4, 8, 2, 512, 256)
    assert need > 0
    with pytest.raises(bm.BitMoeError) as ei:
        bm.moe_grouped_w4(w, 1, None, 1, None, None, 4, 1, need - 1)
    assert "workspace" in ei.value.message
    assert bm.last_error() != ""
    # prompt ingestion checks its arguments before any device work
    toks = (ctypes.c_int32 * 2)(1, 2)
    nxt = (ctypes.c_int32 * 1)()
    st = bm.lib().kv_slot_prefill(None, 0, 2, ctypes.addressof(toks), ctypes.addressof(nxt), None, None)
    assert st == 1 and "kv_slot_prefill" in bm.last_error()


def test_slot_map_lifecycle_and_errors():
    m = bm.bm_slot_map_create(3, 16)
    try:
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_acquire(m, 16)
        assert ei.value.status == 2                     # context cap: rejected, not truncated
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_acquire(m, -1)
        assert ei.value.status == 1
        assert [bm.bm_slot_map_acquire(m, n) for n in (15, 0, 7)] == [0, 1, 2]
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_acquire(m, 1)
        assert ei.value.status == 3                     # no free slot
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_check_batch(m, [1, 1])
        assert ei.value.status == 1                     # duplicate
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_check_batch(m, [5])
        assert ei.value.status == 1                     # out of range
        bm.bm_slot_map_advance(m, [0, 2])
        assert bm.bm_slot_map_length(m, 0) == 16 and bm.bm_slot_map_length(m, 2) == 8
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_check_batch(m, [0])
        assert ei.value.status == 2                     # slot 0 is full
        bm.bm_slot_map_release(m, 0)
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_release(m, 0)
        assert ei.value.status == 4                     # double release
        with pytest.raises(bm.BitMoeError) as ei:
            bm.bm_slot_map_check_batch(m, [0, 1])
        assert ei.value.status == 4                     # released slot in a batch
        assert bm.bm_slot_map_active_count(m) == 2
        assert bm.bm_slot_map_acquire(m, 3) == 0        # lowest free slot is reused
        assert bm.bm_slot_map_length(m, 0) == 3
    finally:
        bm.bm_slot_map_destroy(m)


class PyWipeMap:
    """The pre-fix pool behaviour ([Crash root cause] §3): a batch-size change
    resets every continuing stream to its prompt length."""

    def __init__(self, S, cap):
        self.len, self.active, self.prompt, self.last_b = [0] * S, [False] * S, [0] * S, None

    def acquire(self, n):
        s = self.active.index(False)
        self.active[s], self.len[s], self.prompt[s] = True, n, n
        return s

    def release(self, s):
        self.active[s], self.len[s] = False, 0

    def step(self, slots):
        if self.last_b is not None and len(slots) != self.last_b:
            for s in slots:
                self.len[s] = self.prompt[s]
        self.last_b = len(slots)
        for s in slots:
            self.len[s] += 1

    def length(self, s):
        return self.len[s]


class AbiMap:
    def __init__(self, S, cap):
        self.m = bm.bm_slot_map_create(S, cap)

    def acquire(self, n):
        return bm.bm_slot_map_acquire(self.m, n)

    def release(self, s):
        bm.bm_slot_map_release(self.m, s)

    def step(self, slots):
        bm.bm_slot_map_check_batch(self.m, slots)
        bm.bm_slot_map_advance(self.m, slots)

    def length(self, s):
        return bm.bm_slot_map_length(self.m, s)


def drive(map_obj, events):
    """Run a join/finish schedule; every stream's length must equal its prompt
    plus the steps it took, whatever the other streams did."""
    live, expect = [], {}
    for ev in events:
        for n in ev["join"]:
            s = map_obj.acquire(n)
            live.append(s)
            expect[s] = n
        map_obj.step(list(live))
        for s in live:
            expect[s] += 1
            assert map_obj.length(s) == expect[s], (s, map_obj.length(s), expect[s])
        fin = set(ev["finish"])
        for j, s in enumerate(live):
            if j in fin:
                map_obj.release(s)
        live = [s for j, s in enumerate(live) if j not in fin]


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_slot_map_ragged_schedule(seed):
    events = synth.schedule(seed=seed, steps=200, max_streams=16, ctx_cap=8192, max_batch=16)
    sizes = set()
    live = 0
    for ev in events:
        live += len(ev["join"])
        sizes.add(live)
        live -= len(ev["finish"])
    assert len(sizes) > 5          # batch composition really changes
    drive(AbiMap(16, 8192), events)


def test_slot_map_check_catches_wipe_mutant():
    events = synth.schedule(seed=1, steps=200, max_streams=16, ctx_cap=8192, max_batch=16)
    with pytest.raises(AssertionError):
        drive(PyWipeMap(16, 8192), events)
