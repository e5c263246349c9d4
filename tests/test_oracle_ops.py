"""Pins of the oracle's ops: GEMM, RMSNorm, RoPE, attention, routing, experts."""

import math

import numpy as np
import pytest

import oracle
from golden_io import lines, table


# ---------------------------------------------------------------- W4A16 GEMM

def _brute_gemm(X, packed, scales, K, g):
    """Pure-Python loops: nibble extraction written out here, not borrowed."""
    M, N = len(X), len(packed)
    Y = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                byte = int(packed[n][k // 2])
                nib = (byte >> 4) if (k % 2) else (byte & 15)
                acc += float(X[m][k]) * (nib - 8) * float(scales[n][k // g])
            Y[m][n] = acc
    return Y


def test_gemm_hand_value():
    t = table("small_values.txt")
    packed = np.array([[int(b, 16) for b in t["gemm_bytes"]]], np.uint8)
    scales = np.array([[float(t["gemm_scale"][0])]], np.float16)
    x = np.array([[float(v) for v in t["gemm_x"]]])
    assert oracle.w4_gemm(x, packed, scales, K=4, g=4)[0, 0] == float(t["gemm_y"][0])


def test_gemm_brute_force_tiny():
    rng = np.random.default_rng(11)
    for (M, N, K, g) in [(1, 3, 64, 32), (3, 5, 64, 64), (2, 4, 128, 32)]:
        packed = rng.integers(0, 256, size=(N, K // 2)).astype(np.uint8)
        scales = rng.uniform(0.001, 0.05, size=(N, K // g)).astype(np.float16)
        X = oracle.bf16_round(rng.standard_normal((M, K)))
        got = oracle.w4_gemm(X, packed, scales, K, g)
        ref = np.array(_brute_gemm(X, packed, scales, K, g))
        bound = K * 2.0 ** -52 * np.abs(X) @ np.abs(oracle.dequant_w4(packed, scales, K, g)).T
        assert np.all(np.abs(got - ref) <= bound + 1e-300)


def test_gemm_closed_forms_and_row_independence():
    rng = np.random.default_rng(12)
    K, g = 256, 64
    # all codes +1 and unit scales: y = sum(x)
    packed = np.full((2, K // 2), 0x99, np.uint8)
    scales = np.ones((2, K // g), np.float16)
    X = oracle.bf16_round(rng.standard_normal((4, K)))
    Y = oracle.w4_gemm(X, packed, scales, K, g)
    np.testing.assert_allclose(Y[:, 0], X.sum(axis=1), rtol=1e-13)
    # rows are independent: row m of a batch equals the GEMV of row m alone
    packed = rng.integers(0, 256, size=(5, K // 2)).astype(np.uint8)
    scales = rng.uniform(0.001, 0.05, size=(5, K // g)).astype(np.float16)
    Yb = oracle.w4_gemm(X, packed, scales, K, g)
    for m in range(4):
        np.testing.assert_array_equal(Yb[m], oracle.w4_gemm(X[m:m + 1], packed, scales, K, g)[0])
    # transposition check: a weight row that is zero except one input feature
    packed = np.full((3, K // 2), 0x88, np.uint8)
    packed[1, 5] = 0x98   # byte 5: k = 10 -> code 0 (low nibble 8), k = 11 -> code +1 (high nibble 9)
    scales = np.ones((3, K // g), np.float16)
    Y = oracle.w4_gemm(X, packed, scales, K, g)
    np.testing.assert_array_equal(Y[:, 1], X[:, 11])
    assert np.all(Y[:, 0] == 0) and np.all(Y[:, 2] == 0)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_hand_and_invariants():
    t = lines("small_values.txt")
    row = [r for r in t if r[0] == "rmsnorm"][0]
    got = oracle.rmsnorm(np.array([[3.0, 4.0]]), eps=0.0)[0]
    np.testing.assert_allclose(got, [float(row[4]), float(row[5])], rtol=1e-15)
    rng = np.random.default_rng(13)
    x = rng.standard_normal((5, 512)) * 3
    y = oracle.rmsnorm(x, eps=1e-6)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-6)
    np.testing.assert_allclose(oracle.rmsnorm(7.5 * x, eps=0.0), oracle.rmsnorm(x, eps=0.0), rtol=1e-13)
    w = rng.standard_normal(512)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, 1e-6), y * w, rtol=1e-14)


# ---------------------------------------------------------------- RoPE

def test_rope_hand_value():
    t = table("rope.txt")
    x = np.array([[float(v) for v in t["x"]]])
    got = oracle.rope_rotate_half(x, int(t["pos"][0]), float(t["base"][0]))[0]
    np.testing.assert_allclose(got, [float(v) for v in t["expect"]], rtol=1e-14)


def test_rope_invariants():
    rng = np.random.default_rng(14)
    d = 64
    x = rng.standard_normal((3, d))
    np.testing.assert_array_equal(oracle.rope_rotate_half(x, 0, 1e4), x)
    y = oracle.rope_rotate_half(x, 37, 1e4)
    half = d // 2
    np.testing.assert_allclose(x[:, :half] ** 2 + x[:, half:] ** 2,
                               y[:, :half] ** 2 + y[:, half:] ** 2, rtol=1e-12)
    # relative position: q(m)·k(n) depends on m - n only
    q, k = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    dots = [float(oracle.rope_rotate_half(q, m, 1e4)[0] @ oracle.rope_rotate_half(k, n, 1e4)[0])
            for (m, n) in [(5, 2), (103, 100), (4003, 4000)]]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)
    # composition: rotating by m then by n equals rotating by m + n
    np.testing.assert_allclose(oracle.rope_rotate_half(oracle.rope_rotate_half(x, 11, 1e4), 30, 1e4),
                               oracle.rope_rotate_half(x, 41, 1e4), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- attention

def test_attention_hand_value():
    t = table("attention.txt")
    f = lambda k: [float(v) for v in t[k]]
    q = np.array([f("q")])
    K = np.array([[f("k0"), f("k1")]])
    V = np.array([[f("v0"), f("v1")]])
    np.testing.assert_allclose(oracle.slot_attention(q, K, V)[0], f("expect"), rtol=1e-14)


def test_attention_special_cases():
    rng = np.random.default_rng(15)
    qh, kvh, d = 8, 2, 64
    q = rng.standard_normal((qh, d))
    V = rng.standard_normal((kvh, 1, d))
    K = rng.standard_normal((kvh, 1, d))
    out = oracle.slot_attention(q, K, V)
    for h in range(qh):   # one position: o = V0 exactly
        np.testing.assert_array_equal(out[h], V[h // 4, 0])
    L = 9
    K = np.repeat(rng.standard_normal((kvh, 1, d)), L, axis=1)
    V = rng.standard_normal((kvh, L, d))
    out = oracle.slot_attention(q, K, V)
    for h in range(qh):   # equal keys: o = mean(V)
        np.testing.assert_allclose(out[h], V[h // 4].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attention_brute_force_and_gqa_map():
    rng = np.random.default_rng(16)
    qh, kvh, d, L = 8, 2, 16, 13
    q = rng.standard_normal((qh, d))
    K = rng.standard_normal((kvh, L, d))
    V = rng.standard_normal((kvh, L, d))
    out = oracle.slot_attention(q, K, V)
    for h in range(qh):
        kv = h // (qh // kvh)
        s = [sum(q[h][i] * K[kv][j][i] for i in range(d)) / math.sqrt(d) for j in range(L)]
        e = [math.exp(v) for v in s]
        z = sum(e)
        o = [sum(e[j] / z * V[kv][j][i] for j in range(L)) for i in range(d)]
        np.testing.assert_allclose(out[h], o, rtol=1e-12)
    perm = rng.permutation(L)   # positions are a set: permuting K, V together
    np.testing.assert_allclose(oracle.slot_attention(q, K[:, perm], V[:, perm]), out, rtol=1e-12)


def test_causal_block_attention_brute_force_and_causality():
    rng = np.random.default_rng(17)
    qh, kvh, d, start, P = 8, 2, 16, 5, 4
    Q = rng.standard_normal((P, qh, d))
    K = rng.standard_normal((kvh, start + P, d))
    V = rng.standard_normal((kvh, start + P, d))
    out = oracle.causal_block_attention(Q, K, V, start)
    for i in range(P):              # row i: softmax over positions 0..start+i only
        n = start + i + 1
        for h in range(qh):
            kv = h // (qh // kvh)
            s = [sum(Q[i][h][t] * K[kv][j][t] for t in range(d)) / math.sqrt(d) for j in range(n)]
            m = max(s)
            e = [math.exp(v - m) for v in s]
            z = sum(e)
            o = [sum(e[j] / z * V[kv][j][t] for j in range(n)) for t in range(d)]
            np.testing.assert_allclose(out[i][h], o, rtol=1e-12)
    # positions past start + 1 are invisible to rows 0 and 1, visible to rows 2 and 3
    K2, V2 = K.copy(), V.copy()
    K2[:, start + 2:] = rng.standard_normal((kvh, P - 2, d))
    V2[:, start + 2:] = rng.standard_normal((kvh, P - 2, d))
    out2 = oracle.causal_block_attention(Q, K2, V2, start)
    np.testing.assert_array_equal(out2[:2], out[:2])
    assert np.abs(out2[2:] - out[2:]).min() > 0
    # an empty prefix and one query: the one visible position, o = V0
    o1 = oracle.causal_block_attention(Q[:1], K[:, :1], V[:, :1], 0)
    for h in range(qh):
        np.testing.assert_array_equal(o1[0][h], V[h // 4, 0])


# ---------------------------------------------------------------- routing

def test_router_hand_values():
    t = table("router.txt")
    for case in ("case1", "case2"):
        logits = np.array([[float(v) for v in t[case + "_logits"]]])
        # H = E, Wr = identity: the logits are the input row itself
        ids, w = oracle.route_topk(logits, np.eye(logits.shape[1]), int(t[case + "_k"][0]))
        assert list(ids[0]) == [int(v) for v in t[case + "_ids"]]
        np.testing.assert_allclose(w[0], [float(v) for v in t[case + "_weights"]], rtol=1e-13)


def test_router_invariants():
    rng = np.random.default_rng(17)
    B, H, E, k = 6, 64, 32, 4
    x = rng.standard_normal((B, H))
    Wr = rng.standard_normal((E, H)) * 0.1
    ids, w = oracle.route_topk(x, Wr, k)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-13)
    logits = x @ Wr.T
    for b in range(B):   # top-k = the first k of a full descending sort
        full = sorted(range(E), key=lambda e: (-logits[b, e], e))
        assert list(ids[b]) == full[:k]
        assert np.all(np.diff(w[b]) <= 0)
    perm = rng.permutation(E)  # relabelling experts relabels the choice
    ids2, w2 = oracle.route_topk(x, Wr[perm], k)
    np.testing.assert_array_equal(perm[ids2], ids)
    np.testing.assert_allclose(w2, w, rtol=1e-13)
    _, wraw = oracle.route_topk(x, Wr, k, renorm=False)
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(wraw, np.take_along_axis(p, ids, 1), rtol=1e-12)


# ---------------------------------------------------------------- experts

def _q(rng, N, K, g):
    return oracle.quantize_w4((rng.standard_normal((N, K)) * 0.02).astype(np.float32), g)


def test_silu_values():
    for r in lines("small_values.txt"):
        if r[0] == "silu":
            assert oracle.silu(float(r[1])) == pytest.approx(float(r[2]), abs=1e-15)


def test_expert_ffn_special_cases():
    rng = np.random.default_rng(18)
    H, F, g = 128, 64, 32
    wg, wu, wd = _q(rng, F, H, g), _q(rng, F, H, g), _q(rng, H, F, g)
    ident = lambda a: a
    zero = oracle.expert_ffn(np.zeros(H), wg, wu, wd, H, F, g, ident)
    assert np.all(zero == 0)
    x = rng.standard_normal(H)
    Wg = oracle.dequant_w4(*wg, H, g)
    Wu = oracle.dequant_w4(*wu, H, g)
    Wd = oracle.dequant_w4(*wd, F, g)
    plain = Wd @ ((Wg @ x) / (1 + np.exp(-(Wg @ x))) * (Wu @ x))
    np.testing.assert_allclose(oracle.expert_ffn(x, wg, wu, wd, H, F, g, ident), plain, rtol=1e-12)
    # a single expert with weight 1 is the plain FFN plus the residual
    h = rng.standard_normal(H)
    np.testing.assert_allclose(oracle.moe_combine(h, [plain], [1.0]), h + plain, rtol=1e-14)
    # combine is linear in the weights and ordered by rank
    o2 = rng.standard_normal(H)
    np.testing.assert_allclose(oracle.moe_combine(h, [plain, o2], [0.25, 0.75]),
                               h + 0.25 * plain + 0.75 * o2, rtol=1e-13)
