"""The per-op arithmetic of one decode step, in plain fp64 numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Each function states the passage it follows.  Library primitives used as
steps: ``numpy.matmul`` (fp64), ``numpy.exp``, ``numpy.argsort`` (stable).
There is no blocking, fusion or reordering beyond the definitions below.
"""

import math

import numpy as np

from .numerics import dequant_w4


def w4_gemm(X, packed, scales, K, g):
    """Y = X · Wᵀ with W the dequantized int4 weight, fp64 accumulation.

    [Batched serving, §1 Contribution]: each dense projection is one batched
    4-bit GEMM over the B rows, so its packed weights are read once per step;
    [Batched serving, §3 Results]: each row's result is computed independently
    of the other rows.  X is [M][K] (bf16 values as float64), the result is
    [M][N] float64 (unrounded).
    """
    W = dequant_w4(packed, scales, K, g)
    X = np.asarray(X, dtype=np.float64)
    assert X.shape[1] == K
    return rowwise(W, X)


def rowwise(W, X):
    """Y[m] = W · X[m] for each row m on its own (one matrix-vector product
    per row), so a row's result never depends on the other rows."""
    X = np.asarray(X, dtype=np.float64)
    if X.shape[0] == 0:
        return np.zeros((0, W.shape[0]), dtype=np.float64)
    return np.stack([W @ X[m] for m in range(X.shape[0])])


def rmsnorm(x, weight=None, eps=1e-6):
    """y = x / sqrt(mean(x²) + eps) · weight, per row of x.

    The normalisation layer of the decoder; the pages name the model only as
    a 30B-class MoE, so the standard pre-norm RMSNorm is the reading.  A
    weight of None means all ones.
    """
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    y = x * r
    if weight is not None:
        y = y * np.asarray(weight, dtype=np.float64)
    return y


def rope_rotate_half(x, pos, base):
    """Rotary position embedding, rotate-half pairing (i, i + d/2).

    x is [..., heads, d]; pos is an integer position (or an array broadcast
    over the leading axes).  theta_i = base^(-2i/d); angle = pos·theta_i,
    both in fp64.  x'_i = x_i cos − x_{i+d/2} sin, x'_{i+d/2} = x_{i+d/2} cos
    + x_i sin.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * i / d)
    pos = np.asarray(pos, dtype=np.float64)
    ang = pos[..., None, None] * theta if pos.ndim else pos * theta
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def slot_attention(q, K, V):
    """Grouped-query decode attention of one stream over its slot.

    q: [qh][d] (the one new query), K, V: [kvh][L][d] holding positions
    0..L-1 of the stream's slot, the new token included (it is appended
    before attention).  Query head h reads KV head h // (qh / kvh).
    s_j = q·K_j / sqrt(d); p = softmax(s) with max subtraction; o = Σ p_j V_j.
    [KV-slot isolation, §1 Contribution]: attention reads the stream's own
    slot of the batched KV arena and nothing else.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    qh, d = q.shape
    kvh, L, _ = K.shape
    assert L >= 1 and qh % kvh == 0
    group = qh // kvh
    out = np.empty((qh, d), dtype=np.float64)
    for h in range(qh):
        kv = h // group
        s = (K[kv] @ q[h]) / math.sqrt(d)
        p = np.exp(s - s.max())
        p = p / p.sum()
        out[h] = p @ V[kv]
    return out


def causal_block_attention(Q, K, V, start):
    """Causal grouped-query attention of a block of P consecutive queries.

    Q: [P][qh][d], the queries of positions start .. start+P-1; K, V:
    [kvh][start+P][d], the slot's positions with the block's own keys
    already in place.  Query row i may see positions 0..start+i: the score
    matrix of each head is formed whole, entries j > start+i are set to -inf
    before a row-wise softmax (max subtracted), and O = P V.  This is the
    decode attention of ``slot_attention`` applied to every row of a prompt
    at once ([KV-slot isolation, §1 Contribution]: a stream's K/V grows one
    position per token, so row i's keys are those of its own prefix).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    P, qh, d = Q.shape
    kvh, L, _ = K.shape
    assert L == start + P and qh % kvh == 0
    group = qh // kvh
    visible = np.arange(L)[None, :] <= (start + np.arange(P))[:, None]   # [P][L]
    out = np.empty((P, qh, d), dtype=np.float64)
    for h in range(qh):
        kv = h // group
        S = (Q[:, h, :] @ K[kv].T) / math.sqrt(d)
        S = np.where(visible, S, -np.inf)
        E = np.exp(S - S.max(axis=1, keepdims=True))
        out[:, h, :] = (E / E.sum(axis=1, keepdims=True)) @ V[kv]
    return out


def silu(x):
    """SiLU(x) = x / (1 + exp(-x))."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def route_topk(xn, Wr, k, renorm=True):
    """Top-k expert routing of each token.

    [Batched serving, §1 Contribution] sends each stream to the experts its
    router selects; the router's form is not printed.  Reading: logits = xn · Wrᵀ
    (Wr fp32 [E][H]), p = softmax(logits) over all E experts, the k experts of
    largest p are selected (equal p: lower expert id first), and their weights
    are p renormalised to sum to one (or left as p when renorm is False).
    Returns (ids int32 [B][k] in rank order, weights float64 [B][k]).
    """
    xn = np.asarray(xn, dtype=np.float64)
    logits = rowwise(np.asarray(Wr, dtype=np.float64), xn)
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)
    B = p.shape[0]
    ids = np.empty((B, k), dtype=np.int32)
    w = np.empty((B, k), dtype=np.float64)
    for b in range(B):
        order = np.argsort(-p[b], kind="stable")[:k]
        ids[b] = order
        w[b] = p[b, order]
        if renorm:
            w[b] = w[b] / w[b].sum()
    return ids, w


def expert_ffn(x, wg, wu, wd, H, F, g, round_act):
    """One expert's FFN on one token: W_d · (SiLU(W_g x) ⊙ (W_u x)).

    wg, wu are (packed, scales) for [F][H]; wd for [H][F].  ``round_act`` is
    applied to the F-wide activation SiLU(g)·u (the A16 rounding point) before
    the down projection.  Returns the unrounded [H] output.
    """
    x = np.asarray(x, dtype=np.float64)[None, :]
    gv = w4_gemm(x, wg[0], wg[1], H, g)[0]
    uv = w4_gemm(x, wu[0], wu[1], H, g)[0]
    a = round_act(silu(gv) * uv)
    return w4_gemm(a[None, :], wd[0], wd[1], F, g)[0]


def moe_combine(h, outs, weights):
    """y = h + Σ_r w_r · out_r, summed in rank order r = 0..k-1.

    h: [H] residual input; outs: [k][H] expert outputs; weights: [k].
    """
    y = np.asarray(h, dtype=np.float64).copy()
    acc = np.zeros_like(y)
    for r in range(len(weights)):
        acc = acc + weights[r] * np.asarray(outs[r], dtype=np.float64)
    return y + acc
