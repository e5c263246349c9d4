"""Comparison rules of the GPU-vs-oracle parity tests.

Float outputs: per row (stream), max |gpu - oracle| <= 2e-2 and cosine
similarity >= 0.9999 (the tolerance the decode path is specified to).
Integer decisions taken from floating point (greedy ids, top-k expert ids):
bit-exact, except where the oracle's own margin between the candidates is
below the float error bound, where either choice is correct.

Every comparison is recorded (``RECORD``): the measured max-abs error, the
lowest row cosine, and how many elements differ by more than 2e-2.  The
session prints the table at its end and, when the environment variable
BM_PARITY_LOG names a file, writes it there as JSON.
"""

import numpy as np
import torch

MAX_ABS = 2e-2
MIN_COS = 0.9999

RECORD = []


def to64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def assert_close_rows(gpu, ref, max_abs=MAX_ABS, min_cos=MIN_COS, what="", bf16_out=True):
    """Rows of gpu vs oracle.  For bf16 outputs an element may also differ by
    one bf16 ulp of the oracle value: both sides round once to bf16 from
    values that differ only by accumulation order, and a rounding boundary
    between them flips one ulp (0.031 at |y| in [4, 8)).  Elements that use
    that allowance are counted in the record (``ulp_flips``)."""
    g, r = to64(gpu), to64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    g2, r2 = g.reshape(g.shape[0], -1), r.reshape(r.shape[0], -1)
    diff = np.abs(g2 - r2)
    allowed = np.maximum(max_abs, bf16_ulp(r2)) if bf16_out else max_abs
    bad = diff > allowed
    over = diff > max_abs
    err = diff.max(axis=1) if diff.size else np.zeros(1)
    num = (g2 * r2).sum(axis=1)
    den = np.linalg.norm(g2, axis=1) * np.linalg.norm(r2, axis=1)
    cos = np.where(den > 0, num / np.where(den > 0, den, 1), 1.0)
    RECORD.append({"what": what, "elements": int(diff.size), "max_abs": float(err.max()),
                   "min_cos": float(cos.min()) if cos.size else 1.0, "bound": float(max_abs),
                   "ulp_flips": int(over.sum()) if bf16_out else 0})
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond max({max_abs:g}, 1 bf16 ulp); worst "
                           f"|diff| {diff[bad].max():.3g} at |y| {np.abs(r2[bad]).max():.3g}; rows "
                           f"{np.nonzero(bad.any(axis=1))[0][:8].tolist()}")
    assert np.all(cos >= min_cos), f"{what}: cosine {cos.min():.8f} < {min_cos}"
    return float(err.max()), float(cos.min())


def check_greedy(gpu_ids, ref_logits, err_bound):
    """Greedy ids equal the oracle's argmax unless the oracle's top-1/top-2
    margin is within 4x the measured logit error (a tie).  Returns the number
    of rows that were ties."""
    ref = to64(ref_logits)
    ties = 0
    for b, gid in enumerate(np.asarray(gpu_ids).reshape(-1)):
        best = int(np.argmax(ref[b]))
        if int(gid) == best:
            continue
        margin = ref[b, best] - ref[b, int(gid)]
        assert margin <= 4 * err_bound, f"row {b}: gpu id {gid} vs oracle {best}, margin {margin:.3g}"
        ties += 1
    return ties


def topk_near_tie(logits_row, ids, eps):
    """True if the oracle's ranking of the top-k+1 logits has a gap below eps."""
    s = np.sort(np.asarray(logits_row))[::-1][: len(ids) + 1]
    return bool(np.any(np.abs(np.diff(s)) < eps))
