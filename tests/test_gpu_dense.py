"""GPU parity of the int4 encoder and the batched W4A16 GEMM (dense micro:
K = 2048 with N = 5120, K = 4096 with N = 2048, M in {1, 2, 4, 8, 16, 32, 64},
group 64), plus ragged shapes and solo-vs-batched byte identity."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_rows

pytestmark = pytest.mark.gpu

NAME = "dense_micro"
ROWS = (1, 2, 4, 8, 16, 32, 64)


@pytest.fixture(scope="module")
def bm():
    import bit_moe_decode_w4a16_gb300 as m
    m.build()
    return m


def _weights(bm, N, K, g, tag):
    raw = synth.normal((N, K), 0.02, synth.seed_of(NAME, "w", tag, N, K))
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, K // g), dtype=torch.float16, device="cuda")
    bm.bm_w4_quantize(raw.cuda(), N, K, g, packed, scales)
    torch.cuda.synchronize()
    return raw, packed, scales


def _gemm(bm, packed, scales, X, N, K, g, R=None):
    M = X.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bm.w4_gemm_batched(packed, scales, X, Y, R, M, N, K, g)
    torch.cuda.synchronize()
    return Y


@pytest.mark.parametrize("N,K,g", [(5120, 2048, 64), (2048, 4096, 64), (1000, 768, 32), (96, 512, 32),
                                   (130, 256, 128)])
def test_encoder_matches_oracle(bm, N, K, g):
    raw, packed, scales = _weights(bm, N, K, g, "enc")
    raw_np = raw.numpy().copy()
    raw_np[N // 3, :g] = 0.0           # an all-zero group
    raw_np[1, g: 2 * g] *= 1e-6        # a group whose scale is subnormal in fp16
    raw_t = torch.from_numpy(raw_np)
    bm.bm_w4_quantize(raw_t.cuda(), N, K, g, packed, scales)
    torch.cuda.synchronize()
    p_ref, s_ref = oracle.quantize_w4(raw_np, g)
    np.testing.assert_array_equal(packed.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint16), s_ref.view(np.uint16))


@pytest.mark.parametrize("N,K", [(5120, 2048), (2048, 4096)])
def test_w4_gemm_matches_oracle_all_batch_sizes(bm, N, K):
    g = 64
    raw, packed, scales = _weights(bm, N, K, g, "gemm")
    p_ref, s_ref = oracle.quantize_w4(raw.numpy(), g)
    X = synth.activations(NAME, "x", (64, K))
    Xg = X.cuda()
    X64 = X.double().numpy()
    ref = oracle.bf16_round(oracle.w4_gemm(X64, p_ref, s_ref, K, g))
    full = _gemm(bm, packed, scales, Xg, N, K, g)
    for M in ROWS:
        Y = _gemm(bm, packed, scales, Xg[:M].contiguous(), N, K, g)
        assert_close_rows(Y, ref[:M], what=f"w4_gemm N={N} K={K} M={M}")
        # solo == batched, byte for byte: a row's result never depends on M
        assert torch.equal(Y.view(torch.int16), full[:M].view(torch.int16)), f"M={M} differs from M=64 rows"
    for m in (0, 17, 63):
        solo = _gemm(bm, packed, scales, Xg[m:m + 1].contiguous(), N, K, g)
        assert torch.equal(solo.view(torch.int16), full[m:m + 1].view(torch.int16))


@pytest.mark.parametrize("N,K,g,M", [(1000, 768, 32, 5), (96, 512, 32, 3), (130, 256, 128, 7), (5120, 2048, 64, 33)])
def test_w4_gemm_ragged_and_residual(bm, N, K, g, M):
    raw, packed, scales = _weights(bm, N, K, g, "ragged")
    p_ref, s_ref = oracle.quantize_w4(raw.numpy(), g)
    X = synth.activations(NAME, "xr", (M, K))
    R = synth.activations(NAME, "res", (M, N))
    ref = oracle.bf16_round(oracle.w4_gemm(X.double().numpy(), p_ref, s_ref, K, g) + R.double().numpy())
    Y = _gemm(bm, packed, scales, X.cuda(), N, K, g, R.cuda())
    assert_close_rows(Y, ref, what=f"w4_gemm+res N={N} K={K} M={M}")


def test_w4_gemm_closed_form(bm):
    # every code +1 (byte 0x99) and unit scales: y = sum(x), exactly representable
    N, K, g, M = 16, 2048, 64, 3
    packed = torch.full((N, K // 2), 0x99, dtype=torch.uint8, device="cuda")
    scales = torch.ones((N, K // g), dtype=torch.float16, device="cuda")
    X = torch.zeros((M, K), dtype=torch.bfloat16)
    X[0, :] = 1.0
    X[1, ::2] = 0.5
    X[2, 7] = -3.0
    Y = _gemm(bm, packed, scales, X.cuda(), N, K, g).float().cpu()
    assert torch.all(Y[0] == 2048) and torch.all(Y[1] == 512) and torch.all(Y[2] == -3)


def test_w4_gemm_deterministic(bm):
    N, K, g = 5120, 2048, 64
    _, packed, scales = _weights(bm, N, K, g, "det")
    X = synth.activations(NAME, "xd", (32, K)).cuda()
    a = _gemm(bm, packed, scales, X, N, K, g)
    b = _gemm(bm, packed, scales, X, N, K, g)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
