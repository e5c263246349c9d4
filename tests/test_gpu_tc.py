"""GPU parity of the tensor-core (tcgen05) W4A16 GEMM: the repack into the
tensor-core layout, dense shapes of the dense micro (K = 2048 / N = 5120,
K = 4096 / N = 2048, M in {1, 2, 4, 8, 16, 32, 64}) and of the tiny layer,
against the oracle; and the same token gives the same bytes whatever column,
padding and neighbours it has in its MMA (a stream's result does not depend
on its batch)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_close_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bm():
    import bit_moe_decode_w4a16_gb300 as m
    m.build()
    return m


def _weights_tc(bm, N, K, g, tag):
    raw = synth.normal((N, K), 0.02, synth.seed_of("dense_micro", "tc", tag, N, K))
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, K // g), dtype=torch.float16, device="cuda")
    bm.bm_w4_quantize(raw.cuda(), N, K, g, packed, scales)
    wtc = torch.empty_like(packed)
    stc = torch.empty_like(scales)
    bm.bm_w4_repack_tc(packed, scales, N, K, g, wtc, stc)
    torch.cuda.synchronize()
    return raw, wtc, stc


def _gemm_tc(bm, wtc, stc, X, N, K, g, R=None):
    M = X.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bm.w4_gemm_batched_tc(wtc, stc, X, Y, R, M, N, K, g)
    torch.cuda.synchronize()
    return Y


@pytest.mark.parametrize("N,K,g", [(5120, 2048, 64), (2048, 4096, 64), (768, 512, 32), (512, 256, 32),
                                   (256, 768, 128)])
def test_tc_gemm_matches_oracle(bm, N, K, g):
    raw, wtc, stc = _weights_tc(bm, N, K, g, "t")
    p_ref, s_ref = oracle.quantize_w4(raw.numpy(), g)
    X = synth.activations("dense_micro", "xtc", (64, K))
    R = synth.activations("dense_micro", "rtc", (64, N))
    ref = oracle.w4_gemm(X.double().numpy(), p_ref, s_ref, K, g)
    full = _gemm_tc(bm, wtc, stc, X.cuda(), N, K, g)
    for M in (1, 2, 4, 8, 16, 17, 32, 64):
        Y = _gemm_tc(bm, wtc, stc, X[:M].contiguous().cuda(), N, K, g)
        assert_close_rows(Y, oracle.bf16_round(ref[:M]), what=f"tc gemm N={N} K={K} M={M}")
        # same token, other column / padding / neighbours -> same bytes
        assert torch.equal(Y.view(torch.int16), full[:M].view(torch.int16)), f"M={M}"
    Yr = _gemm_tc(bm, wtc, stc, X[:5].contiguous().cuda(), N, K, g, R[:5].contiguous().cuda())
    assert_close_rows(Yr, oracle.bf16_round(ref[:5] + R[:5].double().numpy()), what="tc gemm + residual")


def test_tc_token_position_independence(bm):
    N, K, g = 1024, 2048, 64
    _, wtc, stc = _weights_tc(bm, N, K, g, "pos")
    X = synth.activations("dense_micro", "xpos", (48, K)).cuda()
    full = _gemm_tc(bm, wtc, stc, X, N, K, g)
    for m in (0, 7, 15, 16, 31, 47):
        solo = _gemm_tc(bm, wtc, stc, X[m:m + 1].contiguous(), N, K, g)
        assert torch.equal(solo.view(torch.int16), full[m:m + 1].view(torch.int16)), m
    perm = torch.randperm(48, generator=torch.Generator().manual_seed(3)).tolist()
    shuffled = _gemm_tc(bm, wtc, stc, X[perm].contiguous(), N, K, g)
    assert torch.equal(shuffled.view(torch.int16), full[perm].view(torch.int16))


def test_tc_closed_form(bm):
    N, K, g, M = 128, 2048, 64, 3
    packed = torch.full((N, K // 2), 0x99, dtype=torch.uint8, device="cuda")
    scales = torch.ones((N, K // g), dtype=torch.float16, device="cuda")
    wtc, stc = torch.empty_like(packed), torch.empty_like(scales)
    bm.bm_w4_repack_tc(packed, scales, N, K, g, wtc, stc)
    X = torch.zeros((M, K), dtype=torch.bfloat16)
    X[0, :] = 1.0
    X[1, ::2] = 0.5
    X[2, 7] = -3.0
    Y = _gemm_tc(bm, wtc, stc, X.cuda(), N, K, g).float().cpu()
    assert torch.all(Y[0] == 2048) and torch.all(Y[1] == 512) and torch.all(Y[2] == -3)
    # one nonzero code per row at a known k checks the K order of the layout
    packed.fill_(0x88)
    rows = torch.arange(N)
    ks = (rows * 37) % K
    pk = packed.cpu()
    for r, k in zip(rows.tolist(), ks.tolist()):
        pk[r, k // 2] = 0x98 if k % 2 else 0x89        # code +1 at element k (high nibble if k is odd)
    packed.copy_(pk)
    bm.bm_w4_repack_tc(packed, scales, N, K, g, wtc, stc)
    k_all = torch.arange(K)
    # two exact bf16 probes whose pair identifies k: k mod 256 and k div 256
    Xp = torch.stack([(k_all % 256).float(), (k_all // 256).float()]).to(torch.bfloat16)
    Y = _gemm_tc(bm, wtc, stc, Xp.cuda(), N, K, g).float().cpu()
    assert torch.equal(Y[0], (ks % 256).float()) and torch.equal(Y[1], (ks // 256).float())
