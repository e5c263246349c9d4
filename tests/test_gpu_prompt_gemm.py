"""GPU parity of the prompt-length W4A16 GEMM on the tcgen05 tensor cores
(w4_gemm_prompt_tc, the kernel of prompt ingestion with prefill_tc): the
dense micro's shapes and the expert and tiny-layer shapes, M from one row to
512 (partial column groups, one and several 128-row tiles, a ragged last
tile), against the oracle; a row's bytes do not depend on M or on its
neighbours, and repeated launches give the same bytes."""

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


def _weights(bm, N, K, g, tag):
    raw = synth.normal((N, K), 0.02, synth.seed_of("dense_micro", "prompt", tag, N, K))
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, K // g), dtype=torch.float16, device="cuda")
    bm.bm_w4_quantize(raw.cuda(), N, K, g, packed, scales)
    wm = torch.empty_like(packed)
    sm = torch.empty((N * (K // g) // 2,), dtype=torch.int32, device="cuda")
    bm.bm_w4_repack_mma(packed, scales, N, K, g, wm, sm)
    torch.cuda.synchronize()
    return raw, wm, sm


def _gemm(bm, wm, sm, X16, N, K, g, R=None):
    M = X16.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bm.w4_gemm_prompt_tc(wm, sm, X16, Y, R, M, N, K, g)
    torch.cuda.synchronize()
    return Y


@pytest.mark.parametrize("N,K,g", [(5120, 2048, 64), (2048, 4096, 64), (1536, 2048, 64), (2048, 768, 64),
                                   (768, 512, 32), (512, 256, 32), (256, 768, 128)])
def test_prompt_gemm_matches_oracle(bm, N, K, g):
    raw, wm, sm = _weights(bm, N, K, g, "t")
    p_ref, s_ref = oracle.quantize_w4(raw.numpy(), g)
    X = synth.activations("dense_micro", "xprompt", (512, K))
    ref = oracle.bf16_round(oracle.w4_gemm(X.double().numpy(), p_ref, s_ref, K, g))
    X16 = X.cuda().half()
    full = _gemm(bm, wm, sm, X16, N, K, g)
    assert_close_rows(full, ref, what=f"prompt gemm N={N} K={K} g={g} M=512")
    for rep in range(2):
        again = _gemm(bm, wm, sm, X16, N, K, g)
        assert torch.equal(again.view(torch.int16), full.view(torch.int16)), f"repeat {rep}: bytes differ"
    for M in (1, 13, 16, 128, 129, 300):
        Y = _gemm(bm, wm, sm, X16[:M].contiguous(), N, K, g)
        assert torch.equal(Y.view(torch.int16), full[:M].view(torch.int16)), f"M={M}: bytes depend on M"
    # rows in another order: each row keeps its bytes
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(5))
    Yp = _gemm(bm, wm, sm, X16[perm.cuda()].contiguous(), N, K, g)
    assert torch.equal(Yp.view(torch.int16), full[perm.cuda()].view(torch.int16))


def test_prompt_gemm_residual_and_rejections(bm):
    N, K, g = 2048, 4096, 64
    raw, wm, sm = _weights(bm, N, K, g, "r")
    p_ref, s_ref = oracle.quantize_w4(raw.numpy(), g)
    X = synth.activations("dense_micro", "xprompt_r", (200, K))
    R = synth.activations("dense_micro", "rprompt_r", (200, N))
    ref = oracle.bf16_round(oracle.w4_gemm(X.double().numpy(), p_ref, s_ref, K, g) + R.double().numpy())
    Y = _gemm(bm, wm, sm, X.cuda().half(), N, K, g, R.cuda())
    assert_close_rows(Y, ref, what="prompt gemm + residual")
    with pytest.raises(bm.BitMoeError) as ei:
        bm.w4_gemm_prompt_tc(wm, sm, X.cuda().half(), Y, None, 200, 96, K, g)   # N not a multiple of 128
    assert ei.value.status == 1
    with pytest.raises(bm.BitMoeError) as ei:
        bm.w4_gemm_prompt_tc(wm, sm, X.cuda().half(), Y, None, 200, N, 384, g)   # K not a multiple of 256
    assert ei.value.status == 1
