"""GPU parity of the warp-MMA (mma.sync m16n8k16, bf16) W4A16 GEMM: the
repack into the mma layout and the projection kernel on the dense micro's
shapes (K = 2048 / N = 5120, K = 4096 / N = 2048, M in {1, 2, 4, 8, 16, 32,
64}), the tiny layer's shapes and ragged ones (rows not a multiple of the
CTA's row block, every group size), against the oracle; a token's bytes do
not depend on its column, padding or neighbours; closed forms and a probe of
the K order of the layout."""

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


def _repack(bm, packed, scales, N, K, g):
    wm = torch.empty_like(packed)
    sm = torch.empty((N * (K // g) // 2,), dtype=torch.int32, device="cuda")
    bm.bm_w4_repack_mma(packed, scales, N, K, g, wm, sm)
    return wm, sm


def _weights(bm, N, K, g, tag):
    raw = synth.normal((N, K), 0.02, synth.seed_of("dense_micro", "mma", tag, N, K))
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, K // g), dtype=torch.float16, device="cuda")
    bm.bm_w4_quantize(raw.cuda(), N, K, g, packed, scales)
    wm, sm = _repack(bm, packed, scales, N, K, g)
    torch.cuda.synchronize()
    return raw, wm, sm


def _gemm(bm, wm, sm, X, N, K, g, R=None):
    M = X.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bm.w4_gemm_batched_mma(wm, sm, X, Y, R, M, N, K, g)
    torch.cuda.synchronize()
    return Y


@pytest.mark.parametrize("N,K,g", [(5120, 2048, 64), (2048, 4096, 64), (768, 512, 32), (512, 256, 32),
                                   (256, 768, 128), (96, 384, 128), (2048, 768, 64), (160, 1024, 32)])
def test_mma_gemm_matches_oracle(bm, N, K, g):
    raw, wm, sm = _weights(bm, N, K, g, "t")
    p_ref, s_ref = oracle.quantize_w4(raw.numpy(), g)
    X = synth.activations("dense_micro", "xmma", (64, K))
    R = synth.activations("dense_micro", "rmma", (64, N))
    ref = oracle.w4_gemm(X.double().numpy(), p_ref, s_ref, K, g)
    full = _gemm(bm, wm, sm, X.cuda(), N, K, g)
    for M in (1, 2, 4, 8, 9, 16, 17, 32, 33, 64):
        Y = _gemm(bm, wm, sm, X[:M].contiguous().cuda(), N, K, g)
        assert_close_rows(Y, oracle.bf16_round(ref[:M]), what=f"mma gemm N={N} K={K} g={g} M={M}")
        # same token, other column / padding / neighbours -> same bytes
        assert torch.equal(Y.view(torch.int16), full[:M].view(torch.int16)), f"M={M}"
    Yr = _gemm(bm, wm, sm, X[:5].contiguous().cuda(), N, K, g, R[:5].contiguous().cuda())
    assert_close_rows(Yr, oracle.bf16_round(ref[:5] + R[:5].double().numpy()), what="mma gemm + residual")


def test_mma_token_position_independence(bm):
    N, K, g = 1024, 2048, 64
    _, wm, sm = _weights(bm, N, K, g, "pos")
    X = synth.activations("dense_micro", "xpos", (48, K)).cuda()
    full = _gemm(bm, wm, sm, X, N, K, g)
    for m in (0, 7, 8, 15, 16, 31, 47):
        solo = _gemm(bm, wm, sm, X[m:m + 1].contiguous(), N, K, g)
        assert torch.equal(solo.view(torch.int16), full[m:m + 1].view(torch.int16)), m
    perm = torch.randperm(48, generator=torch.Generator().manual_seed(3)).tolist()
    shuffled = _gemm(bm, wm, sm, X[perm].contiguous(), N, K, g)
    assert torch.equal(shuffled.view(torch.int16), full[perm].view(torch.int16))


@pytest.mark.parametrize("g", [32, 64, 128])
def test_mma_closed_form_and_k_order(bm, g):
    N, K, M = 128, 2048, 3
    packed = torch.full((N, K // 2), 0x99, dtype=torch.uint8, device="cuda")   # every code q = +1
    scales = torch.ones((N, K // g), dtype=torch.float16, device="cuda")
    wm, sm = _repack(bm, packed, scales, N, K, g)
    X = torch.zeros((M, K), dtype=torch.bfloat16)
    X[0, :] = 1.0
    X[1, ::2] = 0.5
    X[2, 7] = -3.0
    Y = _gemm(bm, wm, sm, X.cuda(), N, K, g).float().cpu()
    assert torch.all(Y[0] == 2048) and torch.all(Y[1] == 512) and torch.all(Y[2] == -3)
    # one nonzero code per row at a known k checks the K order of the layout
    packed.fill_(0x88)
    rows = torch.arange(N)
    ks = (rows * 37 + 5) % K
    pk = packed.cpu()
    for r, k in zip(rows.tolist(), ks.tolist()):
        pk[r, k // 2] = 0x98 if k % 2 else 0x89        # code +1 at element k (high nibble if k is odd)
    packed.copy_(pk)
    wm, sm = _repack(bm, packed, scales, N, K, g)
    k_all = torch.arange(K)
    # two exact bf16 probes whose pair identifies k: k mod 256 and k div 256
    Xp = torch.stack([(k_all % 256).float(), (k_all // 256).float()]).to(torch.bfloat16)
    Y = _gemm(bm, wm, sm, Xp.cuda(), N, K, g).float().cpu()
    assert torch.equal(Y[0], (ks % 256).float()) and torch.equal(Y[1], (ks // 256).float())
    # per-row, per-group scales land on their own rows and groups: scale
    # (r % 7 + 1) * 2^-(j % 3) on group j of row r, all codes -8, x = 1
    packed.fill_(0x00)
    sc = torch.tensor([[(r % 7 + 1) * 2.0 ** -(j % 3) for j in range(K // g)] for r in range(N)],
                      dtype=torch.float16)
    wm, sm = _repack(bm, packed, sc.cuda(), N, K, g)
    Y = _gemm(bm, wm, sm, torch.ones((1, K), dtype=torch.bfloat16, device="cuda"), N, K, g).float().cpu()[0]
    want = torch.tensor([-8.0 * g * float(sc[r].double().sum()) for r in range(N)])
    assert torch.equal(Y, want.to(torch.bfloat16).float())
