"""Host arithmetic of bench.py: the weight-bytes roofline per B."""

import pytest

import bench
import synth


def test_weight_roofline_matches_hand_count():
    cfg = dict(synth.CONFIGS["full_model"])
    # int4 bytes of one matrix = rows * K / 2 + rows * (K / 64) * 2
    qkv = 5120 * 1024 + 5120 * 32 * 2        # 5,570,560
    o = 2048 * 2048 + 2048 * 64 * 2          # 4,456,448
    expert = (1536 * 1024 + 1536 * 32 * 2) + (2048 * 384 + 2048 * 12 * 2)
    assert expert == 2_506_752
    router = 128 * 2048 * 4
    head = 151936 * 2048 * 2
    for B, active in ((1, 8.0), (2, 15.5), (32, 128 * (1 - (15 / 16) ** 32))):
        step = 48 * (qkv + o + router + active * expert) + head
        want = B * 6776.3e9 / step
        assert bench.weight_roofline_tok_s(cfg, 48, B, 6776.3) == pytest.approx(want, rel=1e-12)
    # B = 1 streams ~2.12 GB per token: ~3.2k tok/s at the measured copy bandwidth
    assert bench.weight_roofline_tok_s(cfg, 48, 1, 6776.3) == pytest.approx(3201.6, abs=0.1)
    # more streams share the same bytes: the roofline rises with B
    r = [bench.weight_roofline_tok_s(cfg, 48, B, 6776.3) for B in (1, 2, 4, 8, 16, 32, 64, 128)]
    assert all(a < b for a, b in zip(r, r[1:]))
