"""Pins of the oracle's byte arithmetic against the numbers the pages print
(tests/golden/pages_capacity.txt)."""
import pytest

from conftest import read_golden

ROWS = read_golden("pages_capacity.txt")


def test_bytes_per_token_70b(orc):
    for r in ROWS:
        if r[0] == "bytes_per_token":
            fmt, L, H, D, expect = r[1], int(r[2]), int(r[3]), int(r[4]), int(r[5])
            assert orc.bytes_per_token(fmt, L, H, D) == expect
    # FP8 halves BF16; the 4.5-bit block formats carry one scale byte per 16 elements
    assert orc.bytes_per_token("fp8_e4m3", 80, 8, 128) == 163840
    assert orc.bytes_per_token("fp4_mx_block16", 80, 8, 128) == 92160
    assert orc.bytes_per_token("nvfp4", 80, 8, 128) == 92160


def test_capacity_ratios(orc):
    for r in ROWS:
        if r[0] == "ratio":
            a, b, printed = r[1], r[2], float(r[3])
            ratio = orc.bytes_per_token(b, 80, 8, 128) / orc.bytes_per_token(a, 80, 8, 128)
            assert round(ratio, 2) == pytest.approx(printed, abs=1e-9)


def test_kv_size_grid(orc):
    bpt16 = orc.bytes_per_token("bf16", 80, 8, 128)
    bpt8 = orc.bytes_per_token("fp8_e4m3", 80, 8, 128)
    # 4-bit data without the scale bytes (the grid's INT4 column)
    bpt4 = orc.bytes_per_token("fp4_mx_block16", 80, 8, 128) * 4 // 4.5
    n = 0
    for r in ROWS:
        if r[0] == "grid":
            ctx, batch = int(r[1]), int(r[2])
            for bpt, printed in ((bpt16, r[3]), (bpt8, r[4]), (bpt4, r[5])):
                gib = bpt * ctx * batch / 2 ** 30
                assert abs(gib - float(printed)) <= 0.05 + 1e-12, (ctx, batch, gib, printed)
            n += 1
    assert n == 9


def test_fp8_doubles_token_capacity(orc):
    for r in ROWS:
        if r[0] == "capacity":
            L, H, D, bf16_tokens, fp8_tokens = map(int, r[2:7])
            budget = bf16_tokens * orc.bytes_per_token("bf16", L, H, D)
            assert budget // orc.bytes_per_token("fp8_e4m3", L, H, D) == fp8_tokens
