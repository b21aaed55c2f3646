"""Accounting helper against the counts printed on the pages (tests/golden/accounting_pins.txt)."""
import os

import pytest

from compressed_kv_cache_lrkv_gb300 import accounting as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accounting_pins.txt")


def _rows():
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        kind, params, expected, cite = (s.strip() for s in line.split("|"))
        kv = {k: int(v) for k, v in (p.split("=") for p in params.split())}
        yield kind, kv, float(expected), cite


@pytest.mark.parametrize("row", list(_rows()), ids=lambda r: f"{r[0]}-{r[1]}")
def test_page_counts(row):
    kind, kv, expected, cite = row
    # printed percentages agree to half a unit of their last printed decimal
    if kind == "ratio":
        assert abs(100 * A.cache_ratio(kv["H"], kv["d_h"], kv["r"]) - expected) <= 0.005 + 1e-12, cite
    elif kind == "ratio1":
        assert abs(100 * A.cache_ratio(kv["H"], kv["d_h"], kv["r"]) - expected) <= 0.05 + 1e-12, cite
    elif kind == "lrkv_elements":
        assert A.lrkv_cache_elements(kv["H"], kv["d_h"], kv["r"]) == expected, cite
    elif kind == "mha_elements":
        assert A.mha_cache_elements(kv["H"], kv["d_h"]) == expected, cite
    elif kind == "mha_elements_layers":
        assert A.mha_cache_elements(kv["H"], kv["d_h"], kv["layers"]) == expected, cite
    elif kind == "mha_bytes_layers":
        assert A.mha_cache_elements(kv["H"], kv["d_h"], kv["layers"]) * A.BF16_BYTES == expected, cite
    elif kind == "gqa_elements_layers":
        assert A.gqa_cache_elements(kv["groups"], kv["d_h"], kv["layers"]) == expected, cite
    elif kind == "mqa_elements_layers":
        assert A.mqa_cache_elements(kv["d_h"], kv["layers"]) == expected, cite
    elif kind == "mla_elements_layers":
        assert A.mla_cache_elements(kv["d_c"], kv["d_h_r"], kv["layers"]) == expected, cite
    else:
        raise AssertionError(kind)


def test_limits_of_the_rank():
    # r = 0 is MQA-style sharing (ratio 1/H); r = d_h gives 1 + 1/H (Eq. (9) frame).
    for H in (6, 12, 32):
        assert A.lrkv_cache_elements(H, 128, 0) == A.mqa_cache_elements(128)
        assert abs(A.cache_ratio(H, 128, 128) - (1 + 1 / H)) < 1e-15


def test_kv_parameter_counts():
    # Eq. (10): with r = d_h and no shared part LRKV has the MHA count plus the B factors.
    d, d_h, H = 768, 128, 6
    assert A.kv_params_mha(d, d_h, H) == 2 * H * d * d_h
    assert A.kv_params_lrkv(d, d_h, H, 0) == 2 * d * d_h
    assert A.kv_params_lrkv(d, d_h, H, d_h) - 2 * d * d_h == A.kv_params_mha(d, d_h, H) + 2 * H * d_h * d_h


def test_workload_byte_counts():
    # Decode bytes of the long-context workload at the mean length, and the page sizes.
    assert A.page_bytes(32, 128, 32) == 64 * 4608
    assert A.page_bytes(128, 128, 16) == 64 * 8704
    assert A.decode_algorithmic_bytes(8, 64, 8, [256]) == 149504
    assert A.decode_algorithmic_bytes(8, 64, 16, [2048] * 16, layers=12) == 302776320
    assert A.decode_algorithmic_bytes(128, 128, 16, [8192] * 8) == 571998208
    assert A.append_flops(8192, 4096, 32, 128, 16) == 85899345920
    assert A.prefill_flops(2, 4096, 32, 128, 16) - 4 * 2 * 4096 * 32 * 128 * 16 == 4 * 144 * 32 * 2 * 4096 * 4097 // 2
    # the positional key adds its 64 columns to the logit side only; absorbed weights drop the
    # two projections
    assert (A.prefill_flops(2, 4096, 32, 128, 16, d_rope=64) - A.prefill_flops(2, 4096, 32, 128, 16)
            == 2 * 64 * 32 * 2 * 4096 * 4097 // 2)
    assert (A.prefill_flops(2, 4096, 32, 128, 16) - A.prefill_flops(2, 4096, 32, 128, 16, absorbed=True)
            == 4 * 2 * 4096 * 32 * 128 * 16)
