"""The roofline numerator of bench.py: the algorithmic bytes of one layer call -- router rows, the shared-gate
vector, the unique routed experts, the shared expert, x (bf16) and out (fp32) -- worked by hand for the decode
workloads (H=2048, E=128, top_k=8, I=768, Is=512) and the three weight formats.  Each expert is three matrices of
I rows: bf16 rows of 2H bytes; 4-bit rows of H/32 blocks of 16 nibble bytes + a 2-byte fp16 scale (18H/32 bytes);
int8 rows of H codes + a 16-byte scale record."""

from __future__ import annotations

import pytest

pytest.importorskip("torch")

import bench  # noqa: E402
import datagen  # noqa: E402
from datagen import Shapes  # noqa: E402

H, E, I, IS = 2048, 128, 768, 512
FIXED = E * H * 2 + H * 2  # router rows + shared-gate vector


@pytest.mark.parametrize(
    "wfmt,row_bytes",
    [(datagen.WFMT_BF16, 2 * H), (datagen.WFMT_Q4B32, H // 32 * 18), (datagen.WFMT_I8, H + 16)],
)
def test_expert_bytes_by_format(wfmt, row_bytes):
    assert datagen.expert_bytes(wfmt, H, I) == 3 * I * row_bytes
    assert datagen.expert_bytes(wfmt, H, IS) == 3 * IS * row_bytes


def test_decode_bf16_one_token():
    # 524,288 + 4,096 + 8 x 9,437,184 + 6,291,456 + 4,096 + 8,192
    assert bench.algorithmic_bytes(Shapes(1, H, E, 8, I, IS), datagen.WFMT_BF16, 8.0) == 82_329_600


def test_decode_q4_one_token():
    # 524,288 + 4,096 + 8 x 2,654,208 + 1,769,472 + 4,096 + 8,192
    assert bench.algorithmic_bytes(Shapes(1, H, E, 8, I, IS), datagen.WFMT_Q4B32, 8.0) == 23_543_808


def test_decode_i8_one_token():
    # 524,288 + 4,096 + 8 x 4,755,456 + 3,170,304 + 4,096 + 8,192
    assert bench.algorithmic_bytes(Shapes(1, H, E, 8, I, IS), datagen.WFMT_I8, 8.0) == 41_754_624


def test_bytes_grow_with_unique_experts_and_tokens():
    s8 = Shapes(8, H, E, 8, I, IS)
    eb = 3 * I * 2 * H
    a = bench.algorithmic_bytes(s8, datagen.WFMT_BF16, 40.0)
    b = bench.algorithmic_bytes(s8, datagen.WFMT_BF16, 41.0)
    assert b - a == eb
    assert a == FIXED + 40 * eb + 3 * IS * 2 * H + 8 * H * 2 + 8 * H * 4
