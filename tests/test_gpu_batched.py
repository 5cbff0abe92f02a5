"""GPU parity of the batched path (T > 8 tokens: routing, expert-sorted gather,
two grouped GEMMs on the tcgen05 tensor cores, fixed-order combine) against
the oracle.

Bar as for the decode path: top-k ids bit-exact, output max|d| <= 1e-2
rms(oracle) + 1e-5, bucketing equal to the oracle's stable counting sort,
repeated runs bitwise identical.  At the full layer size (T = 64, 256) every
token's ids, weights and output are compared with the oracle.
"""

from __future__ import annotations

import numpy as np
import pytest

import datagen
import oracle
from datagen import ACT_BF16, WFMT_BF16, WFMT_Q4B32, Shapes
from tests.cases import DECODE, draw_tokens, with_T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _layer(seed, shapes, wfmt=WFMT_BF16):
    return datagen.make_layer(seed, Shapes(1, shapes.H, shapes.E, shapes.top_k, shapes.I, shapes.Is), wfmt)


SMALL = [
        Shapes(T=9, H=256, E=8, top_k=2, I=128, Is=128),      # the smallest batch
        Shapes(T=40, H=512, E=16, top_k=4, I=256, Is=128),    # several row / column tiles, ragged groups
        Shapes(T=300, H=256, E=4, top_k=2, I=128, Is=256),    # groups and the shared expert past 128 slots
        Shapes(T=64, H=768, E=32, top_k=8, I=384, Is=256),    # three column-tile pairs, three row tiles
        Shapes(T=33, H=256, E=64, top_k=1, I=128, Is=128),    # top-1, most experts idle
]


@pytest.mark.parametrize("shapes", SMALL)
def test_batched_small(shapes):
    from tests.test_gpu_parity import check_case

    layer = _layer(4001, shapes)
    x, _ = draw_tokens(4001, layer, shapes.T, ACT_BF16)
    check_case(layer, x, ACT_BF16, str(shapes))


@pytest.mark.parametrize("shapes", SMALL)
def test_batched_small_q4(shapes):
    """4-bit block weights on the grouped GEMMs (fp16 operands)."""
    from tests.test_gpu_parity import check_case

    layer = _layer(4011, shapes, WFMT_Q4B32)
    x, _ = draw_tokens(4011, layer, shapes.T, ACT_BF16)
    check_case(layer, x, ACT_BF16, "q4 " + str(shapes))


@pytest.mark.parametrize("wfmt", [WFMT_BF16, WFMT_Q4B32])
@pytest.mark.parametrize("T", [3, 150])
def test_router_ties_take_lower_index(T, wfmt):
    """Zero router weights: every logit is exactly 0, so each token takes experts 0 .. k-1 (ties to the lower
    index) with p = 1/k.  At T = 150 (batched path) experts 0 .. 3 each hold 150 slots (three 64-slot chunks) and
    the other twelve are idle; at T = 3 the decode path takes the same decision."""
    from tests.test_gpu_parity import check_case

    shapes = Shapes(T=T, H=256, E=16, top_k=4, I=128, Is=128)
    layer = _layer(4021, shapes, wfmt)
    layer.router_w[...] = 0
    x, _ = draw_tokens(4021, layer, T, ACT_BF16, gap=-1.0)
    got, ref = check_case(layer, x, ACT_BF16, f"ties T={T} wfmt={wfmt}")
    np.testing.assert_array_equal(ref["ids"], np.tile(np.arange(4, dtype=ref["ids"].dtype), (T, 1)))


@pytest.mark.parametrize("wfmt", [WFMT_BF16, WFMT_Q4B32])
def test_batched_repeat_bitwise(wfmt):
    from tests.devlayer import DevLayer

    shapes = Shapes(T=40, H=512, E=16, top_k=4, I=256, Is=128)
    layer = _layer(4002, shapes, wfmt)
    x, _ = draw_tokens(4002, layer, shapes.T, ACT_BF16)
    dl = DevLayer(layer)
    a = dl.run(x, ACT_BF16)
    b = dl.run(x, ACT_BF16, ws_fill=0x5A)
    assert a["status"] == 0 and b["status"] == 0
    assert a["out"].tobytes() == b["out"].tobytes()
    assert a["ids"].tobytes() == b["ids"].tobytes()


@pytest.fixture(scope="module", params=[WFMT_BF16, WFMT_Q4B32], ids=["bf16", "q4"])
def full_layer(request):
    return datagen.make_layer(2024, DECODE, request.param)


@pytest.mark.parametrize("T", [64, 256])
def test_batched_full_size_every_token(full_layer, T):
    """The full layer (H=2048, E=128, top_k=8, I=768, Is=512) at T = 64 and 256: the ids, weights and output of
    every token against the oracle, and the bucketing against the oracle's bucketing of those ids."""
    from tests.devlayer import DevLayer, tolerance_ok

    s = with_T(DECODE, T)
    x, _ = draw_tokens(2024, full_layer, T, ACT_BF16, first_token=1000 + T)
    got = DevLayer(full_layer).run(x, ACT_BF16)
    assert got["status"] == 0
    ref = oracle.moe_ffn(s, ACT_BF16, full_layer.wfmt, x, full_layer.router_w, full_layer.expert_w,
                         full_layer.shexp_w, full_layer.shexp_gate_w)
    np.testing.assert_array_equal(got["ids"], ref["ids"])
    np.testing.assert_allclose(got["p"], ref["p"], rtol=1e-5, atol=1e-7)
    counts, offsets, perm, active = oracle.bucketing(ref["ids"], s.E)
    g_counts, g_offsets, g_perm, g_active = got["routing"]
    np.testing.assert_array_equal(g_counts, counts)
    np.testing.assert_array_equal(g_offsets, offsets)
    np.testing.assert_array_equal(g_perm, perm)
    np.testing.assert_array_equal(g_active, active)
    ok, err, rms = tolerance_ok(got["out"], ref["out"])
    assert ok, f"T={T}: max|d| = {err:.3e} > 1e-2 * rms({rms:.3e}) + 1e-5"
