"""GPU parity: the CUDA path against the oracle on the same seeded inputs.

Bar: top-k ids bit-exact; output max|d| <= 1e-2 rms(oracle) + 1e-5; softmax
weights within 1e-5 relative; bucketing equal to the oracle's stable counting
sort; repeated runs bitwise identical.
"""

from __future__ import annotations

import numpy as np
import pytest

import datagen
import oracle
from datagen import ACT_BF16, ACT_F32, WFMT_BF16, WFMT_Q4B32, Shapes
from tests.cases import DECODE, SMALL_Q4, TINY, draw_tokens, with_T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev():
    from tests.devlayer import DevLayer, tolerance_ok

    return DevLayer, tolerance_ok


def check_case(layer, x, act, label, **kw):
    DevLayer, tolerance_ok = _dev()
    dl = DevLayer(layer)
    s = with_T(layer.shapes, x.shape[0])
    ref = oracle.moe_ffn(s, act, layer.wfmt, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w)
    got = dl.run(x, act, **kw)
    assert got["status"] == 0, f"{label}: device status {got['status']}"
    np.testing.assert_array_equal(got["ids"], ref["ids"], err_msg=f"{label}: top-k ids")
    np.testing.assert_allclose(got["p"], ref["p"], rtol=1e-5, atol=1e-7, err_msg=f"{label}: top-k weights")
    ok, err, rms = tolerance_ok(got["out"], ref["out"])
    assert ok, f"{label}: max|d| = {err:.3e} > 1e-2 * rms({rms:.3e}) + 1e-5"
    counts, offsets, perm, active = oracle.bucketing(ref["ids"], s.E)
    g_counts, g_offsets, g_perm, g_active = got["routing"]
    np.testing.assert_array_equal(g_counts, counts)
    np.testing.assert_array_equal(g_offsets, offsets)
    np.testing.assert_array_equal(g_perm, perm)
    np.testing.assert_array_equal(g_active, active)
    return got, ref


@pytest.mark.parametrize("T", [1, 2, 3, 8])
def test_tiny_layer_fp32_x(T):
    layer = datagen.make_layer(1001, TINY, WFMT_BF16)
    x, _ = draw_tokens(1001, layer, T, ACT_F32)
    check_case(layer, x, ACT_F32, f"tiny T={T}")


def test_tiny_layer_bf16_x_and_repeat_bitwise():
    DevLayer, _ = _dev()
    layer = datagen.make_layer(1002, TINY, WFMT_BF16)
    x, _ = draw_tokens(1002, layer, 4, ACT_BF16)
    got, _ = check_case(layer, x, ACT_BF16, "tiny bf16")
    dl = DevLayer(layer)
    again = dl.run(x, ACT_BF16, ws_fill=0xA5)
    assert got["out"].tobytes() == again["out"].tobytes()
    assert got["ids"].tobytes() == again["ids"].tobytes()
    assert got["p"].tobytes() == again["p"].tobytes()


@pytest.mark.parametrize(
    "shapes",
    [
        Shapes(T=3, H=264, E=5, top_k=3, I=136, Is=72),   # ragged segments (H, I, Is not multiples of 256)
        Shapes(T=2, H=512, E=1, top_k=1, I=64, Is=8),     # a single expert
        Shapes(T=5, H=128, E=4, top_k=4, I=40, Is=16),    # every expert selected
        Shapes(T=8, H=1024, E=64, top_k=6, I=320, Is=256),
        Shapes(T=7, H=776, E=33, top_k=32, I=24, Is=48),  # top_k = 32, E not a multiple of 32
        Shapes(T=1, H=2304, E=16, top_k=4, I=256, Is=128),  # H > 2048: the general kernel
        Shapes(T=3, H=3072, E=8, top_k=2, I=64, Is=64),    # H > 2048, several tokens
    ],
)
def test_ragged_and_degenerate_shapes(shapes):
    layer = datagen.make_layer(1003, Shapes(1, shapes.H, shapes.E, shapes.top_k, shapes.I, shapes.Is), WFMT_BF16)
    gap = 1e-3 if shapes.top_k < shapes.E else 0.0
    x, _ = draw_tokens(1003, layer, shapes.T, ACT_BF16, gap=gap)
    check_case(layer, x, ACT_BF16, str(shapes))


def test_out_aliases_x():
    layer = datagen.make_layer(1004, TINY, WFMT_BF16)
    x, _ = draw_tokens(1004, layer, 2, ACT_F32)
    check_case(layer, x, ACT_F32, "alias", out_alias=True)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_small_q4_layer(T):
    layer = datagen.make_layer(1005, SMALL_Q4, WFMT_Q4B32)
    x, _ = draw_tokens(1005, layer, T, ACT_BF16)
    check_case(layer, x, ACT_BF16, f"small q4 T={T}")


def test_small_q4_layer_fp32_x_general_kernel():
    layer = datagen.make_layer(1008, SMALL_Q4, WFMT_Q4B32)
    x, _ = draw_tokens(1008, layer, 3, ACT_F32)
    check_case(layer, x, ACT_F32, "small q4 fp32 x")


@pytest.fixture(scope="module")
def decode_bf16_layer():
    return datagen.make_layer(2024, DECODE, WFMT_BF16)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_bf16_full_size(decode_bf16_layer, T):
    x, _ = draw_tokens(2024, decode_bf16_layer, T, ACT_BF16, first_token=10 * T)
    check_case(decode_bf16_layer, x, ACT_BF16, f"decode bf16 T={T}")


@pytest.fixture(scope="module")
def decode_q4_layer():
    return datagen.make_layer(2025, DECODE, WFMT_Q4B32)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_q4_full_size(decode_q4_layer, T):
    x, _ = draw_tokens(2025, decode_q4_layer, T, ACT_BF16, first_token=10 * T)
    check_case(decode_q4_layer, x, ACT_BF16, f"decode q4 T={T}")


def test_block_form_matches_oracle_teacher_forced():
    """Pre-norm block form over a few layers; ids compared with the oracle fed the GPU's layer input."""
    import fusion_backend_gb300 as fb
    from tests.devlayer import DevLayer, tolerance_ok

    shapes = SMALL_Q4
    x_res = datagen.normal_f32(77, 1, shapes.H).reshape(1, shapes.H)
    xd = torch.from_numpy(x_res.copy()).cuda()
    m = fb.MoeFFN(shapes, ACT_BF16, WFMT_Q4B32)
    for l in range(4):
        layer = datagen.make_layer(3000 + l, shapes, WFMT_Q4B32)
        dl = DevLayer(layer)
        x_in = xd.cpu().numpy()
        ids = torch.full((1, shapes.top_k), -1, dtype=torch.int32, device="cuda")
        m.block(xd, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, eps=1e-6, topk_ids=ids)
        torch.cuda.synchronize()
        assert m.status() == 0
        new, ref_ids, _ = oracle.block_step(shapes, WFMT_Q4B32, x_in, layer.router_w, layer.expert_w, layer.shexp_w,
                                            layer.shexp_gate_w)
        np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
        ok, err, rms = tolerance_ok(xd.cpu().numpy() - x_in, new - x_in)
        assert ok, f"layer {l}: {err} vs rms {rms}"
    m.close()


def test_cuda_graph_capture_and_replay():
    import fusion_backend_gb300 as fb
    from tests.devlayer import DevLayer

    layer = datagen.make_layer(1006, TINY, WFMT_BF16)
    dl = DevLayer(layer)
    x, _ = draw_tokens(1006, layer, 2, ACT_F32)
    s = with_T(TINY, 2)
    m = fb.MoeFFN(s, ACT_F32, WFMT_BF16)
    xd = torch.from_numpy(x).cuda()
    out = torch.zeros((2, s.H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        m(xd, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, out=out)  # warm-up outside capture
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        m(xd, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    xd.copy_(torch.from_numpy(draw_tokens(1007, layer, 2, ACT_F32)[0]).cuda())
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.moe_ffn(s, ACT_F32, WFMT_BF16, xd.cpu().numpy(), layer.router_w, layer.expert_w, layer.shexp_w,
                         layer.shexp_gate_w)
    from tests.devlayer import tolerance_ok

    assert tolerance_ok(out.cpu().numpy(), ref["out"])[0]
    m.close()
