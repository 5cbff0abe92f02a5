"""GPU parity of the int8 weight format: int8 rows with an fp32 row scale and
an int8 activation (the int8 linear, sd.linear_i8.v1, of "ggml operator
extensions", section "sd.cpp integration": float(int32_dot(W, X)) * X_scale
* W_scale), with the SwiGLU epilogue, on the decode path: the tensor-core
loop (H = 2048, bf16 x or the block form) and the general loop (other
shapes, fp32 x).

The activation quantiser and the gate/up projections are the same fp32
operations on both sides, so the GPU's g and u equal the oracle's bit for
bit; what is left is the fp32 arithmetic of h, the down projection and the
sums, about 1e-6 of rms(out).  The bar here is therefore tighter than the
layer's general one: max|d| <= 1e-4 rms(oracle) + 1e-6, on top of bit-exact
ids.  A quantiser that rounded halves to even, or a scale applied in another
order, moves g by ~1 % on the tie inputs below and fails it.
"""

from __future__ import annotations

import numpy as np
import pytest

import datagen
import oracle
from datagen import ACT_BF16, ACT_F32, WFMT_I8, Shapes
from tests.cases import DECODE, NEAR_TIE_GAP, draw_tokens, kth_gap, with_T, x_as_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

I8_REL = 1e-4
I8_ABS = 1e-6


def _tight(got, ref):
    ref = ref.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    return err <= I8_REL * rms + I8_ABS, err, rms


def check_i8(layer, x, act, label, **kw):
    from tests.devlayer import DevLayer

    dl = DevLayer(layer)
    s = with_T(layer.shapes, x.shape[0])
    ref = oracle.moe_ffn(s, act, WFMT_I8, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w)
    got = dl.run(x, act, **kw)
    assert got["status"] == 0, f"{label}: device status {got['status']}"
    np.testing.assert_array_equal(got["ids"], ref["ids"], err_msg=f"{label}: top-k ids")
    np.testing.assert_allclose(got["p"], ref["p"], rtol=1e-5, atol=1e-7, err_msg=f"{label}: top-k weights")
    ok, err, rms = _tight(got["out"], ref["out"])
    print(f"\n{label}: max|d| {err:.3e}, rms {rms:.3e}, max|d|/rms {err / max(rms, 1e-30):.2e}")
    assert ok, f"{label}: max|d| = {err:.3e} > {I8_REL} * rms({rms:.3e}) + {I8_ABS}"
    counts, offsets, perm, active = oracle.bucketing(ref["ids"], s.E)
    g_counts, g_offsets, g_perm, g_active = got["routing"]
    np.testing.assert_array_equal(g_counts, counts)
    np.testing.assert_array_equal(g_offsets, offsets)
    np.testing.assert_array_equal(g_perm, perm)
    np.testing.assert_array_equal(g_active, active)
    return got, ref


@pytest.mark.parametrize(
    "shapes,act",
    [
        (Shapes(T=1, H=272, E=8, top_k=2, I=130, Is=70), ACT_BF16),   # ragged stages, 34 of 256 column chunks
        (Shapes(T=3, H=528, E=5, top_k=3, I=40, Is=24), ACT_F32),     # fp32 x, ragged
        (Shapes(T=8, H=1024, E=64, top_k=6, I=320, Is=256), ACT_BF16),
        (Shapes(T=5, H=128, E=4, top_k=4, I=17, Is=9), ACT_F32),      # every expert selected, I < rows of a stage
        (Shapes(T=2, H=2320, E=16, top_k=4, I=64, Is=48), ACT_BF16),  # H > 2048: two column chunks per thread
        (Shapes(T=1, H=4096, E=8, top_k=2, I=40, Is=24), ACT_F32),    # H at its maximum
        (Shapes(T=3, H=2048, E=32, top_k=4, I=96, Is=40), ACT_F32),   # H = 2048 with fp32 x: the general loop
        (Shapes(T=1, H=2048, E=16, top_k=4, I=130, Is=70), ACT_BF16),  # tensor-core loop, ragged 8-row stages
        (Shapes(T=5, H=2048, E=24, top_k=3, I=20, Is=12), ACT_BF16),   # tensor-core loop, T=5, I < 3 stages
    ],
)
def test_i8_small_and_ragged(shapes, act):
    layer = datagen.make_layer(7100 + shapes.H + shapes.T, shapes, WFMT_I8)
    x, _ = draw_tokens(7100 + shapes.H, layer, shapes.T, act)
    check_i8(layer, x, act, f"i8 {shapes}")


@pytest.fixture(scope="module")
def decode_i8_layer():
    return datagen.make_layer(2026, DECODE, WFMT_I8)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_i8_full_size(decode_i8_layer, T):
    x, _ = draw_tokens(2026, decode_i8_layer, T, ACT_BF16, first_token=10 * T)
    check_i8(decode_i8_layer, x, ACT_BF16, f"decode i8 T={T}")


def test_i8_activation_rounding_ties(decode_i8_layer):
    """Every code of x sits on a rounding tie: max|x| = 127 gives x_scale = 1 exactly, and the other elements are
    k + 1/2 (exact in bf16 for |k| < 127), so x / x_scale is a half-integer and the quantiser's rounding rule (half
    away from zero) decides every code."""
    layer = decode_i8_layer
    H = DECODE.H
    rng = np.random.default_rng(2027)
    for sub in range(16):
        v = rng.integers(-120, 120, size=H).astype(np.float32) + 0.5
        v[(7 * sub) % H] = 127.0 if sub % 2 == 0 else -127.0
        x = datagen.f32_to_bf16(v).reshape(1, H)
        assert np.array_equal(datagen.bf16_to_f32(x), v.reshape(1, H))
        lg = oracle.router_logits(layer.router_w, DECODE.E, H, x_as_f64(x, ACT_BF16)[0])
        if kth_gap(lg, DECODE.top_k) >= NEAR_TIE_GAP:
            break
    else:
        pytest.fail("no tie input without a router near-tie")
    qx, xs = oracle.quantize_i8(x_as_f64(x, ACT_BF16)[0])
    assert xs == 1.0 and np.all(np.abs(qx[np.abs(v) < 127]) == np.floor(np.abs(v[np.abs(v) < 127])) + 1)
    check_i8(layer, x, ACT_BF16, "i8 rounding ties")


def test_i8_zero_activation():
    """x = 0: x_scale = 0, every code 0, so g = u = 0 and the output is exactly zero; the router logits are all
    zero and the top-k takes the lowest expert indices."""
    from tests.devlayer import DevLayer

    s = Shapes(T=2, H=272, E=8, top_k=3, I=40, Is=24)
    layer = datagen.make_layer(7200, s, WFMT_I8)
    x = np.zeros((2, s.H), np.float32)
    got = DevLayer(layer).run(x, ACT_F32)
    assert got["status"] == 0
    assert np.all(got["out"] == 0.0)
    np.testing.assert_array_equal(got["ids"], np.tile(np.arange(3, dtype=np.int32), (2, 1)))
    ref = oracle.moe_ffn(s, ACT_F32, WFMT_I8, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w)
    np.testing.assert_array_equal(got["ids"], ref["ids"])
    assert np.all(ref["out"] == 0.0)


@pytest.mark.parametrize("T", [1, 8])
def test_decode_i8_bitwise_repeat(decode_i8_layer, T):
    """Two runs on differently filled workspaces and streams give the same bytes."""
    import fusion_backend_gb300 as fb
    from tests.devlayer import DevLayer

    dl = DevLayer(decode_i8_layer)
    s = with_T(DECODE, T)
    x = np.stack([datagen.token_x(2026, 500 + t, DECODE.H, ACT_BF16) for t in range(T)])
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    plan, ws_bytes = fb.moe_ffn_prepare(s, ACT_BF16, WFMT_I8)
    res = []
    for fill, off in ((0xA5, 0), (0x5A, 1280)):
        buf = torch.full((ws_bytes + 4096,), fill, dtype=torch.uint8, device="cuda")
        ws = buf[off : off + ws_bytes]
        stream = torch.cuda.Stream()
        out = torch.full((T, DECODE.H), float("nan"), dtype=torch.float32, device="cuda")
        ids = torch.full((T, DECODE.top_k), -1, dtype=torch.int32, device="cuda")
        stream.wait_stream(torch.cuda.current_stream())
        fb.moe_ffn_execute_ex(plan, ws, xd, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, out, ids, None,
                              stream=stream)
        stream.synchronize()
        assert fb.moe_ffn_read_status(plan, ws, stream) == 0
        res.append((out.cpu().numpy().tobytes(), ids.cpu().numpy().tobytes()))
    fb.moe_ffn_destroy(plan)
    assert res[0] == res[1]


def test_i8_block_form_full_size():
    """The pre-norm block form with int8 weights at full size, two layers teacher-forced: the normalised input
    xn = bf16(RMSNorm(x_res)) is quantised per token inside the kernel."""
    import fusion_backend_gb300 as fb
    from tests.devlayer import DevLayer

    s1 = with_T(DECODE, 1)
    m = fb.MoeFFN(s1, ACT_BF16, WFMT_I8)
    xd = torch.from_numpy(datagen.normal_f32(7300, 7, DECODE.H).reshape(1, DECODE.H) * 2.0).cuda()
    ids = torch.full((1, DECODE.top_k), -1, dtype=torch.int32, device="cuda")
    for l in range(2):
        L = datagen.make_layer(7300 + l, s1, WFMT_I8)
        D = DevLayer(L)
        x_in = xd.cpu().numpy()
        m.block(xd, D.router_w, D.expert_w, D.shexp_w, D.gate_w, eps=1e-6, topk_ids=ids)
        torch.cuda.synchronize()
        assert m.status() == 0
        new_ref, ids_ref, xn_ref = oracle.block_step(s1, WFMT_I8, x_in, L.router_w, L.expert_w, L.shexp_w,
                                                     L.shexp_gate_w, eps=1e-6)
        lg = oracle.router_logits(L.router_w, DECODE.E, DECODE.H, datagen.bf16_to_f32(xn_ref[0]).astype(np.float64))
        if kth_gap(lg, DECODE.top_k) >= NEAR_TIE_GAP:
            np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
        ok, err, rms = _tight(xd.cpu().numpy() - x_in, new_ref - x_in)
        assert ok, f"layer {l}: max|d| {err:.3e} > {I8_REL} * rms({rms:.3e}) + {I8_ABS}"
        del D
    m.close()
