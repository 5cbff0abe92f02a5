"""Pins of the oracle against things other than itself.

Each check below is chosen so that a plausible slip in the oracle (a dropped
term, a wrong index or sign, a transposed matrix, a wrong tie rule, a wrong
nibble order) fails at least one of them:

* dense brute force: every expert evaluated with numpy/torch fp64 matmuls,
  full softmax over all experts, non-top-k weights zeroed and renormalised;
* one-hot router: the layer reduces to a single dense SwiGLU FFN plus the
  gated shared expert, and the tie rule picks the lowest other index;
* zero shared gate: shared down weights all zero, or a gate vector driving
  sigmoid to 0, must both give the routed-only output;
* g = 0 gives s = 0.5 exactly;
* token independence, expert-permutation invariance;
* bucketing equals Python's stable sort;
* the fp16 decoder on known bit patterns; the 4-bit nibble order.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import datagen
import oracle
from datagen import ACT_BF16, ACT_F32, WFMT_BF16, WFMT_Q4B32
from tests.cases import SMALL_Q4, TINY, draw_tokens, with_T, x_as_f64

torch.set_num_threads(4)

# ----------------------------------------------------------------------------
# Independent decoding of the stored formats (numpy's own fp16 and bit views)


def np_matrix(buf: np.ndarray, wfmt: int, rows: int, cols: int) -> np.ndarray:
    if wfmt == WFMT_BF16:
        return datagen.bf16_to_f32(buf.view(np.uint16).reshape(rows, cols)).astype(np.float64)
    b = buf.reshape(rows, cols * 9 // 16)
    nib = b[:, : cols // 2]
    q = np.empty((rows, cols), np.int64)
    q[:, 0::2] = nib & 0x0F
    q[:, 1::2] = nib >> 4
    d = np.ascontiguousarray(b[:, cols // 2 :]).view("<f2").astype(np.float64)  # [rows, cols/32]
    return (q - 8) * np.repeat(d, 32, axis=1)


def np_layer(layer: datagen.Layer):
    s, f = layer.shapes, layer.wfmt
    H, E, I, Is = s.H, s.E, s.I, s.Is
    eb = datagen.expert_bytes(f, H, I)
    gu = datagen.matrix_bytes(f, I, H)
    experts = []
    for e in range(E):
        blk = layer.expert_w[e * eb : (e + 1) * eb]
        # the third matrix is stored transposed ([I,H]); Wd = its transpose
        experts.append((np_matrix(blk[:gu], f, I, H), np_matrix(blk[gu : 2 * gu], f, I, H),
                        np_matrix(blk[2 * gu :], f, I, H).T.copy()))
    sgu = datagen.matrix_bytes(f, Is, H)
    sh = (np_matrix(layer.shexp_w[:sgu], f, Is, H), np_matrix(layer.shexp_w[sgu : 2 * sgu], f, Is, H),
          np_matrix(layer.shexp_w[2 * sgu :], f, Is, H).T.copy())
    router = datagen.bf16_to_f32(layer.router_w.reshape(E, H)).astype(np.float64)
    gvec = datagen.bf16_to_f32(layer.shexp_gate_w).astype(np.float64)
    return router, gvec, experts, sh


def torch_ffn(W, x):
    """SwiGLU FFN with torch fp64 library ops: down(silu(gate x) * (up x))."""
    Wg, Wu, Wd = (torch.from_numpy(w) for w in W)
    xt = torch.from_numpy(x)
    return (Wd @ (torch.nn.functional.silu(Wg @ xt) * (Wu @ xt))).numpy()


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def run_oracle(layer, x, act):
    s = with_T(layer.shapes, x.shape[0])
    return oracle.moe_ffn(s, act, layer.wfmt, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w)


def order_desc_then_index(logits: np.ndarray) -> np.ndarray:
    """Python's stable sort on (-logit, index): the tie rule stated by the workload."""
    return np.array(sorted(range(logits.size), key=lambda e: (-float(logits[e]), e)), np.int64)


# ----------------------------------------------------------------------------


@pytest.fixture(scope="module")
def tiny_layer():
    return datagen.make_layer(101, TINY, WFMT_BF16)


@pytest.mark.parametrize("act", [ACT_F32, ACT_BF16])
def test_dense_bruteforce_full_softmax(tiny_layer, act):
    """Every expert evaluated densely; full softmax; zero the non-top-k; renormalise."""
    layer = tiny_layer
    s = layer.shapes
    x, _ = draw_tokens(5, layer, 4, act)
    res = run_oracle(layer, x, act)
    router, gvec, experts, sh = np_layer(layer)
    for t in range(x.shape[0]):
        xt = x_as_f64(x[t], act)
        logit64 = router @ xt
        logit32 = logit64.astype(np.float32)
        np.testing.assert_array_equal(res["logits"][t], logit32)
        order = order_desc_then_index(logit32)
        top = order[: s.top_k]
        np.testing.assert_array_equal(res["ids"][t], top)
        full = torch.softmax(torch.from_numpy(logit32.astype(np.float64)), 0).numpy()
        w = np.zeros(s.E)
        w[top] = full[top]
        w /= w.sum()
        dense = sum(w[e] * torch_ffn(experts[e], xt) for e in range(s.E))
        sg = 1.0 / (1.0 + np.exp(-(gvec @ xt)))
        ref = dense + sg * torch_ffn(sh, xt)
        assert rel_err(res["out"][t], ref) < 1e-6  # fp32 output vs fp64 reference
        np.testing.assert_allclose(res["p"][t], w[top], rtol=1e-6)
        assert abs(float(np.sum(res["p"][t].astype(np.float64))) - 1.0) < 1e-6
        assert np.all(np.diff(res["p"][t]) <= 0)
        assert abs(res["s"][t] - sg) < 1e-7


def test_expert_ffn_matches_torch(tiny_layer):
    layer = tiny_layer
    s = layer.shapes
    _, _, experts, _ = np_layer(layer)
    eb = datagen.expert_bytes(WFMT_BF16, s.H, s.I)
    x = datagen.normal_f32(9, 9, s.H).astype(np.float64)
    for e in (0, 3, s.E - 1):
        y = oracle.swiglu_ffn(layer.expert_w[e * eb : (e + 1) * eb], WFMT_BF16, s.H, s.I, x)
        assert rel_err(y, torch_ffn(experts[e], x)) < 1e-12


def test_expert_ffn_q4_matches_torch():
    layer = datagen.make_layer(7, SMALL_Q4, WFMT_Q4B32)
    s = layer.shapes
    _, _, experts, sh = np_layer(layer)
    eb = datagen.expert_bytes(WFMT_Q4B32, s.H, s.I)
    x = datagen.normal_f32(9, 10, s.H).astype(np.float64)
    for e in (0, s.E - 1):
        y = oracle.swiglu_ffn(layer.expert_w[e * eb : (e + 1) * eb], WFMT_Q4B32, s.H, s.I, x)
        assert rel_err(y, torch_ffn(experts[e], x)) < 1e-12
    y = oracle.swiglu_ffn(layer.shexp_w, WFMT_Q4B32, s.H, s.Is, x)
    assert rel_err(y, torch_ffn(sh, x)) < 1e-12


@pytest.mark.parametrize("j", [0, 5])
def test_one_hot_router_reduces_to_dense_ffn(tiny_layer, j):
    """Router row j = bf16(alpha*sign(x)), other rows zero: ids = (j, lowest other index), p = (1, ~0)."""
    layer = tiny_layer
    s = layer.shapes
    x = datagen.token_x(77, 0, s.H, ACT_F32)
    alpha = 256.0 / np.sum(np.abs(x.astype(np.float64)))
    router = np.zeros((s.E, s.H), np.float32)
    router[j] = alpha * np.sign(x)
    rw = datagen.f32_to_bf16(router).reshape(-1)
    onehot = datagen.Layer(s, WFMT_BF16, rw, layer.shexp_gate_w, layer.expert_w, layer.shexp_w)
    res = run_oracle(onehot, x[None, :], ACT_F32)
    expect_second = 0 if j != 0 else 1
    np.testing.assert_array_equal(res["ids"][0], [j, expect_second])
    assert res["logits"][0][j] >= 200.0
    assert res["p"][0][0] == 1.0 and res["p"][0][1] == 0.0
    _, gvec, experts, sh = np_layer(onehot)
    xt = x.astype(np.float64)
    sg = 1.0 / (1.0 + np.exp(-(gvec @ xt)))
    ref = torch_ffn(experts[j], xt) + sg * torch_ffn(sh, xt)
    assert rel_err(res["out"][0], ref) < 1e-6


def test_exact_tie_goes_to_lower_index(tiny_layer):
    """Duplicate router rows 2 and 6 and make them the largest: 2 must rank first."""
    layer = tiny_layer
    s = layer.shapes
    x = datagen.token_x(78, 0, s.H, ACT_F32)
    router = datagen.bf16_to_f32(layer.router_w.reshape(s.E, s.H)).copy()
    row = (0.05 * np.sign(x)).astype(np.float32)
    router[2] = row
    router[6] = row
    rw = datagen.f32_to_bf16(router).reshape(-1)
    tie = datagen.Layer(s, WFMT_BF16, rw, layer.shexp_gate_w, layer.expert_w, layer.shexp_w)
    res = run_oracle(tie, x[None, :], ACT_F32)
    assert res["logits"][0][2] == res["logits"][0][6]
    np.testing.assert_array_equal(res["ids"][0], [2, 6])
    assert res["p"][0][0] == res["p"][0][1] == 0.5


def test_zero_shared_gate_two_ways(tiny_layer):
    """(i) shared down = 0 and (ii) g = -c x/|x|^2 (sigmoid -> 0) both give routed-only output."""
    layer = tiny_layer
    s = layer.shapes
    x, _ = draw_tokens(11, layer, 1, ACT_F32)
    xt = x[0].astype(np.float64)
    sgu = datagen.matrix_bytes(WFMT_BF16, s.Is, s.H)
    sh_zero = layer.shexp_w.copy()
    sh_zero[2 * sgu :] = 0
    l1 = datagen.Layer(s, WFMT_BF16, layer.router_w, layer.shexp_gate_w, layer.expert_w, sh_zero)
    g = (-256.0 * xt / np.dot(xt, xt)).astype(np.float32)
    l2 = datagen.Layer(s, WFMT_BF16, layer.router_w, datagen.f32_to_bf16(g), layer.expert_w, layer.shexp_w)
    r1 = run_oracle(l1, x, ACT_F32)
    r2 = run_oracle(l2, x, ACT_F32)
    assert r2["s"][0] == 0.0
    np.testing.assert_array_equal(r1["out"], r2["out"])
    router, _, experts, _ = np_layer(layer)
    logit32 = (router @ xt).astype(np.float32)
    top = order_desc_then_index(logit32)[: s.top_k]
    z = np.exp(logit32[top].astype(np.float64) - logit32[top[0]])
    p = z / z.sum()
    routed = sum(p[i] * torch_ffn(experts[e], xt) for i, e in enumerate(top))
    assert rel_err(r1["out"][0], routed) < 1e-6


def test_gate_zero_gives_half(tiny_layer):
    layer = tiny_layer
    s = layer.shapes
    x, _ = draw_tokens(12, layer, 1, ACT_F32)
    xt = x[0].astype(np.float64)
    l0 = datagen.Layer(s, WFMT_BF16, layer.router_w, np.zeros(s.H, np.uint16), layer.expert_w, layer.shexp_w)
    r = run_oracle(l0, x, ACT_F32)
    assert r["s"][0] == 0.5
    router, _, experts, sh = np_layer(layer)
    logit32 = (router @ xt).astype(np.float32)
    top = order_desc_then_index(logit32)[: s.top_k]
    z = np.exp(logit32[top].astype(np.float64) - logit32[top[0]])
    p = z / z.sum()
    ref = sum(p[i] * torch_ffn(experts[e], xt) for i, e in enumerate(top)) + 0.5 * torch_ffn(sh, xt)
    assert rel_err(r["out"][0], ref) < 1e-6


def test_tokens_are_independent(tiny_layer):
    layer = tiny_layer
    x, _ = draw_tokens(13, layer, 8, ACT_F32)
    full = run_oracle(layer, x, ACT_F32)
    for t in range(8):
        one = run_oracle(layer, x[t : t + 1], ACT_F32)
        np.testing.assert_array_equal(one["out"][0], full["out"][t])
        np.testing.assert_array_equal(one["ids"][0], full["ids"][t])


def test_thread_count_does_not_change_bits(tiny_layer):
    layer = tiny_layer
    s = with_T(layer.shapes, 4)
    x, _ = draw_tokens(14, layer, 4, ACT_F32)
    a = oracle.moe_ffn(s, ACT_F32, WFMT_BF16, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w, threads=1)
    b = oracle.moe_ffn(s, ACT_F32, WFMT_BF16, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w, threads=7)
    np.testing.assert_array_equal(a["out"], b["out"])


@pytest.mark.parametrize("wfmt", [WFMT_BF16, WFMT_Q4B32])
@pytest.mark.parametrize("threads", [1, 5])
def test_layer_split_over_rows_equals_whole_ffns(wfmt, threads):
    """The layer evaluates its FFNs in row and column tasks spread over threads; with top_k = 1 (p = 1) and the
    shared down projection zeroed (shared term exactly 0) each output row must equal, bit for bit, one whole
    SwiGLU FFN of the chosen expert (or_swiglu_ffn, pinned against torch above), rounded to fp32.  Sizes that are
    not multiples of the task size check the ragged last task."""
    if wfmt == WFMT_BF16:
        shapes = datagen.Shapes(T=3, H=264, E=5, top_k=1, I=136, Is=72)
    else:
        shapes = datagen.Shapes(T=3, H=288, E=5, top_k=1, I=96, Is=160)
    layer = datagen.make_layer(41, with_T(shapes, 1), wfmt)
    sh = layer.shexp_w.copy()
    mb = sh.size // 3
    if wfmt == WFMT_BF16:
        sh[2 * mb :] = 0
    else:
        # zero every scale of the shared downT rows: its weights decode to exactly 0
        sh[2 * mb :].reshape(shapes.Is, -1)[:, shapes.H // 2 :] = 0
    x, _ = draw_tokens(41, layer, shapes.T, ACT_F32)
    r = oracle.moe_ffn(shapes, ACT_F32, wfmt, x, layer.router_w, layer.expert_w, sh, layer.shexp_gate_w,
                       threads=threads)
    eb = layer.expert_w.size // shapes.E
    for t in range(shapes.T):
        e = int(r["ids"][t, 0])
        y = oracle.swiglu_ffn(layer.expert_w[e * eb : (e + 1) * eb], wfmt, shapes.H, shapes.I, x[t].astype(np.float64))
        np.testing.assert_array_equal(r["out"][t], y.astype(np.float32))


def test_expert_permutation_invariance(tiny_layer):
    layer = tiny_layer
    s = layer.shapes
    x, _ = draw_tokens(15, layer, 3, ACT_F32)
    perm = np.random.default_rng(0).permutation(s.E)
    eb = datagen.expert_bytes(WFMT_BF16, s.H, s.I)
    router = layer.router_w.reshape(s.E, s.H)[perm].reshape(-1)
    experts = np.concatenate([layer.expert_w[e * eb : (e + 1) * eb] for e in perm])
    pl = datagen.Layer(s, WFMT_BF16, router, layer.shexp_gate_w, experts, layer.shexp_w)
    a = run_oracle(layer, x, ACT_F32)
    b = run_oracle(pl, x, ACT_F32)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(perm[b["ids"]], a["ids"])


def test_bucketing_equals_stable_sort():
    rng = np.random.default_rng(3)
    for T, k, E in [(1, 2, 8), (8, 8, 128), (64, 8, 128), (5, 3, 4)]:
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, perm, active = oracle.bucketing(ids, E)
        flat = ids.reshape(-1)
        expect = sorted(range(T * k), key=lambda ts: (int(flat[ts]), ts))
        np.testing.assert_array_equal(perm, expect)
        np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
        np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        np.testing.assert_array_equal(active, np.nonzero(counts)[0])
        assert offsets[-1] == T * k


# ----------------------------------------------------------------------------
# Stored-format decoders


@pytest.mark.parametrize(
    "bits,value",
    [(0x3C00, 1.0), (0xC000, -2.0), (0x7BFF, 65504.0), (0x0001, 2.0**-24), (0x0400, 2.0**-14),
     (0x3555, 0.333251953125), (0x8000, -0.0), (0x03FF, 1023 * 2.0**-24), (0x2E66, 0.0999755859375)],
)
def test_f16_decoder_known_values(bits, value):
    assert oracle.f16_to_double(bits) == value
    assert float(np.array([bits], np.uint16).view(np.float16)[0]) == value


def test_bf16_decoder_known_values():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC040) == -3.0
    assert oracle.bf16_to_double(0x3E80) == 0.25
    assert oracle.bf16_to_double(0x0001) == 2.0**-133


def test_q4_hand_built_block():
    """Nibbles 0..15 with d = 0.5 decode to exactly (n - 8) * 0.5, low nibble first."""
    cols = 32
    nib = np.arange(32) % 16
    row = np.zeros(cols * 9 // 16, np.uint8)
    row[:16] = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    row[16:18] = [0x00, 0x38]  # fp16 0.5, little endian
    vals = oracle.decode_row(row, WFMT_Q4B32, cols, 0)
    np.testing.assert_array_equal(vals, (nib - 8) * 0.5)


def test_q4_encoder_byte_order_and_exact_values():
    """Values q*2^-4 with max |q| = 7 give d = 2^-4 exactly and nibble q+8, even element low."""
    q = np.array([(j % 15) - 7 for j in range(32)], np.int64)
    w = datagen.f32_to_bf16((q * 0.0625).astype(np.float32)).reshape(1, 32)
    enc = datagen.encode_q4b32(w)[0]
    assert enc[16] == 0x00 and enc[17] == 0x2C  # fp16 0.0625 = 0x2C00
    for j in range(16):
        assert enc[j] & 0x0F == q[2 * j] + 8
        assert enc[j] >> 4 == q[2 * j + 1] + 8
    np.testing.assert_array_equal(oracle.decode_row(enc, WFMT_Q4B32, 32, 0), q * 0.0625)


def test_q4_zero_block():
    w = np.zeros((2, 64), np.uint16)
    enc = datagen.encode_q4b32(w)
    assert np.all(enc[:, :32] == 0x88) and np.all(enc[:, 32:] == 0)
    assert np.all(oracle.decode_row(enc.reshape(-1), WFMT_Q4B32, 64, 1) == 0.0)


def test_q4_round_trip_bound():
    rows, cols = 64, 256
    w = datagen.normal_bf16(5, 5, rows * cols, 0.02).reshape(rows, cols)
    enc = datagen.encode_q4b32(w)
    wf = datagen.bf16_to_f32(w).astype(np.float64)
    d = np.ascontiguousarray(enc[:, cols // 2 :]).view("<f2").astype(np.float64)
    dd = np.repeat(d, 32, axis=1)
    for r in range(rows):
        dec = oracle.decode_row(enc.reshape(-1), WFMT_Q4B32, cols, r)
        err = np.abs(dec - wf[r])
        assert np.all(err <= dd[r] * 0.5 * (1 + 2.0**-10) + 1e-12)
        amax = np.abs(wf[r].reshape(-1, 32)).max(axis=1)
        np.testing.assert_allclose(d[r], amax / 7, rtol=2.0**-11)


# ----------------------------------------------------------------------------
# Transformer-block form (layer stack)


def test_rmsnorm_constant_vector():
    y = oracle.rmsnorm_bf16(np.full(2048, 3.0, np.float32))
    # 3 / sqrt(9 + 1e-6) rounds to bf16 1.0
    assert np.all(y == 0x3F80)


def test_rmsnorm_matches_numpy():
    x = datagen.normal_f32(21, 1, 2048) * 3.0
    y = datagen.bf16_to_f32(oracle.rmsnorm_bf16(x)).astype(np.float64)
    ref = x.astype(np.float64) / np.sqrt(np.mean(x.astype(np.float64) ** 2) + 1e-6)
    assert np.max(np.abs(y - ref) / np.maximum(np.abs(ref), 1e-30)) <= 2.0**-8


def test_float_to_bf16_rounds_ties_to_even():
    """bf16 keeps 8 significant bits.  Values exactly halfway between two bf16 neighbours go to the one with an
    even last bit (tests/golden/bf16_round_to_nearest_even.txt, worked from the bit patterns): truncation or
    rounding half up each fail one of the tie rows."""
    from tests.cases import golden

    for row in golden("bf16_round_to_nearest_even.txt"):
        f32_bits, bf16_bits = row.split()[:2]
        v = float(np.array([int(f32_bits, 16)], np.uint32).view(np.float32)[0])
        assert oracle.float_to_bf16(v) == int(bf16_bits, 16), row


def test_rmsnorm_exact_ties_with_unit_factor():
    """H = 16 values n/256 whose squares sum to exactly 16, so mean(x^2) = 1 and with eps = 0 the factor is exactly
    1: the output is bf16(x), and the tie values must round to even (see the test above)."""
    n = [259, 257, -259, 258, 1, 2, 86, 880] + [0] * 8
    assert sum(v * v for v in n) == 16 * 256 * 256
    y = oracle.rmsnorm_bf16((np.array(n, np.float64) / 256).astype(np.float32), eps=0.0)
    assert list(y[:8]) == [0x3F82, 0x3F80, 0xBF82, 0x3F81, 0x3B80, 0x3C00, 0x3EAC, 0x405C]
    assert np.all(y[8:] == 0)


def test_rmsnorm_eps_inside_the_root():
    """x = 1e-3 everywhere: y = c / sqrt(c^2 + eps) (tests/golden/rmsnorm_eps.txt, worked by hand): the eps
    values tell eps inside the root from eps outside it or scaled by H."""
    from tests.cases import golden

    for row in golden("rmsnorm_eps.txt"):
        H, eps, want = row.split()
        c = np.full(int(H), 1e-3, np.float32)
        assert np.all(oracle.rmsnorm_bf16(c, eps=float(eps)) == int(want, 16)), row


def test_block_step_is_norm_then_layer_then_residual():
    layer = datagen.make_layer(31, SMALL_Q4, WFMT_Q4B32)
    s = layer.shapes
    x_res = datagen.normal_f32(31, 99, s.H).reshape(1, s.H)
    new, ids, xn = oracle.block_step(s, WFMT_Q4B32, x_res, layer.router_w, layer.expert_w, layer.shexp_w,
                                     layer.shexp_gate_w)
    np.testing.assert_array_equal(xn[0], oracle.rmsnorm_bf16(x_res[0]))
    r = oracle.moe_ffn(s, ACT_BF16, WFMT_Q4B32, xn, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w)
    np.testing.assert_array_equal(ids, r["ids"])
    np.testing.assert_array_equal(new, (x_res + r["out"]).astype(np.float32))


# ----------------------------------------------------------------------------
# int8 weights with an int8 activation (the int8 linear of "ggml operator extensions", sd.cpp integration)


def test_i8_activation_quantizer_known_values():
    """tests/golden/int8_activation_quantizer.txt, worked by hand: max|x| = 127 gives the scale 127 / 127 = 1
    exactly, so q is x rounded half away from zero; max|x| = 1 gives fp32(1/127) and 0.5 / s = 63.5 -> 64; a
    zero row gives scale 0 and zero codes."""
    from tests.cases import golden

    for row in golden("int8_activation_quantizer.txt"):
        xs, fill, codes, scale = [f.strip() for f in row.split("|")]
        vals = [float(v) for v in xs.split(",")]
        x = np.array(vals + [float(fill)] * (16 - len(vals)))
        q, s = oracle.quantize_i8(x)
        assert s == float(np.array([int(scale, 16)], np.uint32).view(np.float32)[0]), row
        assert list(q[: len(vals)]) == [int(c) for c in codes.split(",")], row
        if float(fill) == 0.0:
            assert not q[len(vals):].any()


def test_i8_weight_rows_decode():
    """An int8 row is its C signed bytes, then its fp32 scale; the value is scale * q."""
    cols = 32
    row = np.zeros(cols + 16, np.uint8)
    qv = (np.arange(cols) - 16).astype(np.int8)
    row[:cols] = qv.view(np.uint8)
    row[cols : cols + 4] = np.array([0.25], "<f4").view(np.uint8)
    np.testing.assert_array_equal(oracle.decode_row(row, datagen.WFMT_I8, cols, 0), qv.astype(np.float64) * 0.25)


def _i8_block_dequant(block, H, inter):
    rb = H + 16
    mats = []
    for m in range(3):
        rows = block[m * inter * rb : (m + 1) * inter * rb].reshape(inter, rb)
        q = rows[:, :H].view(np.int8).astype(np.float64)
        sc = rows[:, H : H + 4].copy().view("<f4").astype(np.float64)
        mats.append(q * sc)
    return mats


def test_i8_ffn_matches_torch_for_integral_activation():
    """x integral with max|x| = 127: the scale is 1 and the int8 activation is x itself, so the int8 path must
    equal the plain SwiGLU FFN of the dequantised weights (torch, fp64) up to the fp32 rounding of
    float(dot) * xs * s."""
    H, inter = 256, 96
    block = datagen.expert_block(51, 0, H, inter, datagen.WFMT_I8)
    Wg, Wu, WdT = (torch.from_numpy(m) for m in _i8_block_dequant(block, H, inter))
    x = np.round(datagen.normal_f32(51, 3, H).astype(np.float64) * 40.0)
    x = np.clip(x, -126, 126)
    x[7] = 127.0
    xt = torch.from_numpy(x)
    g, u = Wg @ xt, Wu @ xt
    h = torch.nn.functional.silu(g) * u
    ref = h @ WdT
    y = oracle.swiglu_ffn(block, datagen.WFMT_I8, H, inter, x)
    # the projections round twice in fp32 (float(dot) is exact here, then * xs = 1 and * s), so h carries a
    # relative error of a few 2^-24; each output moves by at most that times sum_i |WdT[i,c] h_i|
    bound = 4e-7 * (h.abs() @ WdT.abs()).numpy() + 1e-12
    assert np.all(np.abs(y - ref.numpy()) <= bound)


def test_i8_ffn_quantization_error_is_bounded():
    """For a general x the int8 activation differs from x by at most half a step (xs / 2) per element; the
    resulting change of the FFN output stays within the bound that half a step per element gives through the
    gate and up projections (checked against torch on the unquantised x, loosely)."""
    H, inter = 256, 64
    block = datagen.expert_block(52, 0, H, inter, datagen.WFMT_I8)
    Wg, Wu, WdT = (torch.from_numpy(m) for m in _i8_block_dequant(block, H, inter))
    x = datagen.normal_f32(52, 4, H).astype(np.float64)
    q, s = oracle.quantize_i8(x)
    assert np.all(np.abs(x - q.astype(np.float64) * s) <= s / 2 * (1 + 1e-6))
    xq = torch.from_numpy(q.astype(np.float64) * s)
    ref_q = (torch.nn.functional.silu(Wg @ xq) * (Wu @ xq)) @ WdT
    y = oracle.swiglu_ffn(block, datagen.WFMT_I8, H, inter, x)
    # the oracle is the FFN of the quantised activation (up to fp32 rounding of the projections)
    np.testing.assert_allclose(y, ref_q.numpy(), rtol=1e-5, atol=1e-6 * float(ref_q.abs().max()))
    ref = (torch.nn.functional.silu(Wg @ torch.from_numpy(x)) * (Wu @ torch.from_numpy(x))) @ WdT
    assert float((torch.from_numpy(y) - ref).abs().max()) < 0.05 * float(ref.abs().max())


def test_i8_zero_activation_gives_zero_output():
    H, inter = 128, 64
    block = datagen.expert_block(53, 0, H, inter, datagen.WFMT_I8)
    y = oracle.swiglu_ffn(block, datagen.WFMT_I8, H, inter, np.zeros(H))
    assert np.all(y == 0.0)


def test_i8_layer_routing_is_format_independent():
    """The router and the top-k do not depend on the expert weight format."""
    s = datagen.Shapes(T=3, H=256, E=8, top_k=2, I=64, Is=64)
    lb = datagen.make_layer(54, with_T(s, 1), WFMT_BF16)
    li = datagen.make_layer(54, with_T(s, 1), datagen.WFMT_I8)
    x, _ = draw_tokens(54, lb, 3, ACT_BF16)
    rb = oracle.moe_ffn(s, ACT_BF16, WFMT_BF16, x, lb.router_w, lb.expert_w, lb.shexp_w, lb.shexp_gate_w)
    ri = oracle.moe_ffn(s, ACT_BF16, datagen.WFMT_I8, x, li.router_w, li.expert_w, li.shexp_w, li.shexp_gate_w)
    np.testing.assert_array_equal(rb["ids"], ri["ids"])
    np.testing.assert_array_equal(rb["p"], ri["p"])
