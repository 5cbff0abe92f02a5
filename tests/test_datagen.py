"""The seeded input generator: published splitmix64 outputs, counter-based
slicing, distribution and the bf16 / fp16 roundings it applies."""

import numpy as np

import datagen

GAMMA = 0x9E3779B97F4A7C15
MASK = (1 << 64) - 1


def test_splitmix64_published_sequence():
    # splitmix64 started from state 0 (tests/golden/splitmix64_state0.txt: Steele, Lea and Flood 2014; Vigna's
    # reference code)
    from tests.cases import golden

    L = datagen.lib()
    for row in golden("splitmix64_state0.txt"):
        i, want = row.split()
        assert L.dg_mix64((GAMMA * int(i)) & MASK) == int(want, 16), f"output {i}"


def test_slices_regenerate_exactly():
    full = datagen.normal_bf16(3, 17, 10_000, 0.02)
    part = datagen.normal_bf16(3, 17, 1_001, 0.02, offset=4_321)
    np.testing.assert_array_equal(full[4_321:5_322], part)
    f32 = datagen.normal_f32(3, 17, 10_000, 0.02)
    np.testing.assert_array_equal(datagen.f32_to_bf16(f32), full)


def test_streams_and_seeds_differ():
    a = datagen.normal_f32(1, 1, 1000)
    assert not np.array_equal(a, datagen.normal_f32(1, 2, 1000))
    assert not np.array_equal(a, datagen.normal_f32(2, 1, 1000))


def test_normal_moments():
    v = datagen.normal_f32(11, 5, 2_000_000).astype(np.float64)
    assert abs(v.mean()) < 3e-3
    assert abs(v.std() - 1.0) < 3e-3
    assert abs(np.mean(v**4) / v.var() ** 2 - 3.0) < 0.03


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 65504.0], np.float32)
    got = datagen.f32_to_bf16(vals)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 is a tie -> 1+2^-6; 1+2^-9 rounds down.
    np.testing.assert_array_equal(got, [0x3F80, 0x3F80, 0x3F82, 0x3F80, 0xC020, 0x4780])


def test_f16_rounding_matches_numpy():
    L = datagen.lib()
    x = np.concatenate([datagen.normal_f32(4, 4, 20000) * s for s in (1e-7, 1e-4, 1.0, 300.0, 3e4)])
    mine = np.array([L.dg_f32_to_f16(float(v)) for v in x], np.uint16)
    ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


def test_layer_block_sizes():
    s = datagen.Shapes(1, 256, 4, 2, 256, 256)
    for wfmt in (datagen.WFMT_BF16, datagen.WFMT_Q4B32):
        L = datagen.make_layer(1, s, wfmt)
        eb = datagen.expert_bytes(wfmt, s.H, s.I)
        assert L.expert_w.size == s.E * eb
        assert L.shexp_w.size == datagen.expert_bytes(wfmt, s.H, s.Is)
        assert eb % 16 == 0


def test_i8_encoder_scale_rounding_and_layout():
    """Per row: s = fp32(max|w|) / 127, q = round half away from zero of w / s, then s and 12 zero bytes."""
    w = datagen.f32_to_bf16(np.array([[1.0, -0.5, 0.25, 0.49609375] + [0.0] * 12], np.float32))
    e = datagen.encode_i8(w)
    assert e.shape == (1, 32)
    assert list(e[0, :4].view(np.int8)) == [127, -64, 32, 63]
    assert e[0, 16:20].view("<f4")[0] == np.float32(1.0) / np.float32(127.0)
    assert not e[0, 20:].any()
    z = datagen.encode_i8(np.zeros((1, 16), np.uint16))
    assert not z.any()
    rows = datagen.normal_bf16(9, 9, 64 * 256, 0.02).reshape(64, 256)
    enc = datagen.encode_i8(rows)
    q = enc[:, :256].view(np.int8).astype(np.float64)
    s = enc[:, 256:260].copy().view("<f4").astype(np.float64)
    wf = datagen.bf16_to_f32(rows).astype(np.float64)
    # w / s is formed in fp32 before the rounding: up to 127 * 2^-24 beyond half a step
    assert np.all(np.abs(wf - q * s) <= s * (0.5 + 1e-5) + 1e-12)
