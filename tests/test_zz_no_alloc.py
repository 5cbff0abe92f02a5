"""The allocation-free entry point, moe_ffn_execute_static_scratch.

It exists for callers that cannot allocate device memory (a library embedded
in a runtime that already owns all free device memory, or a plugin given no
allocator): instead of a caller workspace it uses one device array inside the
library.  Here it is called through the C ABI and its output is compared with
moe_ffn_execute's on the same inputs, for two calls in a row on different
tokens.  Both run the same deterministic kernels, so the outputs must be equal
bit for bit (a stale or misplaced scratch region would show up there); the
parity tests' tolerance (max|d| <= 1e-2 rms + 1e-5) is checked as well.  The
cases cover the decode path and the batched path (grouped GEMMs whose tensor
maps then point into the library's array), with bf16 and 4-bit weights.

This file is collected last on purpose, and passes both alone in a fresh
process and after the rest of the suite.
"""

from __future__ import annotations

import numpy as np
import pytest

import datagen
from datagen import ACT_BF16, ACT_F32, WFMT_BF16, WFMT_Q4B32, Shapes
from tests.cases import DECODE, TINY, draw_tokens, with_T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _tol_ok(got, ref):
    ref = ref.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    return err <= 1e-2 * rms + 1e-5, err, rms


@pytest.mark.parametrize(
    "base,T,act,wfmt",
    [(TINY, 2, ACT_F32, WFMT_BF16), (DECODE, 1, ACT_BF16, WFMT_BF16), (DECODE, 8, ACT_BF16, WFMT_Q4B32),
     (DECODE, 64, ACT_BF16, WFMT_BF16), (DECODE, 64, ACT_BF16, WFMT_Q4B32)],
)
def test_static_scratch_matches_workspace_entry_point(base, T, act, wfmt):
    import fusion_backend_gb300 as fb
    from tests.devlayer import DevLayer

    layer = datagen.make_layer(4242, with_T(base, 1), wfmt)
    dl = DevLayer(layer)
    shapes = with_T(base, T)
    plan, ws_bytes = fb.moe_ffn_prepare(shapes, act, wfmt)
    assert ws_bytes <= fb.STATIC_SCRATCH_BYTES
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for call, first_token in enumerate((0, 100)):  # two calls in a row, different inputs
        x, _ = draw_tokens(4242, layer, T, act, first_token=first_token)
        xd = torch.from_numpy(x.view(np.int16) if act == ACT_BF16 else x).cuda()
        ref = torch.empty((T, shapes.H), dtype=torch.float32, device="cuda")
        got = torch.full((T, shapes.H), float("nan"), dtype=torch.float32, device="cuda")
        fb.moe_ffn_execute(plan, ws, xd, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, ref)
        fb.moe_ffn_execute_static_scratch(plan, xd, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, got)
        torch.cuda.synchronize()
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert g.tobytes() == r.tobytes(), f"call {call}: outputs differ bitwise"
        ok, err, rms = _tol_ok(g, r)
        assert ok, f"call {call}: max|d| {err:.3e} vs rms {rms:.3e}"
    fb.moe_ffn_destroy(plan)


def test_static_scratch_rejects_plans_larger_than_the_array():
    import fusion_backend_gb300 as fb

    big = Shapes(T=8, H=4096, E=128, top_k=8, I=768, Is=512)  # per-block partial outputs alone exceed 16 MiB
    plan, ws_bytes = fb.moe_ffn_prepare(big, ACT_BF16, WFMT_BF16)
    assert ws_bytes > fb.STATIC_SCRATCH_BYTES
    fake = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(fb.MoeFFNError) as e:
        fb.moe_ffn_execute_static_scratch(plan, fake, fake, fake, fake, fake, fake)
    assert e.value.status == fb.ERR_WORKSPACE
    fb.moe_ffn_destroy(plan)
