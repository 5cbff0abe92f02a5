"""The two-stream form of the layer (moe_ffn_execute_two_stream), the design of
"ggml-cuda: overlap the MoE shared expert on a separate stream" (section
"What this changes"): the routed branch on the main stream, the gated shared
expert on a second stream forked from it, joined by add(ffn_moe_out,
ffn_shexp).

Checked: the overlapped run is byte-identical to the same kernels run one
after the other (the page's "Output is byte-identical to sequential", section
"Gated to small batches"), its ids and output match the oracle, and it agrees
with the fused kernel within the tolerance (the fused kernel forms its sums
in another order).
"""

from __future__ import annotations

import numpy as np
import pytest

import datagen
import oracle
from datagen import ACT_BF16, ACT_F32, WFMT_BF16, WFMT_I8, WFMT_Q4B32
from tests.cases import DECODE, TINY, draw_tokens, with_T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize(
    "base,T,act,wfmt",
    [(TINY, 2, ACT_F32, WFMT_BF16), (DECODE, 1, ACT_BF16, WFMT_BF16), (DECODE, 8, ACT_BF16, WFMT_BF16),
     (DECODE, 1, ACT_BF16, WFMT_Q4B32), (DECODE, 4, ACT_BF16, WFMT_Q4B32), (DECODE, 2, ACT_BF16, WFMT_I8),
     (TINY, 3, ACT_F32, WFMT_I8)],
)
def test_two_streams_match_sequential_oracle_and_fused(base, T, act, wfmt):
    import fusion_backend_gb300 as fb
    from tests.devlayer import DevLayer, tolerance_ok

    layer = datagen.make_layer(5300, with_T(base, 1), wfmt)
    dl = DevLayer(layer)
    shapes = with_T(base, T)
    x, _ = draw_tokens(5300, layer, T, act, first_token=7)
    xd = torch.from_numpy(x.view(np.int16) if act == ACT_BF16 else x).cuda()
    plan, ws_bytes = fb.moe_ffn_prepare(shapes, act, wfmt)
    two_bytes = fb.moe_ffn_query(plan, fb.QUERY_TWO_STREAM_WORKSPACE)
    main, aux = torch.cuda.Stream(), torch.cuda.Stream()
    fork, join = torch.cuda.Event(), torch.cuda.Event()
    outs = []
    for overlapped, fill in ((True, 0xA5), (False, 0x5A)):
        ws = torch.full((two_bytes,), fill, dtype=torch.uint8, device="cuda")
        out = torch.full((T, shapes.H), float("nan"), dtype=torch.float32, device="cuda")
        main.wait_stream(torch.cuda.current_stream())
        fb.moe_ffn_execute_two_stream(plan, ws, xd, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, out,
                                      aux_stream=aux if overlapped else None, fork_event=fork, join_event=join,
                                      stream=main)
        main.synchronize()
        aux.synchronize()
        outs.append(out.cpu().numpy())
    assert outs[0].tobytes() == outs[1].tobytes(), "two-stream and sequential runs differ"
    ref = oracle.moe_ffn(shapes, act, wfmt, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w)
    ok, err, rms = tolerance_ok(outs[0], ref["out"])
    assert ok, f"max|d| {err:.3e} > 1e-2 * rms({rms:.3e}) + 1e-5"
    fused = dl.run(x, act)
    assert fused["status"] == 0
    np.testing.assert_array_equal(fused["ids"], ref["ids"])
    ok, err, rms = tolerance_ok(outs[0], fused["out"].astype(np.float64))
    assert ok, f"two-stream vs fused: max|d| {err:.3e} vs rms {rms:.3e}"
    fb.moe_ffn_destroy(plan)


def test_two_streams_reject_batched_plans():
    import fusion_backend_gb300 as fb

    plan, _ = fb.moe_ffn_prepare(with_T(DECODE, 64), ACT_BF16, WFMT_BF16)
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(fb.MoeFFNError) as e:
        fb.moe_ffn_execute_two_stream(plan, buf, buf, buf, buf, buf, buf, buf)
    assert e.value.status == fb.ERR_UNSUPPORTED
    fb.moe_ffn_destroy(plan)
