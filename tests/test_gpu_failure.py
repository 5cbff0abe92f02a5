"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up, records MOE_FFN_ERR_TIMEOUT in the status word, and the
context stays usable -- the next execute on the same workspace runs, matches
the oracle and clears the word."""

from __future__ import annotations

import time

import numpy as np
import pytest

import datagen
from datagen import ACT_F32, WFMT_BF16
from tests.cases import TINY, draw_tokens, with_T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


# 0: an mbarrier phase that never completes; 1: a barrier flag that never receives the epoch; 2: a tagged word
# that never carries the call's tag
@pytest.mark.parametrize("which", [0, 1, 2])
def test_bounded_wait_gives_up_and_context_stays_usable(which):
    import fusion_backend_gb300 as fb
    import oracle
    from tests.devlayer import DevLayer, tolerance_ok

    layer = datagen.make_layer(1101, TINY, WFMT_BF16)
    s = with_T(TINY, 2)
    plan, ws_bytes = fb.moe_ffn_prepare(s, ACT_F32, WFMT_BF16)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    fb.moe_ffn_probe_timeout(plan, ws, which)
    status = fb.moe_ffn_read_status(plan, ws)
    elapsed = time.perf_counter() - t0
    assert status == fb.ERR_TIMEOUT, f"status {status}"
    assert elapsed < 30.0, f"the bounded wait took {elapsed:.1f} s"
    # the context and the workspace are usable at once
    dl = DevLayer(layer)
    x, _ = draw_tokens(1101, layer, 2, ACT_F32)
    out = torch.zeros((2, s.H), dtype=torch.float32, device="cuda")
    fb.moe_ffn_execute(plan, ws, torch.from_numpy(x).cuda(), dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, out)
    assert fb.moe_ffn_read_status(plan, ws) == 0
    ref = oracle.moe_ffn(s, ACT_F32, WFMT_BF16, x, layer.router_w, layer.expert_w, layer.shexp_w, layer.shexp_gate_w)
    assert tolerance_ok(out.cpu().numpy(), ref["out"])[0]
    fb.moe_ffn_destroy(plan)


def test_probe_rejects_bad_arguments():
    import fusion_backend_gb300 as fb

    plan, ws_bytes = fb.moe_ffn_prepare(with_T(TINY, 1), ACT_F32, WFMT_BF16)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(fb.MoeFFNError) as e:
        fb.moe_ffn_probe_timeout(plan, ws, 3)
    assert e.value.status == fb.ERR_INVALID_ARG
    with pytest.raises(fb.MoeFFNError) as e:
        fb.moe_ffn_probe_timeout(plan, ws, 0, workspace_bytes=ws_bytes - 1)
    assert e.value.status == fb.ERR_WORKSPACE
    fb.moe_ffn_destroy(plan)
