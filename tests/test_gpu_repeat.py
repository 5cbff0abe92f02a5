"""Bitwise repeatability at the full layer size.

GPU runs of the layer must be bitwise identical to each other: the output,
the top-k ids and their weights of two executes on the same inputs are
compared with memcmp semantics, the second run on a differently pre-filled
workspace at another base address and on another stream.  This is the "byte
identical" property that "ggml-cuda: overlap the MoE shared expert on a
separate stream" (section "Gated to small batches") requires of its
overlapped schedule; here it must hold for every path: the decode row kernel
(bf16 and 4-bit weights, T = 1 and 8), the grouped GEMMs of the batched path
(T = 256) and the pre-norm block form of the 48-layer stack's layer.
"""

from __future__ import annotations

import numpy as np
import pytest

import datagen
from datagen import ACT_BF16, WFMT_BF16, WFMT_Q4B32
from tests.cases import DECODE, with_T

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", params=[WFMT_BF16, WFMT_Q4B32], ids=["bf16", "q4"])
def full_layer(request):
    from tests.devlayer import DevLayer

    layer = datagen.make_layer(5150, DECODE, request.param)
    return layer, DevLayer(layer)


def _run_twice(dl, shapes, wfmt, x_dev, block=False):
    """Two executes: workspace A (0xA5 fill, offset 0, stream 1) and workspace B (0x5A fill, offset 1280 bytes,
    stream 2).  Returns [(out, ids, p)] * 2 as host arrays."""
    import fusion_backend_gb300 as fb

    plan, ws_bytes = fb.moe_ffn_prepare(shapes, ACT_BF16, wfmt)
    res = []
    for fill, off in ((0xA5, 0), (0x5A, 1280)):
        buf = torch.full((ws_bytes + 4096,), fill, dtype=torch.uint8, device="cuda")
        ws = buf[off : off + ws_bytes]
        stream = torch.cuda.Stream()
        ids = torch.full((shapes.T, shapes.top_k), -1, dtype=torch.int32, device="cuda")
        p = torch.full((shapes.T, shapes.top_k), -1.0, dtype=torch.float32, device="cuda")
        if block:
            out = x_dev.clone()
        else:
            out = torch.full((shapes.T, shapes.H), float("nan"), dtype=torch.float32, device="cuda")
        stream.wait_stream(torch.cuda.current_stream())
        if block:
            fb.moe_ffn_execute_block(plan, ws, out, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w,
                                     eps=1e-6, topk_ids=ids, topk_w=p, stream=stream)
        else:
            fb.moe_ffn_execute_ex(plan, ws, x_dev, dl.router_w, dl.expert_w, dl.shexp_w, dl.gate_w, out, ids, p,
                                  stream=stream)
        stream.synchronize()
        assert fb.moe_ffn_read_status(plan, ws, stream) == 0
        res.append((out.cpu().numpy(), ids.cpu().numpy(), p.cpu().numpy()))
    fb.moe_ffn_destroy(plan)
    return res


def _assert_same(a, b, label):
    for name, u, v in zip(("out", "ids", "p"), a, b):
        assert u.tobytes() == v.tobytes(), f"{label}: {name} differs between runs"
    assert np.all(a[1] >= 0) and np.all(np.isfinite(a[0]))


@pytest.mark.parametrize("T", [1, 8, 256])
def test_full_size_runs_are_bitwise_identical(full_layer, T):
    layer, dl = full_layer
    shapes = with_T(DECODE, T)
    x = np.stack([datagen.token_x(5150, 3000 + t, DECODE.H, ACT_BF16) for t in range(T)])
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    a, b = _run_twice(dl, shapes, layer.wfmt, xd)
    _assert_same(a, b, f"wfmt={layer.wfmt} T={T}")


def test_full_size_block_form_is_bitwise_identical(full_layer):
    layer, dl = full_layer
    shapes = with_T(DECODE, 1)
    x_res = torch.from_numpy(datagen.normal_f32(5151, 9, DECODE.H).reshape(1, DECODE.H) * 4.0).cuda()
    a, b = _run_twice(dl, shapes, layer.wfmt, x_res, block=True)
    _assert_same(a, b, f"block form wfmt={layer.wfmt}")
