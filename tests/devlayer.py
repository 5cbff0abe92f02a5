"""Upload seeded layers to the GPU and run the library on them (tests only)."""

from __future__ import annotations

import numpy as np
import torch

import datagen
import fusion_backend_gb300 as fb


class DevLayer:
    def __init__(self, layer: datagen.Layer):
        self.layer = layer
        dev = "cuda"
        self.router_w = torch.from_numpy(layer.router_w.view(np.int16).copy()).to(dev)
        self.gate_w = torch.from_numpy(layer.shexp_gate_w.view(np.int16).copy()).to(dev)
        self.expert_w = torch.from_numpy(layer.expert_w).to(dev)
        self.shexp_w = torch.from_numpy(layer.shexp_w).to(dev)

    def run(self, x: np.ndarray, act: int, T: int | None = None, ws_fill: int | None = None, out_alias=False):
        s = self.layer.shapes
        T = x.shape[0] if T is None else T
        shapes = datagen.Shapes(T, s.H, s.E, s.top_k, s.I, s.Is)
        m = fb.MoeFFN(shapes, act, self.layer.wfmt)
        if ws_fill is not None:
            m.workspace.fill_(ws_fill)
        xd = torch.from_numpy(x.view(np.int16) if act == datagen.ACT_BF16 else x).cuda()
        ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device="cuda")
        p = torch.full((T, s.top_k), -1.0, dtype=torch.float32, device="cuda")
        if out_alias:
            # out occupies the same storage as x (x is read completely before out is written)
            buf = torch.zeros(T * s.H, dtype=torch.float32, device="cuda")
            xv = buf.view(torch.int16 if act == datagen.ACT_BF16 else torch.float32)[: T * s.H].view(T, s.H)
            xv.copy_(xd)
            out = buf.view(T, s.H)
            m(xv, self.router_w, self.expert_w, self.shexp_w, self.gate_w, out=out, topk_ids=ids, topk_w=p)
        else:
            out = m(xd, self.router_w, self.expert_w, self.shexp_w, self.gate_w, topk_ids=ids, topk_w=p)
        torch.cuda.synchronize()
        status = m.status()
        routing = m.routing()
        res = {"out": out.cpu().numpy(), "ids": ids.cpu().numpy(), "p": p.cpu().numpy(), "status": status,
               "routing": routing}
        m.close()
        return res


def tolerance_ok(gpu_out: np.ndarray, ref_out: np.ndarray) -> tuple[bool, float, float]:
    """max|d| <= 1e-2 * rms(oracle) + 1e-5 over all outputs."""
    ref = ref_out.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = float(np.max(np.abs(gpu_out.astype(np.float64) - ref)))
    return err <= 1e-2 * rms + 1e-5, err, rms
