"""Seeded test cases: the workload shapes and the near-tie resampling rule.

Inputs come from ``datagen``; the resampling rule needs router logits, so it
lives here (tests may call the oracle, the generator may not).
"""

from __future__ import annotations

import os

import numpy as np

import datagen
import oracle
from datagen import ACT_BF16, ACT_F32, WFMT_BF16, WFMT_Q4B32, Shapes

# Workload shapes: the tiny layer, the decode layer, and a small 4-bit layer
# whose reduction sizes are multiples of 256 (the 4-bit row format needs it).
TINY = Shapes(T=1, H=256, E=8, top_k=2, I=128, Is=256)
DECODE = Shapes(T=1, H=2048, E=128, top_k=8, I=768, Is=512)
SMALL_Q4 = Shapes(T=1, H=256, E=8, top_k=2, I=256, Is=256)

NEAR_TIE_GAP = 1e-3


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> list[str]:
    """The data lines of tests/golden/<name> (comment lines, starting with '#', skipped)."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


def with_T(s: Shapes, T: int) -> Shapes:
    return Shapes(T=T, H=s.H, E=s.E, top_k=s.top_k, I=s.I, Is=s.Is)


def x_as_f64(x: np.ndarray, act: int) -> np.ndarray:
    return x.astype(np.float64) if act == ACT_F32 else datagen.bf16_to_f32(x).astype(np.float64)


def kth_gap(logits: np.ndarray, k: int) -> float:
    srt = np.sort(logits.astype(np.float64))[::-1]
    return float(srt[k - 1] - srt[k]) if k < logits.size else np.inf


def draw_tokens(seed: int, layer: datagen.Layer, T: int, act: int, first_token: int = 0, gap: float = NEAR_TIE_GAP):
    """T token activations; a token whose k-th and (k+1)-th oracle router
    logits differ by less than ``gap`` (absolute, fp32 logits) is redrawn with
    the next sub-seed.  Returns (x [T,H], number of redraws)."""
    s = layer.shapes
    rows = []
    redraws = 0
    for t in range(T):
        sub = 0
        while True:
            x = datagen.token_x(seed, first_token + t, s.H, act, sub)
            lg = oracle.router_logits(layer.router_w, s.E, s.H, x_as_f64(x, act))
            if kth_gap(lg, s.top_k) >= gap:
                break
            sub += 1
            redraws += 1
        rows.append(x)
    return np.stack(rows), redraws
