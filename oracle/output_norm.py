"""fp64 oracle of the output norm fused into the decode-side calls (TEST
INFRASTRUCTURE: imported only by ``tests/`` through ``oracle``).

blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "三条容易被忽略的
代价" (1), lists an output norm among the steps K3 fuses into its replay
kernel without defining it.  The reading taken here is a per-head RMS norm of
each output row over its dv channels with a per-head, per-channel weight:

    y[.., h, j] = o[.., h, j] / sqrt(mean_j' o[.., h, j']^2 + eps) * w[h, j].
"""
from __future__ import annotations

import numpy as np


def rms_norm(o, weight, eps):
    """o [..., H, dv], weight [H, dv] -> float64 [..., H, dv]."""
    if hasattr(o, "detach"):
        o = o.detach().to("cpu").double().numpy()
    if hasattr(weight, "detach"):
        weight = weight.detach().to("cpu").double().numpy()
    o = np.asarray(o, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return o / np.sqrt(ms + float(eps)) * w
