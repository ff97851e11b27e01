"""SwiGLU between the two expert GEMMs.  Test infrastructure only.

Chinese translation, Figure 5 legend: an expert runs the w13 GEMM, a
quantization ("Q") and the w2 GEMM.  The pages do not name the activation;
the MoE expert-forward workload has SwiGLU gate/up projections [4096 -> 1536
x 2] and a down projection [1536 -> 4096], so w13 stacks gate (output columns
0..I-1) above up (columns I..2I-1) and h = silu(gate) * up with
silu(x) = x / (1 + e^-x).  Float64 here; the library computes fp32 and
rounds h to bf16, so comparisons allow a few bf16 ulps.
"""
from __future__ import annotations

import numpy as np


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def forward(y13):
    """h [M, I] from y13 [M, 2I]."""
    y13 = np.asarray(y13, dtype=np.float64)
    I = y13.shape[1] // 2
    return silu(y13[:, :I]) * y13[:, I:]


def backward(dh, y13):
    """d y13 [M, 2I] from dh [M, I]: d gate = dh * up * silu'(gate) with
    silu'(x) = s(x) (1 + x (1 - s(x))), s the logistic function; d up =
    dh * silu(gate)."""
    y13 = np.asarray(y13, dtype=np.float64)
    dh = np.asarray(dh, dtype=np.float64)
    I = y13.shape[1] // 2
    gate, up = y13[:, :I], y13[:, I:]
    s = 1.0 / (1.0 + np.exp(-gate))
    dgate = dh * up * s * (1.0 + gate * (1.0 - s))
    dup = dh * gate * s
    return np.concatenate([dgate, dup], axis=1)
