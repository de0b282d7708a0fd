"""Gated RMSNorm of the KDA output -- TEST INFRASTRUCTURE ONLY (see oracle/__init__).

The pages name a "gated RMSNorm in the epilogue (fuse_output_norm)" of the KDA
kernel (TensorRT-LLM page "Kimi K3 work for Rubin (SM107)", Description: the
mixer applies the gated RMSNorm and the output gate in the kernel's epilogue,
with the o_norm weights) without writing the formula.  Reading taken here, the
plainest one the page supports: per (token, head), over the 128 value
channels c,

    y_c = o_c / sqrt(mean_c(o_c^2) + eps) * w_c * sigmoid(gate_c)

with o the attention output before rounding, w the o_norm weight (one per value
channel, shared by all heads) and gate the output-gate activations (indexed like
o).  Plain fp64 numpy, written straight from that definition.
"""
import numpy as np


def gated_rmsnorm(o, gate, weight, eps):
    """o, gate: [..., V]; weight: [V].  Returns y [..., V] in fp64."""
    o = np.asarray(o, dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + float(eps))
    return o / rms * w * (1.0 / (1.0 + np.exp(-gate)))
