"""Weight-only grouped affine quantization (8 or 4 bits, groups of 64 along the input axis)
for the oracle: codes, scales and biases from bf16 weights, and the exact dequantization.

TEST INFRASTRUCTURE ONLY (see the package docstring). The page "Dentro de un LLM: Inferencia
en Python puro para Qwen3-0.6B en MLX" ("Lo que omite el script") names 4- and 8-bit weights
as what production inference uses and keeps bfloat16; it gives no algorithm. Reading taken
(the affine group quantization that MLX's quantized layers use, restated):

* Each row of a weight matrix [out, in] is cut into groups of 64 consecutive inputs.
* Per group, with w the bf16 values widened to fp32: scale = (max(w) - min(w)) / (2^bits - 1)
  in fp32, then the scale and bias = min(w) are rounded to fp16 (round to nearest even),
  which is how they are stored.
* Code q = clamp(rint((w - bias) / scale), 0, 2^bits - 1), computed in fp32 (division and
  rint round to nearest even); a group whose fp16 scale is 0 gets code 0 everywhere.
* The dequantized weight is scale * q + bias, evaluated here in fp64 from the fp16 values.

The codes are integers decided in fp32 on both sides (here and in the GPU's quantizer), so
they agree bit for bit; only the dequantized products differ by fp32 rounding.
"""

from __future__ import annotations

from typing import Dict, Tuple

import numpy as np

GROUP = 64
QUANT_TENSORS = ("self_attn.q_proj.weight", "self_attn.k_proj.weight", "self_attn.v_proj.weight",
                 "self_attn.o_proj.weight", "mlp.gate_proj.weight", "mlp.up_proj.weight",
                 "mlp.down_proj.weight")


def _bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantize(bits: np.ndarray, nbits: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """bf16 bits [out, in] -> codes uint8 [out, in], scales and biases fp16 [out, in / 64]."""
    w = _bf16_to_f32(bits)
    out, k = w.shape
    assert k % GROUP == 0 and nbits in (4, 8)
    g = w.reshape(out, k // GROUP, GROUP)
    lo = g.min(axis=2)
    hi = g.max(axis=2)
    levels = np.float32(2 ** nbits - 1)
    scale16 = ((hi - lo) / levels).astype(np.float16)
    bias16 = lo.astype(np.float16)
    s = scale16.astype(np.float32)[..., None]
    b = bias16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((g - b) / s)
    q = np.where(s == 0, np.float32(0), q)
    q = np.clip(q, 0, levels).astype(np.uint8)
    return q.reshape(out, k), scale16, bias16


def dequantize(codes: np.ndarray, scale16: np.ndarray, bias16: np.ndarray) -> np.ndarray:
    """scale * q + bias in fp64, [out, in]."""
    out, k = codes.shape
    q = codes.reshape(out, k // GROUP, GROUP).astype(np.float64)
    return (scale16.astype(np.float64)[..., None] * q + bias16.astype(np.float64)[..., None]).reshape(out, k)


class QuantizedWeights:
    """A weight provider for ``oracle.Model`` whose projection matrices are the dequantized
    values (fp64) of the given provider's bf16 weights; norms and the tied embedding stay bf16."""

    def __init__(self, base, nbits: int):
        self.base = base
        self.nbits = nbits
        self.shape = base.shape
        self._layers: Dict[int, Dict[str, np.ndarray]] = {}

    @property
    def embed(self):
        return self.base.embed

    @property
    def final_norm(self):
        return self.base.final_norm

    def layer(self, i: int) -> Dict[str, np.ndarray]:
        if i not in self._layers:
            d = dict(self.base.layer(i))
            for name in QUANT_TENSORS:
                d[name] = dequantize(*quantize(d[name], self.nbits))
            self._layers[i] = d
        return self._layers[i]
