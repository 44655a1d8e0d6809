"""Seeded synthetic inputs for the Qwen3-style decoder: weights, token ids, lengths, KV fills.

This module is shared by the CUDA path's callers (tests, bench) and by the CPU oracle. It
holds none of the decoder's arithmetic: it only draws random numbers and rounds them to the
storage formats the decoder consumes (bf16 bit patterns, int32 ids).

Recipes (all seeded, all reproducible):

* Weights: every tensor of the Qwen3 layout gets its own generator,
  ``numpy.random.default_rng(SeedSequence([seed, group, index]))`` (PCG64), so any layer can
  be drawn without drawing the others. Matrices are ``0.02 * N(0, 1)``, norm weights are
  ``1 + 0.02 * N(0, 1)``; the normal draws are float32 and the scaling is done in float32,
  then the value is rounded to bf16 (round to nearest even).
* Token ids: uniform integers in ``[0, vocab)``.
* Cached lengths of the long-context workload: uniform integers in ``[lo, hi]``.
* Injected KV-cache contents: the counter-based SplitMix64 generator (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014) hashed over the element
  index. The top byte of each 64-bit output, read as a signed int8 ``b``, gives
  ``K = b / 64`` and ``V = b / 128``. Both are exact in fp16 (and bf16), so a device-side fill that
  implements the same published generator produces bit-identical values.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Iterable, Optional

import numpy as np

# ----------------------------------------------------------------------------------------
# Model shape presets (dimensions printed on the page "Dentro de un LLM: Inferencia en
# Python puro para Qwen3-0.6B en MLX": Paso 2 vocab/hidden, Paso 5 heads, Paso 6 FFN,
# Paso 7 layer count, Paso 3 EPS, Paso 4 THETA).
# ----------------------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Shape:
    n_layers: int = 28
    hidden: int = 1024
    n_heads: int = 16
    n_kv_heads: int = 8
    head_dim: int = 128
    inter: int = 3072
    vocab: int = 151936
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    page_size: int = 16


QWEN3_0_6B = Shape()
ONE_BLOCK = dataclasses.replace(QWEN3_0_6B, n_layers=1)
# A tiny shape with the same structure (GQA ratio 2, rotate-half RoPE) for CPU-only tests.
TINY = Shape(n_layers=2, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, inter=96,
             vocab=512, rms_eps=1e-6, rope_theta=1e6, page_size=4)

# The five-token prompt printed on the page (Paso 1).
PAGE_PROMPT = (785, 6722, 315, 9625, 374)

LAYER_TENSORS = (
    "input_layernorm.weight",
    "self_attn.q_proj.weight",
    "self_attn.k_proj.weight",
    "self_attn.v_proj.weight",
    "self_attn.o_proj.weight",
    "self_attn.q_norm.weight",
    "self_attn.k_norm.weight",
    "post_attention_layernorm.weight",
    "mlp.gate_proj.weight",
    "mlp.up_proj.weight",
    "mlp.down_proj.weight",
)


def layer_tensor_shapes(s: Shape) -> Dict[str, tuple]:
    qd, kd = s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
    return {
        "input_layernorm.weight": (s.hidden,),
        "self_attn.q_proj.weight": (qd, s.hidden),
        "self_attn.k_proj.weight": (kd, s.hidden),
        "self_attn.v_proj.weight": (kd, s.hidden),
        "self_attn.o_proj.weight": (s.hidden, qd),
        "self_attn.q_norm.weight": (s.head_dim,),
        "self_attn.k_norm.weight": (s.head_dim,),
        "post_attention_layernorm.weight": (s.hidden,),
        "mlp.gate_proj.weight": (s.inter, s.hidden),
        "mlp.up_proj.weight": (s.inter, s.hidden),
        "mlp.down_proj.weight": (s.hidden, s.inter),
    }


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK = 1 << 22


def _draw(seed: int, group: int, index: int, shape, is_norm: bool) -> np.ndarray:
    """Draws the tensor's normals in consecutive chunks of one stream (identical to a single
    draw of the whole tensor) into reused buffers, then rounds each chunk to bf16."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, group, index]))
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    buf = np.empty(min(n, _CHUNK), dtype=np.float32)
    u = buf.view(np.uint32)
    tmp = np.empty_like(u)
    for a in range(0, n, _CHUNK):
        m = min(_CHUNK, n - a)
        z, uu, tt = buf[:m], u[:m], tmp[:m]
        rng.standard_normal(out=z, dtype=np.float32)
        z *= np.float32(0.02)
        if is_norm:
            z += np.float32(1.0)
        # round to nearest even on the upper 16 bits
        np.right_shift(uu, np.uint32(16), out=tt)
        tt &= np.uint32(1)
        tt += np.uint32(0x7FFF)
        uu += tt
        uu >>= np.uint32(16)
        out[a:a + m] = uu
    return out.reshape(shape)


def make_layer(s: Shape, layer: int, seed: int = 0) -> Dict[str, np.ndarray]:
    """bf16 bits (uint16) of one decoder layer, keyed by the HF tensor name suffix."""
    shapes = layer_tensor_shapes(s)
    out = {}
    for idx, name in enumerate(LAYER_TENSORS):
        out[name] = _draw(seed, 1 + layer, idx, shapes[name], name.endswith("norm.weight"))
    return out


def make_embedding(s: Shape, seed: int = 0) -> np.ndarray:
    """bf16 bits [vocab, hidden] of model.embed_tokens.weight (also the tied LM head)."""
    return _draw(seed, 0, 0, (s.vocab, s.hidden), False)


def make_final_norm(s: Shape, seed: int = 0) -> np.ndarray:
    return _draw(seed, 0, 1, (s.hidden,), True)


class Weights:
    """Lazily drawn bf16 weights of a whole model, HF names, [out, in] layout."""

    def __init__(self, s: Shape, seed: int = 0):
        self.shape = s
        self.seed = seed
        self._layers: Dict[int, Dict[str, np.ndarray]] = {}
        self._embed: Optional[np.ndarray] = None
        self._norm: Optional[np.ndarray] = None

    @property
    def embed(self) -> np.ndarray:
        if self._embed is None:
            self._embed = make_embedding(self.shape, self.seed)
        return self._embed

    @property
    def final_norm(self) -> np.ndarray:
        if self._norm is None:
            self._norm = make_final_norm(self.shape, self.seed)
        return self._norm

    def layer(self, i: int) -> Dict[str, np.ndarray]:
        if i not in self._layers:
            self._layers[i] = make_layer(self.shape, i, self.seed)
        return self._layers[i]

    def named(self) -> Iterable[tuple]:
        """(HF name, bf16 bits) for every tensor, in the fixed layout order."""
        yield "model.embed_tokens.weight", self.embed
        for i in range(self.shape.n_layers):
            for name in LAYER_TENSORS:
                yield f"model.layers.{i}.{name}", self.layer(i)[name]
        yield "model.norm.weight", self.final_norm


def make_tokens(vocab: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed]))
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def make_lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi, size=n, endpoint=True).astype(np.int64)


# ----------------------------------------------------------------------------------------
# Counter-based KV fill (SplitMix64).
# ----------------------------------------------------------------------------------------

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Element index of the injected cache, independent of any capacity:
#   idx = (((layer * 2 + which) * 2**22 + pos) * n_kv_heads + head) * head_dim + dim
POS_BITS = 22


def splitmix64(counter: np.ndarray, seed: int) -> np.ndarray:
    """SplitMix64 output for state ``seed + (counter + 1) * golden`` (uint64, wrapping)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (counter.astype(np.uint64) + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def kv_fill_values(seed: int, layer: int, which: int, positions: np.ndarray,
                   n_kv_heads: int, head_dim: int) -> np.ndarray:
    """Injected K (which=0) or V (which=1) values, float32 [n_kv_heads, len(positions), head_dim]."""
    pos = np.asarray(positions, dtype=np.uint64)
    h = np.arange(n_kv_heads, dtype=np.uint64)
    d = np.arange(head_dim, dtype=np.uint64)
    base = (np.uint64(layer * 2 + which) << np.uint64(POS_BITS)) + pos        # [n]
    idx = ((base[None, :, None] * np.uint64(n_kv_heads) + h[:, None, None])
           * np.uint64(head_dim) + d[None, None, :])
    b = (splitmix64(idx, seed) >> np.uint64(56)).astype(np.uint8).view(np.int8)
    scale = np.float32(1.0 / 64.0) if which == 0 else np.float32(1.0 / 128.0)
    return b.astype(np.float32) * scale
