"""fp64 oracle of the Qwen3-style decoder forward pass.

TEST INFRASTRUCTURE ONLY (see the package docstring): plain NumPy in float64 over the same
bf16-rounded weights the CUDA library gets (widened exactly), with no intermediate rounding,
no blocking and no fusion. Each function cites the step of the page "Dentro de un LLM:
Inferencia en Python puro para Qwen3-0.6B en MLX" that it restates.

Readings taken where the page is silent or ambiguous:

* ``forward`` is called but never printed (Paso 9): embedding gather (Paso 2), the blocks of
  Paso 7, final norm and LM head (Paso 8). Positions are ``start + arange(n)``.
* The causal mask (Paso 5) is written for an empty cache; it is generalised to "key visible
  iff its position <= the query's position", which equals the page's mask whenever the
  cache is empty and adds no mask for a single decode token, as the page says.
* The masked scores get ``-1e9`` added as on the page; in float64 ``exp`` of such a score
  underflows to exactly zero.
* GQA uses ``repeat`` along the head axis (Paso 5), so query head ``h`` reads KV head
  ``h // (n_heads / n_kv_heads)``.
* RoPE pairs dimension ``i`` with ``i + head_dim/2`` (rotate-half, Paso 4); the frequencies,
  angles, cos and sin are evaluated in float64 here (the page's MLX code uses float32).
* QK-norm weights (Paso 5) have ``head_dim`` entries shared by all heads of a projection.
* The LM head is tied to the embedding matrix; only the last position of a prefill is
  projected, as only ``logits[-1]`` is consumed (Pasos 8-9).
* Greedy sampling is ``argmax``; ties go to the lowest index.
"""

from __future__ import annotations

import dataclasses
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np


def _widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly; float arrays (e.g. dequantized
    weights) are taken as they are."""
    if np.asarray(bits).dtype.kind == "f":
        return np.asarray(bits, dtype=np.float64)
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------------------
# Operators
# ----------------------------------------------------------------------------------------


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Paso 3: divide by the root of the mean square over the last axis (plus EPS inside the
    root), then scale per feature. No mean subtraction, no bias."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_angles(positions: Sequence[int], head_dim: int, theta: float) -> np.ndarray:
    """Paso 4: angle[p, i] = position_p * theta ** (-i / half), i < half = head_dim / 2."""
    half = head_dim // 2
    inv_freq = 1.0 / (float(theta) ** (np.arange(half, dtype=np.float64) / half))
    return np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]


def apply_rope(x: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Paso 4: rotate each pair (x[i], x[i + half]) by angle[:, i] (rotate-half layout).

    ``x`` is [..., n, head_dim]; ``angles`` is [n, half]."""
    half = x.shape[-1] // 2
    c, s = np.cos(angles), np.sin(angles)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    """Paso 6: SiLU(x) = x * sigmoid(x)."""
    with np.errstate(over="ignore"):
        return x * (1.0 / (1.0 + np.exp(-x)))


def gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
                  k_pos: np.ndarray, return_probs: bool = False):
    """Paso 5: grouped-query causal attention.

    q: [Hq, nq, d]; k, v: [Hkv, nk, d]; positions give the causal rule. Returns
    out [Hq, nq, d] (and the softmax probabilities [Hq, nq, nk] when asked)."""
    hq, hkv, d = q.shape[0], k.shape[0], q.shape[-1]
    group = hq // hkv
    k_rep = np.repeat(k, group, axis=0)            # head h -> KV head h // group
    v_rep = np.repeat(v, group, axis=0)
    scores = (q @ k_rep.transpose(0, 2, 1)) * (d ** -0.5)
    future = np.asarray(k_pos)[None, :] > np.asarray(q_pos)[:, None]
    if future.any():
        scores = scores + np.where(future, -1e9, 0.0)[None, :, :]
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    probs = e / e.sum(axis=-1, keepdims=True)
    out = probs @ v_rep
    return (out, probs) if return_probs else out


def ffn(h: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """Paso 6: (SiLU(h Wg^T) * (h Wu^T)) Wd^T."""
    return (silu(h @ wg.T) * (h @ wu.T)) @ wd.T


def argmax_lowest(logits: np.ndarray) -> int:
    """Paso 8 greedy pick; on ties the lowest index wins (np.argmax returns the first)."""
    return int(np.argmax(logits))


# ----------------------------------------------------------------------------------------
# Model state
# ----------------------------------------------------------------------------------------


@dataclasses.dataclass
class LayerW:
    in_norm: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    q_norm: np.ndarray
    k_norm: np.ndarray
    post_norm: np.ndarray
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray


class Model:
    """fp64 view of a weight provider (any object with ``shape``, ``embed``, ``final_norm``
    and ``layer(i)`` returning bf16 bits keyed by HF suffix names)."""

    def __init__(self, weights, keep_layers: bool = True):
        self.src = weights
        self.s = weights.shape
        self.keep = keep_layers
        self._layers: Dict[int, LayerW] = {}
        self._embed32: Optional[np.ndarray] = None

    def layer(self, i: int) -> LayerW:
        if i in self._layers:
            return self._layers[i]
        b = self.src.layer(i)
        lw = LayerW(
            in_norm=_widen(b["input_layernorm.weight"]),
            wq=_widen(b["self_attn.q_proj.weight"]),
            wk=_widen(b["self_attn.k_proj.weight"]),
            wv=_widen(b["self_attn.v_proj.weight"]),
            wo=_widen(b["self_attn.o_proj.weight"]),
            q_norm=_widen(b["self_attn.q_norm.weight"]),
            k_norm=_widen(b["self_attn.k_norm.weight"]),
            post_norm=_widen(b["post_attention_layernorm.weight"]),
            wg=_widen(b["mlp.gate_proj.weight"]),
            wu=_widen(b["mlp.up_proj.weight"]),
            wd=_widen(b["mlp.down_proj.weight"]),
        )
        if self.keep:
            self._layers[i] = lw
        return lw

    @property
    def embed32(self) -> np.ndarray:
        """The embedding as float32 (exact widening of bf16; saves half the memory of fp64)."""
        if self._embed32 is None:
            u = self.src.embed.astype(np.uint32) << np.uint32(16)
            self._embed32 = u.view(np.float32)
        return self._embed32

    def embed_rows(self, ids: Sequence[int]) -> np.ndarray:
        """Paso 2: x = E[ids]."""
        return self.embed32[np.asarray(ids, dtype=np.int64)].astype(np.float64)

    def lm_head(self, h: np.ndarray, chunk: int = 16384) -> np.ndarray:
        """Paso 8 with the LM head tied to E: logits = h E^T. h is [n, D] -> [n, V]."""
        e = self.embed32
        out = np.empty((h.shape[0], e.shape[0]), dtype=np.float64)
        for a in range(0, e.shape[0], chunk):
            out[:, a:a + chunk] = h @ e[a:a + chunk].astype(np.float64).T
        return out


class SeqCache:
    """Per-sequence KV cache of Paso 5: per layer K and V as [Hkv, n, d] in float64.

    ``prior`` optionally supplies an injected prefix for layer i as (K, V) arrays of length
    ``prior_len``; it is called lazily so that a long injected cache never has to be held for
    all layers at once."""

    def __init__(self, n_layers: int, prior: Optional[Callable[[int], Tuple[np.ndarray, np.ndarray]]] = None,
                 prior_len: int = 0):
        self.n_layers = n_layers
        self.k: List[Optional[np.ndarray]] = [None] * n_layers
        self.v: List[Optional[np.ndarray]] = [None] * n_layers
        self.prior = prior
        self.prior_len = prior_len if prior is not None else 0
        self.new_len = 0

    @property
    def length(self) -> int:
        return self.prior_len + self.new_len

    def get(self, layer: int):
        k, v = self.k[layer], self.v[layer]
        if self.prior is not None:
            pk, pv = self.prior(layer)
            if k is None:
                return pk, pv
            return np.concatenate([pk, k], axis=1), np.concatenate([pv, v], axis=1)
        return k, v

    def append(self, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        """Paso 5 (KV cache): concatenate the new keys/values along the sequence axis."""
        if self.k[layer] is None:
            self.k[layer], self.v[layer] = k, v
        else:
            self.k[layer] = np.concatenate([self.k[layer], k], axis=1)
            self.v[layer] = np.concatenate([self.v[layer], v], axis=1)


# ----------------------------------------------------------------------------------------
# Block and forward
# ----------------------------------------------------------------------------------------


def attention_sublayer(h: np.ndarray, lw: LayerW, s, cache: SeqCache, layer: int,
                       positions: np.ndarray, taps: Optional[dict] = None) -> np.ndarray:
    """Paso 5: projections, head split, QK-norm, RoPE, cache append, GQA attention, o_proj."""
    n = h.shape[0]
    q = (h @ lw.wq.T).reshape(n, s.n_heads, s.head_dim).transpose(1, 0, 2)
    k = (h @ lw.wk.T).reshape(n, s.n_kv_heads, s.head_dim).transpose(1, 0, 2)
    v = (h @ lw.wv.T).reshape(n, s.n_kv_heads, s.head_dim).transpose(1, 0, 2)
    q = rms_norm(q, lw.q_norm, s.rms_eps)
    k = rms_norm(k, lw.k_norm, s.rms_eps)
    ang = rope_angles(positions, s.head_dim, s.rope_theta)
    q = apply_rope(q, ang)
    k = apply_rope(k, ang)
    if taps is not None:
        taps.setdefault("q", []).append(q)
        taps.setdefault("k", []).append(k)
        taps.setdefault("v", []).append(v)
    prev_len = cache.length
    cache.append(layer, k, v)
    k_all, v_all = cache.get(layer)
    k_pos = np.arange(prev_len + n)
    o = gqa_attention(q, k_all, v_all, positions, k_pos)
    o = o.transpose(1, 0, 2).reshape(n, s.n_heads * s.head_dim)
    if taps is not None:
        taps.setdefault("attn", []).append(o)
    return o @ lw.wo.T


def decoder_layer(x: np.ndarray, lw: LayerW, s, cache: SeqCache, layer: int,
                  positions: np.ndarray, taps: Optional[dict] = None) -> np.ndarray:
    """Paso 7: x += attention(rms_norm(x)); x += ffn(rms_norm(x))."""
    h = rms_norm(x, lw.in_norm, s.rms_eps)
    x = x + attention_sublayer(h, lw, s, cache, layer, positions, taps)
    h = rms_norm(x, lw.post_norm, s.rms_eps)
    return x + ffn(h, lw.wg, lw.wu, lw.wd)


def forward(model: Model, ids: Sequence[int], cache: SeqCache, all_logits: bool = False,
            taps: Optional[dict] = None) -> dict:
    """``forward(ids, cache, start)`` of Paso 9, with start = the cache's current length.

    Returns ``logits`` ([V] for the last position, or [n, V] with ``all_logits``),
    ``hidden`` ([n_layers, n, D], the residual stream after each layer) and ``positions``."""
    s = model.s
    start = cache.length
    positions = np.arange(start, start + len(ids))
    x = model.embed_rows(ids)
    hidden = np.empty((s.n_layers, len(ids), s.hidden))
    for i in range(s.n_layers):
        x = decoder_layer(x, model.layer(i), s, cache, i, positions, taps)
        hidden[i] = x
    cache.new_len += len(ids)
    fin = _widen(model.src.final_norm)
    rows = x if all_logits else x[-1:]
    logits = model.lm_head(rms_norm(rows, fin, s.rms_eps))
    return {"logits": logits if all_logits else logits[0], "hidden": hidden,
            "positions": positions}


def generate(model: Model, prompt: Sequence[int], n_decode: int, cache: Optional[SeqCache] = None,
             keep_hidden: bool = True, eos_id: Optional[int] = None) -> dict:
    """Paso 9 at temperature 0: prefill the prompt, then up to ``n_decode`` single-token
    steps, each fed the previous greedy pick. With ``eos_id`` (the page leaves EOS_ID
    undefined, so it is the caller's): as in the page's loop, a pick equal to it is kept as
    the last output and never fed, so the cache ends with the picks before it.

    Returns ``ids`` (the generated ids: n_decode + 1 without a stop), ``logits`` per step and,
    with ``keep_hidden``, per-step hidden states."""
    cache = cache if cache is not None else SeqCache(model.s.n_layers)
    out = forward(model, list(prompt), cache)
    ids = [argmax_lowest(out["logits"])]
    logits = [out["logits"]]
    hidden = [out["hidden"]] if keep_hidden else None
    for _ in range(n_decode):
        if eos_id is not None and ids[-1] == eos_id:
            break
        out = forward(model, [ids[-1]], cache)
        ids.append(argmax_lowest(out["logits"]))
        logits.append(out["logits"])
        if keep_hidden:
            hidden.append(out["hidden"])
    return {"ids": ids, "logits": np.stack(logits), "hidden": hidden}


# ----------------------------------------------------------------------------------------
# Paged KV allocator mirror
# ----------------------------------------------------------------------------------------


class PagedKVMirror:
    """Mirror of the paged KV allocator (pages of ``page_size`` tokens).

    Reading: a reservation takes pages from the free list lowest id first, in the order of
    the calls; position p of a sequence lives in slot page_table[p // page_size] * page_size
    + p % page_size. A reset returns the sequence's pages to the free list."""

    def __init__(self, n_pages: int, max_seqs: int, page_size: int):
        self.page_size = page_size
        self.free = list(range(n_pages))
        self.tables: Dict[int, List[int]] = {i: [] for i in range(max_seqs)}
        self.lengths: Dict[int, int] = {i: 0 for i in range(max_seqs)}

    def reserve(self, seq: int, total_tokens: int) -> bool:
        need = -(-total_tokens // self.page_size) - len(self.tables[seq])
        if need <= 0:
            return True
        if need > len(self.free):
            return False
        self.free.sort()
        take, self.free = self.free[:need], self.free[need:]
        self.tables[seq].extend(take)
        return True

    def reset(self, seq: int) -> None:
        self.free.extend(self.tables[seq])
        self.tables[seq] = []
        self.lengths[seq] = 0

    def slots(self, seq: int, positions: Sequence[int]) -> np.ndarray:
        t = self.tables[seq]
        return np.array([t[p // self.page_size] * self.page_size + p % self.page_size
                         for p in positions], dtype=np.int64)
