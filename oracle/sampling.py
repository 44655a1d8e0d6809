"""fp64 oracle of temperature + top-p (nucleus) sampling.

TEST INFRASTRUCTURE ONLY (see the package docstring): plain NumPy in float64. It restates
the ``sample`` step of Paso 8 of the page "Dentro de un LLM: Inferencia en Python puro para
Qwen3-0.6B en MLX": divide the logits by the temperature, softmax, sort the probabilities in
descending order, keep the prefix whose length is one more than the number of running sums
below ``top_p``, renormalise, draw one token.

Readings taken where the page is silent or cannot be reproduced:

* ``temperature == 0`` is greedy ``argmax`` with ties to the lowest index (as the rest of the
  oracle).
* ``argsort(-probs)`` names no order for equal probabilities; equal probabilities are ordered
  by ascending token id, so the nucleus keeps the lowest ids among ties at its edge.
* The cutoff ``#(cumsum < top_p) + 1`` can exceed the vocabulary when rounding keeps every
  running sum below ``top_p``; the slice then keeps every token, as the page's slicing does.
* The page draws with ``mx.random.categorical`` over the kept log-probabilities, i.e. from
  MLX's own generator, which cannot be reproduced. Here the draw is an inverse CDF of a
  uniform ``u`` in [0, 1) that the caller supplies: the kept tokens are enumerated in
  ascending token id, and the chosen token is the first whose running renormalised
  probability exceeds ``u``. This samples the same categorical distribution; fixing the
  enumeration order makes the token a function of ``u`` that another implementation can
  reproduce.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np


def softmax_t(logits: np.ndarray, temperature: float) -> np.ndarray:
    """Paso 8: ``softmax(logits / temperature)`` in float64."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def nucleus(probs: np.ndarray, top_p: float) -> Tuple[np.ndarray, np.ndarray]:
    """Paso 8 (top-p): token ids of the kept prefix (in descending probability, ties by
    ascending id) and their probabilities, before renormalisation."""
    probs = np.asarray(probs, dtype=np.float64)
    order = np.lexsort((np.arange(probs.size), -probs))  # primary key: -p; then the id
    sorted_p = probs[order]
    cumsum = np.cumsum(sorted_p)
    cutoff = min(int(np.sum(cumsum < top_p)) + 1, probs.size)
    return order[:cutoff], sorted_p[:cutoff]


def kept_cdf(logits: np.ndarray, temperature: float, top_p: float) -> Tuple[np.ndarray, np.ndarray]:
    """The kept token ids in ascending id order and the running sums of their renormalised
    probabilities (the inverse-CDF table of the draw)."""
    p = softmax_t(logits, temperature)
    kept, _ = nucleus(p, top_p)
    ids = np.sort(kept)
    w = p[ids] / p[ids].sum()
    return ids, np.cumsum(w)


def sample(logits: np.ndarray, temperature: float, top_p: float, u: float) -> int:
    """Paso 8: one token id for one row of logits and one uniform ``u`` in [0, 1)."""
    logits = np.asarray(logits)
    if temperature == 0:
        m = logits.max()
        return int(np.flatnonzero(logits == m)[0])
    ids, c = kept_cdf(logits, temperature, top_p)
    i = int(np.searchsorted(c, u, side="right"))  # first running sum > u
    return int(ids[min(i, ids.size - 1)])
