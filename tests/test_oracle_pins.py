"""Pins of the fp64 oracle against what the page and mathematics fix (CPU only).

Each test pins one operator to something other than the oracle itself: a closed form, an
invariant the page states, a brute-force loop on a tiny input, or a library routine of a
different library (torch, CPU, float64). Together they are chosen so that a plausible slip
in the oracle (a dropped term, a wrong sign or index, a transposed operand, swapped weights)
fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle.qwen3 import LayerW, SeqCache, attention_sublayer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


# ------------------------------------------------------------------ page constants -----

def test_presets_match_page_constants():
    g = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    s = synth.QWEN3_0_6B
    assert tuple(g["prompt_ids"]) == synth.PAGE_PROMPT
    for key in ("vocab", "hidden", "n_heads", "n_kv_heads", "head_dim", "inter", "n_layers"):
        assert getattr(s, key) == g[key], key
    assert s.rms_eps == g["rms_eps"] and s.rope_theta == g["rope_theta"]
    assert s.head_dim // 2 == g["rope_half"]
    assert s.n_heads * s.head_dim == 2048          # q projection width printed in Paso 5
    assert s.n_heads // s.n_kv_heads == 2          # "each KV head serves two query heads"


# ----------------------------------------------------------------------- RMSNorm --------

def test_rmsnorm_constant_vector_closed_form():
    # x = c * 1: mean square c^2, so out = c / sqrt(c^2 + eps) * w. With c = 1e-3 and
    # eps = 1e-6 this is 1/sqrt(2) - sensitive to where EPS sits.
    x = np.full((3, 8), 1e-3)
    w = np.linspace(0.5, 2.0, 8)
    out = oracle.rms_norm(x, w, 1e-6)
    np.testing.assert_allclose(out, np.broadcast_to(w / math.sqrt(2.0), (3, 8)), rtol=1e-14)


def test_rmsnorm_unit_rms_before_weight():
    x = RNG.standard_normal((5, 64)) * 3.0
    out = oracle.rms_norm(x, np.ones(64), 1e-6)
    ms = np.mean(x * x, axis=-1)
    rms_out = np.sqrt(np.mean(out * out, axis=-1))
    np.testing.assert_allclose(rms_out, np.sqrt(ms / (ms + 1e-6)), rtol=1e-13)
    # no mean subtraction (unlike LayerNorm): a constant row keeps its sign and size
    assert np.all(oracle.rms_norm(np.full((1, 4), 5.0), np.ones(4), 1e-6) > 0.99)


def test_rmsnorm_vs_torch():
    x = RNG.standard_normal((7, 33))
    w = RNG.standard_normal(33)
    ref = F.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, w, 1e-6), ref, rtol=1e-12, atol=1e-14)


# -------------------------------------------------------------------------- RoPE --------

def test_rope_position_zero_is_identity():
    x = RNG.standard_normal((2, 3, 16))
    ang = oracle.rope_angles([0, 0, 0], 16, 1e6)
    np.testing.assert_array_equal(oracle.apply_rope(x, ang), x)


def test_rope_rotate_half_pairing_and_sign():
    d, half = 128, 64
    for p in (1, 7, 1000):
        e0 = np.zeros((1, d)); e0[0, 0] = 1.0
        out = oracle.apply_rope(e0, oracle.rope_angles([p], d, 1e6))[0]
        # dim 0 pairs with dim 64 (not dim 1), and rotates counter-clockwise by p rad
        assert out[0] == pytest.approx(math.cos(p), abs=1e-15)
        assert out[half] == pytest.approx(math.sin(p), abs=1e-15)
        assert np.count_nonzero(np.abs(out) > 1e-15) <= 2
        eh = np.zeros((1, d)); eh[0, half] = 1.0
        out = oracle.apply_rope(eh, oracle.rope_angles([p], d, 1e6))[0]
        assert out[0] == pytest.approx(-math.sin(p), abs=1e-15)
        assert out[half] == pytest.approx(math.cos(p), abs=1e-15)


def test_rope_frequencies():
    # pair i turns by theta^(-i/64) per position; i = 32 gives 1e6^(-1/2) = 1e-3 rad
    ang = oracle.rope_angles([1, 2], 128, 1e6)
    assert ang[0, 0] == 1.0
    assert ang[0, 32] == pytest.approx(1e-3, rel=1e-14)
    assert ang[1, 32] == pytest.approx(2e-3, rel=1e-14)
    assert ang[0, 63] == pytest.approx(1e6 ** (-63 / 64), rel=1e-14)
    e = np.zeros((1, 128)); e[0, 32] = 1.0
    out = oracle.apply_rope(e, oracle.rope_angles([1], 128, 1e6))[0]
    assert out[32] == pytest.approx(0.9999995000000417, abs=1e-16)   # cos(0.001)
    assert out[96] == pytest.approx(0.0009999998333333417, abs=1e-18)  # sin(0.001)


def test_rope_norm_and_relative_position():
    d = 128
    q = RNG.standard_normal((1, d)); k = RNG.standard_normal((1, d))
    rot = lambda v, p: oracle.apply_rope(v, oracle.rope_angles([p], d, 1e6))[0]
    for p in (0, 5, 12345):
        r = rot(q, p)
        pair = lambda v: v[:64] ** 2 + v[64:] ** 2
        np.testing.assert_allclose(pair(r), pair(q[0]), rtol=1e-12)
    for m, n, sft in ((3, 1, 10), (100, 40, 977), (0, 7, 32000)):
        a = rot(q, m) @ rot(k, n)
        b = rot(q, m + sft) @ rot(k, n + sft)
        assert a == pytest.approx(b, rel=1e-9, abs=1e-9)
    # composition R_a R_b = R_{a+b}
    np.testing.assert_allclose(rot(rot(q, 11)[None], 31), rot(q, 42), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------- SiLU / FFN --------

def test_silu_closed_forms_and_torch():
    assert oracle.silu(np.array(0.0)) == 0.0
    assert oracle.silu(np.array(40.0)) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.silu(np.array(-40.0))) < 1e-15
    assert oracle.silu(np.array(1.0)) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    x = RNG.standard_normal(100) * 5
    np.testing.assert_allclose(oracle.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-13)


def test_ffn_scalar_closed_form():
    # D = I = 1: out = silu(a g) * (a u) * w; swapping gate and up would give silu(a u)(a g)
    a, g, u, w = 0.7, 1.9, -0.4, 1.3
    out = oracle.ffn(np.array([[a]]), np.array([[g]]), np.array([[u]]), np.array([[w]]))
    x = a * g
    assert out[0, 0] == pytest.approx(x / (1 + math.exp(-x)) * (a * u) * w, rel=1e-14)


# -------------------------------------------------------------------- attention -------

def _brute_attention(q, k, v, q_pos, k_pos):
    """Scalar loops: one query head at a time, its KV head = h // group (Paso 5)."""
    hq, nq, d = q.shape
    hkv, nk, _ = k.shape
    group = hq // hkv
    out = np.zeros((hq, nq, d))
    for h in range(hq):
        kh = h // group
        for i in range(nq):
            vis = [j for j in range(nk) if k_pos[j] <= q_pos[i]]
            sc = [math.fsum(q[h, i, t] * k[kh, j, t] for t in range(d)) / math.sqrt(d) for j in vis]
            m = max(sc)
            ex = [math.exp(s - m) for s in sc]
            z = math.fsum(ex)
            for t in range(d):
                out[h, i, t] = math.fsum(ex[a] / z * v[kh, j, t] for a, j in enumerate(vis))
    return out


def test_attention_brute_force_tiny():
    for (hq, hkv, nq, nk, d) in ((4, 2, 3, 3, 4), (4, 2, 1, 6, 8), (2, 1, 2, 5, 4), (6, 3, 4, 7, 2)):
        q = RNG.standard_normal((hq, nq, d)); k = RNG.standard_normal((hkv, nk, d))
        v = RNG.standard_normal((hkv, nk, d))
        q_pos = np.arange(nk - nq, nk); k_pos = np.arange(nk)
        np.testing.assert_allclose(oracle.gqa_attention(q, k, v, q_pos, k_pos),
                                   _brute_attention(q, k, v, q_pos, k_pos), rtol=1e-12, atol=1e-14)


def test_attention_vs_torch_sdpa_gqa_causal():
    hq, hkv, n, d = 16, 8, 9, 128
    q = RNG.standard_normal((hq, n, d)); k = RNG.standard_normal((hkv, n, d))
    v = RNG.standard_normal((hkv, n, d))
    pos = np.arange(n)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None], torch.from_numpy(k)[None],
                                         torch.from_numpy(v)[None], is_causal=True,
                                         enable_gqa=True)[0].numpy()
    np.testing.assert_allclose(oracle.gqa_attention(q, k, v, pos, pos), ref, rtol=1e-11, atol=1e-13)
    # GQA equals MHA with every KV head repeated for its two query heads (not tiled)
    kr = torch.from_numpy(k).repeat_interleave(2, dim=0)[None]
    vr = torch.from_numpy(v).repeat_interleave(2, dim=0)[None]
    mha = F.scaled_dot_product_attention(torch.from_numpy(q)[None], kr, vr, is_causal=True)[0]
    np.testing.assert_allclose(oracle.gqa_attention(q, k, v, pos, pos), mha.numpy(), rtol=1e-11,
                               atol=1e-13)


def test_attention_softmax_rows_and_future_zero():
    q = RNG.standard_normal((4, 6, 16)); k = RNG.standard_normal((2, 6, 16))
    v = RNG.standard_normal((2, 6, 16)); pos = np.arange(6)
    out, p = oracle.gqa_attention(q, k, v, pos, pos, return_probs=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)
    future = np.triu(np.ones((6, 6), bool), k=1)
    assert np.all(p[:, future] == 0.0)          # exactly zero weight on future keys
    # the first token sees only itself: output equals its value vector exactly
    np.testing.assert_allclose(out[:, 0], np.repeat(v[:, 0], 2, axis=0), rtol=0, atol=1e-15)


def test_attention_equal_keys_average_values():
    k = np.tile(RNG.standard_normal((2, 1, 8)), (1, 5, 1))
    v = RNG.standard_normal((2, 5, 8)); q = RNG.standard_normal((4, 5, 8)); pos = np.arange(5)
    out = oracle.gqa_attention(q, k, v, pos, pos)
    for i in range(5):
        np.testing.assert_allclose(out[:, i], np.repeat(v[:, :i + 1].mean(1), 2, axis=0), rtol=1e-13)


def test_attention_permutation_equivariant_without_positions():
    # with no mask (all positions equal) and no rotation, permuting tokens permutes outputs
    q = RNG.standard_normal((4, 6, 8)); k = RNG.standard_normal((2, 6, 8))
    v = RNG.standard_normal((2, 6, 8)); z = np.zeros(6)
    perm = RNG.permutation(6)
    a = oracle.gqa_attention(q, k, v, z, z)[:, perm]
    b = oracle.gqa_attention(q[:, perm], k[:, perm], v[:, perm], z, z)
    np.testing.assert_allclose(a, b, rtol=1e-12)


# ----------------------------------------------------------------- block structure -----

def _structured_layer(s, post_scale=2.0, qn=None):
    D, I = s.hidden, s.inter
    qd, kd = s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
    eye = lambda r, c: np.eye(r, c)
    return LayerW(in_norm=np.ones(D), wq=np.zeros((qd, D)), wk=np.zeros((kd, D)),
                  wv=eye(kd, D), wo=np.zeros((D, qd)),
                  q_norm=np.ones(s.head_dim) if qn is None else qn, k_norm=np.ones(s.head_dim),
                  post_norm=np.full(D, post_scale), wg=eye(I, D), wu=eye(I, D), wd=eye(D, I))


def test_block_ffn_uses_post_attention_norm():
    s = synth.TINY
    lw = _structured_layer(s)
    c = 10.0
    x = np.full((1, s.hidden), c)
    out = oracle.decoder_layer(x, lw, s, SeqCache(s.n_layers), 0, np.array([0]))
    h = 2.0 * c / math.sqrt(c * c + s.rms_eps)            # rms_norm(x) * post_norm
    expect = c + h / (1 + math.exp(-h)) * h                # + silu(h) * h through identities
    np.testing.assert_allclose(out, expect, rtol=1e-13)


def test_block_single_token_attention_is_value_path():
    # one token, empty cache: softmax over one key gives weight 1, so the attention output is
    # v of KV head h // 2 for query head h; o_proj then picks query heads 1 and 2.
    s = synth.TINY
    lw = _structured_layer(s, post_scale=0.0)
    lw.wd = np.zeros_like(lw.wd)
    d = s.head_dim
    wo = np.zeros((s.hidden, s.n_heads * d))
    wo[:d, d:2 * d] = np.eye(d)            # x[0:d]  += head 1 output (KV head 0)
    wo[d:2 * d, 2 * d:3 * d] = np.eye(d)   # x[d:2d] += head 2 output (KV head 1)
    lw.wo = wo
    x = RNG.standard_normal((1, s.hidden))
    out = oracle.decoder_layer(x, lw, s, SeqCache(s.n_layers), 0, np.array([0]))
    h = oracle.rms_norm(x, lw.in_norm, s.rms_eps)[0]
    expect = x[0].copy()
    expect[:d] += h[:d]            # v head 0 = h[0:d]   (wv = identity rows)
    expect[d:2 * d] += h[d:2 * d]  # v head 1 = h[d:2d]
    np.testing.assert_allclose(out[0], expect, rtol=1e-13, atol=1e-15)


def test_qk_norm_applied_before_rope():
    # q head 0 = e_0 direction; q_norm weight differs between dims 0 and half.
    s = synth.TINY
    d, half = s.head_dim, s.head_dim // 2
    qn = np.ones(d); qn[0], qn[half] = 3.0, 0.5
    lw = _structured_layer(s, qn=qn)
    lw.wq[0, :] = 1.0 / s.hidden
    x = np.full((1, s.hidden), 100.0)
    taps = {}
    p = 5
    cache = SeqCache(s.n_layers)
    attention_sublayer(oracle.rms_norm(x, lw.in_norm, s.rms_eps), lw, s, cache, 0,
                       np.array([p]), taps)
    q = taps["q"][0][0, 0]
    a = 100.0 / math.sqrt(1e4 + s.rms_eps)        # q head 0 before QK-norm: a * e_0
    r = a / math.sqrt(a * a / d + s.rms_eps)      # QK-norm of a * e_0 (before its weight)
    # norm first (weight 3 on dim 0), then rotate: (3r cos p, 3r sin p); the other order
    # would put weight 0.5 on the sin component.
    assert q[0] == pytest.approx(3.0 * r * math.cos(p), rel=1e-12)
    assert q[half] == pytest.approx(3.0 * r * math.sin(p), rel=1e-12)


# --------------------------------------------------------------- forward / LM head -----

class _ArrayWeights:
    def __init__(self, s, embed_bits, final_bits, layers):
        self.shape, self.embed, self.final_norm, self._layers = s, embed_bits, final_bits, layers

    def layer(self, i):
        return self._layers[i]


def _zero_layer_bits(s):
    shapes = synth.layer_tensor_shapes(s)
    one = synth.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    return {n: (np.full(sh, one, np.uint16) if n.endswith("norm.weight") else np.zeros(sh, np.uint16))
            for n, sh in shapes.items()}


def test_tied_lm_head_closed_form():
    # With o_proj = down_proj = 0 every block is the identity, so the last hidden state is
    # E[id]; logits[j] = rms_norm(E[id]) * 2 . E[j], and logits[id] = 2|e|^2 / sqrt(|e|^2/D + eps).
    s = synth.TINY
    emb = synth.make_embedding(s, 7)
    fin = synth.f32_to_bf16_bits(np.full(s.hidden, 2.0, np.float32))
    m = oracle.Model(_ArrayWeights(s, emb, fin, [_zero_layer_bits(s)] * s.n_layers))
    tok = 123
    out = oracle.forward(m, [5, tok], SeqCache(s.n_layers))
    e = synth.bf16_bits_to_f32(emb).astype(np.float64)
    n2 = float(e[tok] @ e[tok])
    assert out["logits"][tok] == pytest.approx(2 * n2 / math.sqrt(n2 / s.hidden + s.rms_eps), rel=1e-12)
    scale = 2.0 / math.sqrt(n2 / s.hidden + s.rms_eps)
    np.testing.assert_allclose(out["logits"], scale * (e @ e[tok]), rtol=1e-11, atol=1e-14)
    np.testing.assert_array_equal(out["hidden"][-1][1], e[tok])


def test_argmax_lowest_index_on_ties():
    l = np.array([0.1, 3.0, -1.0, 3.0, 2.9])
    assert oracle.argmax_lowest(l) == 1


@pytest.fixture(scope="module")
def tiny_model():
    return oracle.Model(synth.Weights(synth.TINY, seed=3))


def test_decode_with_cache_equals_full_recompute(tiny_model):
    s = synth.TINY
    prompt = synth.make_tokens(s.vocab, 6, 1).tolist()
    gen = oracle.generate(tiny_model, prompt, 5)
    for step in range(1, 6):
        seq = prompt + gen["ids"][:step]
        full = oracle.forward(tiny_model, seq, SeqCache(s.n_layers))
        np.testing.assert_allclose(gen["logits"][step], full["logits"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(gen["hidden"][step][:, -1], full["hidden"][:, -1], rtol=1e-10,
                                   atol=1e-12)


def test_chunked_forward_equals_token_by_token(tiny_model):
    s = synth.TINY
    toks = synth.make_tokens(s.vocab, 9, 2).tolist()
    c1 = SeqCache(s.n_layers)
    a = oracle.forward(tiny_model, toks[:4], c1)
    b = oracle.forward(tiny_model, toks[4:], c1, all_logits=True)
    c2 = SeqCache(s.n_layers)
    outs = [oracle.forward(tiny_model, [t], c2)["logits"] for t in toks]
    np.testing.assert_allclose(a["logits"], outs[3], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b["logits"], np.stack(outs[4:]), rtol=1e-10, atol=1e-12)


def test_generate_deterministic(tiny_model):
    p = synth.make_tokens(synth.TINY.vocab, 4, 9).tolist()
    a = oracle.generate(tiny_model, p, 4, keep_hidden=False)
    b = oracle.generate(tiny_model, p, 4, keep_hidden=False)
    assert a["ids"] == b["ids"]
    np.testing.assert_array_equal(a["logits"], b["logits"])


def test_generate_eos_stop_follows_the_page_loop(tiny_model):
    """Paso 9: a pick equal to EOS_ID ends the output (kept as its last id) and is never fed:
    the output is the no-stop run cut after the first EOS, and the cache holds the prompt and
    the picks before it."""
    s = synth.TINY
    p = synth.make_tokens(s.vocab, 5, 12).tolist()
    full = oracle.generate(tiny_model, p, 8, keep_hidden=False)["ids"]
    eos = full[3]
    k = full.index(eos)
    c = SeqCache(s.n_layers)
    got = oracle.generate(tiny_model, p, 8, cache=c, keep_hidden=False, eos_id=eos)["ids"]
    assert got == full[:k + 1]
    assert c.length == len(p) + k
    c2 = SeqCache(s.n_layers)
    never = oracle.generate(tiny_model, p, 8, cache=c2, keep_hidden=False, eos_id=s.vocab + 1)["ids"]
    assert never == full and c2.length == len(p) + 8


# ------------------------------------------------------------------- paged KV mirror ---

def test_paged_mirror_slots_and_lowest_first():
    m = oracle.PagedKVMirror(n_pages=10, max_seqs=4, page_size=16)
    assert m.reserve(2, 20)          # pages 0, 1
    assert m.reserve(0, 16)          # page 2
    assert m.reserve(2, 33)          # + page 3
    assert m.tables[2] == [0, 1, 3] and m.tables[0] == [2]
    np.testing.assert_array_equal(m.slots(2, [0, 15, 16, 31, 32]), [0, 15, 16, 31, 48])
    np.testing.assert_array_equal(m.slots(0, [0, 5]), [32, 37])
    m.reset(2)
    assert m.reserve(1, 40)          # lowest free first: 0, 1, 3
    assert m.tables[1] == [0, 1, 3]
    assert not m.reserve(3, 16 * 7)  # 6 free pages left, 7 needed: refused, nothing taken
    assert m.tables[3] == [] and len(m.free) == 6


# ------------------------------------------------------------------- synthetic inputs --

def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(vals))
    np.testing.assert_array_equal(got, [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0])
    x = RNG.standard_normal(1000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x)), ref)


def test_splitmix64_published_vectors():
    # SplitMix64 seeded with 1234567: the first outputs of the reference generator.
    got = synth.splitmix64(np.arange(3, dtype=np.uint64), 1234567)
    assert [int(v) for v in got] == [6457827717110365317, 3203168211198807973,
                                     9817491932198370423]
