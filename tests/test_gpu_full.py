"""GPU parity at the full sizes of the measured workloads, in the launch configuration that
bench.py times (same shapes, batch composition, input recipe and call sequence), checked on
sampled sequences that the oracle recomputes one by one:

  * batched decode: 64 sequences, 1024-token prompts prefilled 16 sequences per call, then
    4 greedy decode steps of all 64, through the two-stream split path (sequences 0-31 on one
    stream, 32-63 on the other) and again, from the same cache and with the same tokens,
    through the decode-step kernel (the same halves) -- sequences 0, 31, 32 and 63, the
    hidden state after every layer of every decode step, the logits and the ids;
  * prefill: 16 x 512 tokens in one call -- sequences 0 and 15 (every layer's hidden state,
    the final logits and ids), plus positions and KV slots of all 8192 tokens;
  * long-context ragged decode: 8 sequences with cached lengths drawn uniform in
    [1024, 32768] (seed 2000) and filled by the counter-based generator -- the shortest
    sequence end to end through 28 layers, and the longest through all 28 layers one layer at
    a time (the oracle's layer takes the GPU's input to that layer and the injected prefix of
    that layer).

Sequences never interact, so checking a subset of a batch is a valid check of the batch."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, check_hidden, check_logits, check_token, rel_err, HIDDEN_REL, weights

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

S = synth.QWEN3_0_6B


@pytest.fixture(scope="module")
def om():
    return oracle.Model(weights(S))


def _engine(pkg, **kw):
    return pkg.qw.Engine(S, dict(weights(S).named()), **kw)


def test_batched_decode_b64_full(qw, om):
    B, P, ND = 64, 1024, 4
    eng = _engine(qw, max_tokens=16 * P, max_batch=B, max_context=P + ND + 16,
                  kv_pages=B * ((P + ND + 15) // 16 + 1) + 8, max_seqs=B)
    try:
        run = Run(qw, eng)
        toks = synth.make_tokens(S.vocab, B * P, 1000 + 2).reshape(B, P)
        nxt = np.zeros(B, np.int64)
        logits = np.zeros((B, S.vocab))
        for a in range(0, B, 16):
            seqs = list(range(a, a + 16))
            g = run.prefill(seqs, [toks[b].tolist() for b in seqs], debug=False, reserve_extra=ND)
            nxt[a:a + 16] = g["next"]
            logits[a:a + 16] = g["logits"]
        sample = [0, 31, 32, 63]   # first and last sequence of each half of the two-stream split
        caches = {}
        for b in sample:
            caches[b] = oracle.SeqCache(S.n_layers)
            o = oracle.forward(om, toks[b].tolist(), caches[b])
            check_logits(logits[b], o["logits"])
            check_token(nxt[b], o["logits"])
        feeds, want = [], []
        for step in range(ND):
            feed = nxt.copy()
            d = run.decode(list(range(B)), feed.tolist(), debug=True)
            assert d["status"] == 0
            np.testing.assert_array_equal(d["pos"], np.full(B, P + step))
            outs = {}
            for b in sample:
                o = oracle.forward(om, [int(feed[b])], caches[b])
                check_hidden(d["hidden"][:, b:b + 1], o["hidden"])
                check_logits(d["logits"][b], o["logits"])
                check_token(d["next"][b], o["logits"])
                outs[b] = o
            feeds.append(feed)
            want.append(outs)
            nxt = d["next"].astype(np.int64)
        # the same steps through the decode-step kernel, fed the same tokens, from the same cache
        qw.qw.qw_set_option(eng.model, qw.qw.QW_OPT_DECODE_STEP_KERNEL, 1)
        for b in range(B):
            qw.qw.qw_kv_truncate(eng.kv, b, P, eng.stream)
        for step in range(ND):
            d = run.decode(list(range(B)), feeds[step].tolist(), debug=True)
            assert d["status"] == 0
            np.testing.assert_array_equal(d["pos"], np.full(B, P + step))
            for b in sample:
                o = want[step][b]
                check_hidden(d["hidden"][:, b:b + 1], o["hidden"])
                check_logits(d["logits"][b], o["logits"])
                check_token(d["next"][b], o["logits"])
    finally:
        eng.close()


def test_prefill_16x512_full(qw, om):
    B, P = 16, 512
    pages = B * (P // 16 + 1) + 8
    eng = _engine(qw, max_tokens=B * P, max_batch=B, max_context=P + 16, kv_pages=pages, max_seqs=B)
    try:
        run = Run(qw, eng)
        toks = synth.make_tokens(S.vocab, B * P, 1000 + 3).reshape(B, P)
        g = run.prefill(list(range(B)), [t.tolist() for t in toks], debug=True)
        assert g["status"] == 0
        # positions and KV slots of every token (bit-exact)
        mirror = oracle.PagedKVMirror(pages, B, 16)
        for b in range(B):
            assert mirror.reserve(b, P)
        want_slots = np.concatenate([mirror.slots(b, np.arange(P)) for b in range(B)])
        np.testing.assert_array_equal(g["pos"], np.tile(np.arange(P), B))
        np.testing.assert_array_equal(g["slot"], want_slots)
        for b in (0, 15):
            o = oracle.forward(om, toks[b].tolist(), oracle.SeqCache(S.n_layers))
            check_hidden(g["hidden"][:, b * P:(b + 1) * P], o["hidden"])
            check_logits(g["logits"][b], o["logits"])
            check_token(g["next"][b], o["logits"])
    finally:
        eng.close()


def test_long_context_ragged_decode_full(qw, om):
    B, ND, seed = 8, 2, 77
    lens = synth.make_lengths(B, 1024, 32768, 2000)
    eng = _engine(qw, max_tokens=max(B, 8), max_batch=max(B, 8), max_context=int(lens.max()) + ND + 16,
                  kv_pages=int(sum((n + ND + 15) // 16 + 1 for n in lens)) + 8, max_seqs=B)
    try:
        run = Run(qw, eng)
        for b in range(B):
            run.qw.qw_kv_reserve(eng.kv, b, int(lens[b]) + ND, eng.stream)
            run.qw.qw_kv_fill_synthetic(eng.kv, b, int(lens[b]), seed, eng.stream)

        def prior_for(n):
            def prior(layer):
                pos = np.arange(n)
                return (synth.kv_fill_values(seed, layer, 0, pos, S.n_kv_heads, S.head_dim).astype(np.float64),
                        synth.kv_fill_values(seed, layer, 1, pos, S.n_kv_heads, S.head_dim).astype(np.float64))
            return prior

        short, long_ = int(np.argmin(lens)), int(np.argmax(lens))
        cache_short = oracle.SeqCache(S.n_layers, prior=prior_for(int(lens[short])), prior_len=int(lens[short]))
        feed = np.zeros(B, np.int64)  # the first decode step feeds token 0 to every sequence
        for step in range(ND):
            d = run.decode(list(range(B)), feed.tolist(), debug=True)
            assert d["status"] == 0
            np.testing.assert_array_equal(d["pos"], lens + step)
            # shortest sequence: the whole model
            o = oracle.forward(om, [int(feed[short])], cache_short)
            check_hidden(d["hidden"][:, short:short + 1], o["hidden"])
            check_logits(d["logits"][short], o["logits"])
            check_token(d["next"][short], o["logits"])
            if step == 0:
                # longest sequence: every layer, each from the GPU's own input to it
                n = int(lens[long_])
                for layer in range(S.n_layers):
                    x_in = (om.embed_rows([int(feed[long_])]) if layer == 0
                            else d["hidden"][layer - 1, long_:long_ + 1])
                    c = oracle.SeqCache(S.n_layers, prior=prior_for(n), prior_len=n)
                    y = oracle.decoder_layer(np.asarray(x_in, np.float64), om.layer(layer), S, c, layer,
                                             np.array([n]))
                    e = rel_err(d["hidden"][layer, long_], y[0])
                    assert e <= HIDDEN_REL, f"layer {layer}: ||dx||/||x|| = {e:.3e}"
            feed = d["next"].astype(np.int64)
    finally:
        eng.close()
