"""Batch-1 decode as two thread-block-cluster launches per layer (QW_OPT_BATCH1_CLUSTERS, on by
default for multi-layer models where the shape and the device allow it) against the oracle: every layer's hidden
state, the KV slot, the logits and the greedy id of each decode step, for cached lengths
that start, cross and end 16-key pages up to the path's 128-key limit and the step after it
(which takes the launch-per-phase path); the attention outputs against the launch-per-phase
path; the launch count of a step (two per layer); bit-identical repeats."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, check_hidden, check_logits, check_token, weights

pytestmark = pytest.mark.gpu

S = synth.QWEN3_0_6B
S1 = synth.ONE_BLOCK


def _engine(qw, s):
    return qw.qw.Engine(s, dict(weights(s).named()), max_tokens=160, max_batch=4, max_context=256, kv_pages=64,
                        max_seqs=4)


@pytest.fixture(scope="module")
def one(qw):
    eng = _engine(qw, S1)
    yield Run(qw, eng)
    eng.close()


@pytest.fixture(scope="module")
def full(qw):
    eng = _engine(qw, S)
    yield Run(qw, eng)
    eng.close()


def _decode_vs_oracle(run, om, prompt, n_steps):
    """Prefill `prompt` into sequence 0, then n_steps greedy decode steps with the debug dumps
    on, each checked against the oracle fed the same ids."""
    qw = run.qw
    qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    g = run.prefill([0], [prompt], debug=False, reserve_extra=n_steps)
    c = oracle.SeqCache(run.s.n_layers)
    oracle.forward(om, prompt, c)
    tok = int(g["next"][0])
    outs = []
    for i in range(n_steps):
        d = run.decode([0], [tok], debug=True)
        o = oracle.forward(om, [tok], c)
        check_hidden(d["hidden"], o["hidden"])
        check_logits(d["logits"][0], o["logits"])
        check_token(d["next"][0], o["logits"])
        assert d["pos"][0] == len(prompt) + i
        outs.append(d)
        tok = int(d["next"][0])
    return outs


def _set(run, on):
    run.qw.qw_set_option(run.eng.model, run.qw.QW_OPT_BATCH1_CLUSTERS, 1 if on else 0)


def test_full_model_decode_matches_oracle(full):
    """28 layers: a 5-token prompt and 4 decode steps (the default bench workload's shape)."""
    run = full
    _set(run, True)
    om = oracle.Model(weights(S))
    prompt = synth.make_tokens(S.vocab, 5, 4100).tolist()
    _decode_vs_oracle(run, om, prompt, 4)


def test_launch_count_two_per_layer(full):
    """Without the debug dumps a step is: step begin, 2 launches per layer, and the LM head
    (whose last CTA writes the id and advances the length)."""
    run = full
    qw = run.qw
    prompt = synth.make_tokens(S.vocab, 7, 4101).tolist()
    for on, per_layer in ((True, 2), (False, 4)):
        _set(run, on)
        qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
        g = run.prefill([0], [prompt], debug=False, reserve_extra=4)
        run.decode([0], [int(g["next"][0])], debug=False)
        assert qw.qw_last_launch_count(run.eng.model) == 2 + per_layer * S.n_layers
    _set(run, True)


@pytest.mark.parametrize("n_prompt", [1, 15, 16, 17, 32, 126])
def test_page_edges_match_oracle(one, n_prompt):
    """Cached lengths 0 .. 127 at the first step (an empty cache, a page's last slot, a new page,
    a full 8-page cache) and, from the 126-token prompt, the step over 128 keys that leaves the
    cluster path."""
    run = one
    _set(run, True)
    om = oracle.Model(weights(S1))
    prompt = synth.make_tokens(S1.vocab, n_prompt, 4200 + n_prompt).tolist()
    _decode_vs_oracle(run, om, prompt, 3 if n_prompt == 126 else 2)


def test_attention_and_cache_match_launch_per_phase(one):
    """The attention outputs of both paths agree to fp16 rounding, and the K/V each appends
    gives the same next step."""
    import torch
    run = one
    qw = run.qw
    s = S1
    prompt = synth.make_tokens(s.vocab, 40, 4300).tolist()
    res = {}
    for on in (True, False):
        _set(run, on)
        qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
        g = run.prefill([0], [prompt], debug=False, reserve_extra=4)
        tok = int(g["next"][0])
        attn = torch.zeros((s.n_layers, 1, s.n_heads * s.head_dim), dtype=torch.float16, device="cuda")
        qw.qw_debug_set_attn(run.eng.model, attn.data_ptr())
        try:
            d1 = run.decode([0], [tok], debug=True)
        finally:
            qw.qw_debug_set_attn(run.eng.model, 0)
        d2 = run.decode([0], [int(d1["next"][0])], debug=True)
        res[on] = (attn.cpu().numpy().astype(np.float64), d1, d2)
    _set(run, True)
    a_on, a_off = res[True][0], res[False][0]
    assert np.max(np.abs(a_on - a_off)) <= 2e-3 * max(1.0, float(np.max(np.abs(a_off))))
    for k in (1, 2):
        h_on, h_off = res[True][k]["hidden"], res[False][k]["hidden"]
        assert np.linalg.norm(h_on - h_off) <= 1e-3 * np.linalg.norm(h_off)
        assert res[True][k]["slot"][0] == res[False][k]["slot"][0]


def test_repeat_is_bit_identical(one):
    """Fixed reduction orders: the same decode steps twice give identical logits."""
    run = one
    qw = run.qw
    _set(run, True)
    prompt = synth.make_tokens(S1.vocab, 20, 4400).tolist()
    seen = []
    for _ in range(2):
        qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
        g = run.prefill([0], [prompt], debug=False, reserve_extra=4)
        tok = int(g["next"][0])
        lg = []
        for _ in range(3):
            d = run.decode([0], [tok], debug=False)
            lg.append(d["logits"][0])
            tok = int(d["next"][0])
        seen.append(np.stack(lg))
    assert np.array_equal(seen[0], seen[1])


def test_trace_records_follow_the_documented_layout(full):
    """qw_trace_set on the cluster path: for every layer, launch (attention, MLP) and CTA, eight
    %globaltimer values at ((2 l + k) * 128 + c) * 8, in order (entry <= ... <= exit), each launch's
    dependency wait after the previous launch's earliest exit, and nothing written elsewhere."""
    import torch
    run = full
    qw = run.qw
    _set(run, True)
    L = S.n_layers
    prompt = synth.make_tokens(S.vocab, 5, 4500).tolist()
    qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    g = run.prefill([0], [prompt], debug=False, reserve_extra=4)
    buf = torch.zeros(L * 2 * 128 * 8 + 64, dtype=torch.int64, device="cuda")
    qw.qw_trace_set(run.eng.model, buf.data_ptr(), 8)
    try:
        run.decode([0], [int(g["next"][0])], debug=False)
    finally:
        qw.qw_trace_set(run.eng.model, 0, 0)
    tr = buf.cpu().numpy()
    assert not tr[L * 2 * 128 * 8:].any()
    tr = tr[:L * 2 * 128 * 8].reshape(L, 2, 128, 8)
    assert (tr > 0).all()
    assert (np.diff(tr, axis=3) >= 0).all()
    for l in range(L):
        # the MLP kernel's wait ends after the attention kernel's CTAs have all exited
        assert tr[l, 1, :, 1].min() >= tr[l, 0, :, 7].max()
        if l:
            assert tr[l, 0, :, 1].min() >= tr[l - 1, 1, :, 7].max()
