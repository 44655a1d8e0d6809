"""Guards of the fp16 storage: activations and K/V values that leave the fp16 range are
reported through the status word instead of silently turning into inf, and norm weights that
would let a normalised fp16 operand overflow are refused when the model is built.

The inputs are built on the host: one embedding row set to a constant, so that its RMSNorm
output equals the input-norm weight (about 1 per feature), and every v_proj weight set to
128, so that each value of that token is about 128 * 1024 = 131072 > 65504. Every other
weight is the usual seeded one."""

import numpy as np
import pytest

import synth
from gpu_util import Run, weights

pytestmark = pytest.mark.gpu

S1 = synth.ONE_BLOCK
HOT = 7  # the token id whose embedding row is constant


class _Override:
    """The seeded weights with some tensors replaced (bf16 bit patterns)."""

    def __init__(self, base, layer_fn=None, embed_row=None, final_norm=None):
        self.base, self.shape = base, base.shape
        self.layer_fn, self.embed_row, self.fnorm = layer_fn, embed_row, final_norm

    def named(self):
        e = self.base.embed
        if self.embed_row is not None:
            e = e.copy()
            e[HOT] = self.embed_row
        yield "model.embed_tokens.weight", e
        for i in range(self.shape.n_layers):
            d = dict(self.base.layer(i))
            if self.layer_fn:
                d = self.layer_fn(d)
            for name, arr in d.items():
                yield f"model.layers.{i}.{name}", arr
        yield "model.norm.weight", self.base.final_norm if self.fnorm is None else self.fnorm


def _big_v(d):
    d = dict(d)
    d["self_attn.v_proj.weight"] = np.full_like(d["self_attn.v_proj.weight"], 0x4300)  # bf16 bits of 128.0
    return d


@pytest.fixture(scope="module")
def hot(qw):
    w = _Override(weights(S1), layer_fn=_big_v, embed_row=np.full(S1.hidden, 0x3F00, np.uint16))  # 0.5
    eng = qw.qw.Engine(S1, dict(w.named()), max_tokens=64, max_batch=16, max_context=256, kv_pages=64,
                       max_seqs=16)
    yield Run(qw, eng)
    eng.close()


@pytest.mark.parametrize("n", [3, 12])
def test_kv_value_overflow_sets_range_status(hot, n):
    """3 tokens: small-batch path (fp32 q|k|v, fp16 append); 12 tokens: tensor-core path
    (the projection tile staged as fp16). Both report QW_ERR_RANGE; a later clean call on
    the same model reports nothing."""
    run = hot
    qw = run.qw
    qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    g = run.prefill([0], [[HOT] * n], debug=False, check=False, reserve_extra=2)
    assert g["status"] == -9, qw.qw_last_error()
    # decode of the same token on a fresh sequence: the fused small-batch append
    qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    g = run.prefill([1], [[11, 12]], debug=False, reserve_extra=2)
    assert g["status"] == 0
    d = run.decode([1], [HOT], debug=False, check=False)
    assert d["status"] == -9
    qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    g = run.prefill([2], [[11, 12, 13]], debug=False)  # no hot token: clean
    assert g["status"] == 0


def test_batched_decode_overflow_sets_range_status(hot):
    """A decode batch of 12 (tensor-core projections, q|k|v head epilogue) with the hot
    token in one row."""
    run = hot
    qw = run.qw
    qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    seqs = list(range(12))
    g = run.prefill(seqs, [[20 + i, 30 + i] for i in seqs], debug=False, reserve_extra=2)
    assert g["status"] == 0
    feed = [40 + i for i in seqs]
    feed[5] = HOT
    d = run.decode(seqs, feed, debug=False, check=False)
    assert d["status"] == -9


def test_norm_weight_too_large_is_refused(qw):
    """A final-norm weight of 4096 > 65504 / sqrt(1024) = 2047 could make a normalised
    operand overflow: qw_init_weights refuses the model (QW_ERR_INVALID_ARG)."""
    fn = np.array(weights(S1).final_norm, copy=True)
    fn[100] = 0x4580  # bf16 bits of 4096.0
    w = _Override(weights(S1), final_norm=fn)
    with pytest.raises(qw.qw.QwError) as e:
        qw.qw.Engine(S1, dict(w.named()), max_tokens=16, max_batch=4, max_context=64, kv_pages=8, max_seqs=4)
    assert e.value.status == -1


def test_step_kernel_wait_runs_out(qw):
    """A bounded wait of the decode-step kernel that runs out: with a 1 ms limit and one
    arrival more than the attention provides, the first o_proj unit gives up, the kernel
    stops every CTA and qw_sync_status reports QW_ERR_TIMEOUT (no trap, no fault). The next
    normal step on the same model, from the same cache, matches the oracle."""
    import oracle
    from gpu_util import check_hidden, check_logits, check_token

    s = S1
    eng = qw.qw.Engine(s, dict(weights(s).named()), max_tokens=64, max_batch=16, max_context=64, kv_pages=64,
                       max_seqs=16)
    try:
        run = Run(qw, eng)
        om = oracle.Model(weights(s))
        B = 16
        seqs = list(range(B))
        prompts = [synth.make_tokens(s.vocab, 2 + i % 3, 2100 + i).tolist() for i in range(B)]
        g = run.prefill(seqs, prompts, debug=False, reserve_extra=2)
        feed = g["next"].tolist()
        qw.qw.qw_set_option(eng.model, qw.qw.QW_OPT_DECODE_STEP_KERNEL, 1)
        qw.qw.qw_set_option(eng.model, qw.qw.QW_OPT_TEST_WAIT_LIMIT_US, 1000)
        qw.qw.qw_set_option(eng.model, qw.qw.QW_OPT_TEST_EXTRA_ARRIVALS, 1)
        try:
            d = run.decode(seqs, feed, debug=False, check=False)
        finally:
            qw.qw.qw_set_option(eng.model, qw.qw.QW_OPT_TEST_EXTRA_ARRIVALS, 0)
            qw.qw.qw_set_option(eng.model, qw.qw.QW_OPT_TEST_WAIT_LIMIT_US, 2000000)
        assert d["status"] == -6, qw.qw.qw_last_error()
        # the timed-out step is discarded: every sequence back to its prompt
        for sq, p in zip(seqs, prompts):
            qw.qw.qw_kv_truncate(eng.kv, sq, len(p), eng.stream)
        d = run.decode(seqs, feed, debug=True)
        assert d["status"] == 0
        for b, p in enumerate(prompts):
            c = oracle.SeqCache(1)
            oracle.forward(om, p, c)
            o = oracle.forward(om, [feed[b]], c)
            check_hidden(d["hidden"][:, b:b + 1], o["hidden"])
            check_logits(d["logits"][b], o["logits"])
            check_token(d["next"][b], o["logits"])
    finally:
        eng.close()
