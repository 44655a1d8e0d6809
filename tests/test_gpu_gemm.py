"""GPU parity, tensor-core path (> 8 token rows per call: tcgen05 GEMMs for the projections,
SwiGLU and the LM-head argmax), on one Qwen3-0.6B-shaped block plus the tied head.

Shapes span several 128-feature and token tiles with ragged tails (token counts that are
not multiples of 64/128/256)."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, check_hidden, check_logits, check_token, engine, weights

pytestmark = pytest.mark.gpu

S1 = synth.ONE_BLOCK


@pytest.fixture(scope="module")
def blk(qw):
    eng = engine(qw, S1, max_tokens=1024, max_batch=32, max_context=1024, kv_pages=1024, max_seqs=32)
    yield Run(qw, eng), oracle.Model(weights(S1))
    eng.close()


@pytest.mark.parametrize("lens", [(150, 97), (9,), (300, 1, 64, 17)])
def test_prefill_tensor_core_path(blk, lens):
    run, om = blk
    run.qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    seqs = list(range(len(lens)))
    prompts = [synth.make_tokens(S1.vocab, n, 500 + i).tolist() for i, n in enumerate(lens)]
    g = run.prefill(seqs, prompts)
    assert g["status"] == 0
    row = 0
    for b, p in enumerate(prompts):
        o = oracle.forward(om, p, oracle.SeqCache(1))
        check_hidden(g["hidden"][:, row:row + len(p)], o["hidden"])
        check_logits(g["logits"][b], o["logits"])
        check_token(g["next"][b], o["logits"])
        np.testing.assert_array_equal(g["pos"][row:row + len(p)], np.arange(len(p)))
        row += len(p)


def test_batched_decode_argmax_epilogue(blk):
    """B = 12 sequences decode together (12 token rows: tensor-core GEMMs + argmax epilogue)."""
    run, om = blk
    run.qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    B = 12
    seqs = list(range(B))
    prompts = [synth.make_tokens(S1.vocab, 3 + (i % 7), 700 + i).tolist() for i in range(B)]
    g = run.prefill(seqs, prompts, reserve_extra=4)
    caches = []
    for b, p in enumerate(prompts):
        c = oracle.SeqCache(1)
        o = oracle.forward(om, p, c)
        check_logits(g["logits"][b], o["logits"])
        check_token(g["next"][b], o["logits"])
        caches.append(c)
    forced = synth.make_tokens(S1.vocab, 3 * B, 777).reshape(3, B)
    for step in range(3):
        d = run.decode(seqs, forced[step].tolist(), debug=(step != 1))
        assert d["status"] == 0
        for b in range(B):
            o = oracle.forward(om, [int(forced[step, b])], caches[b])
            if step != 1:
                check_hidden(d["hidden"][:, b:b + 1], o["hidden"])
            check_logits(d["logits"][b], o["logits"])
            check_token(d["next"][b], o["logits"])


def test_batch_invariance_and_determinism(blk):
    """A sequence decoded inside a batch of 12 matches the same sequence decoded alone within
    tolerance; repeating the batched run is bit-identical."""
    run, _ = blk
    qw, eng = run.qw, run.eng
    B = 12
    prompts = [synth.make_tokens(S1.vocab, 4 + i, 900 + i).tolist() for i in range(B)]
    res = []
    for _ in range(2):
        qw.qw_kv_reset(eng.kv, -1, eng.stream)
        g = run.prefill(list(range(B)), prompts, debug=False, reserve_extra=2)
        d = run.decode(list(range(B)), g["next"].tolist(), debug=False)
        res.append(d["logits"])
    np.testing.assert_array_equal(res[0], res[1])
    qw.qw_kv_reset(eng.kv, -1, eng.stream)
    g1 = run.prefill([5], [prompts[5]], debug=False, reserve_extra=2)
    d1 = run.decode([5], g1["next"].tolist(), debug=False)
    check_logits(d1["logits"][0], res[0][5], tol=2e-2)


MODES = {  # (QW_OPT_DECODE_STEP_KERNEL, QW_OPT_SPLIT_DECODE)
    "step_kernel": (1, 1),   # the whole decode step as one cooperative kernel
    "two_streams": (0, 1),   # launch per phase, two halves on two streams
    "one_chain": (0, 0),     # launch per phase, one chain
}


@pytest.mark.parametrize("B", [17, 32])
def test_batched_decode_paths(blk, B):
    """A decode batch of >= 16 sequences through each of its three paths (ragged halves for
    odd B): every sequence's hidden state after the layer, logits and id match the oracle,
    and the paths agree with each other within rounding."""
    run, om = blk
    qw, eng = run.qw, run.eng
    seqs = list(range(B))
    prompts = [synth.make_tokens(S1.vocab, 2 + (i % 5), 1100 + i).tolist() for i in range(B)]
    forced = synth.make_tokens(S1.vocab, 2 * B, 1177).reshape(2, B)
    out = {}
    try:
        for mode, (step, split) in MODES.items():
            qw.qw_set_option(eng.model, qw.QW_OPT_DECODE_STEP_KERNEL, step)
            qw.qw_set_option(eng.model, qw.QW_OPT_SPLIT_DECODE, split)
            qw.qw_kv_reset(eng.kv, -1, eng.stream)
            run.prefill(seqs, prompts, debug=False, reserve_extra=3)
            caches = []
            for b, p in enumerate(prompts):
                c = oracle.SeqCache(1)
                oracle.forward(om, p, c)
                caches.append(c)
            logits = []
            for step_i in range(2):
                # the first step dumps every layer's hidden state; the second replays a graph
                d = run.decode(seqs, forced[step_i].tolist(), debug=(step_i == 0))
                assert d["status"] == 0
                for b in range(B):
                    o = oracle.forward(om, [int(forced[step_i, b])], caches[b])
                    if step_i == 0:
                        check_hidden(d["hidden"][:, b:b + 1], o["hidden"])
                    check_logits(d["logits"][b], o["logits"])
                    check_token(d["next"][b], o["logits"])
                logits.append(d["logits"])
            out[mode] = logits
    finally:
        qw.qw_set_option(eng.model, qw.QW_OPT_DECODE_STEP_KERNEL, 0)
        qw.qw_set_option(eng.model, qw.QW_OPT_SPLIT_DECODE, 1)
    for mode in ("two_streams", "one_chain"):
        for a, b in zip(out["step_kernel"], out[mode]):
            check_logits(a, b, tol=2e-2)


def test_step_kernel_deterministic(blk):
    """The decode-step kernel adds its split-K partials and attention splits in a fixed order:
    two runs of the same batch give bit-identical logits."""
    run, _ = blk
    qw, eng = run.qw, run.eng
    B = 24
    prompts = [synth.make_tokens(S1.vocab, 3 + i % 4, 1300 + i).tolist() for i in range(B)]
    res = []
    qw.qw_set_option(eng.model, qw.QW_OPT_DECODE_STEP_KERNEL, 1)
    try:
        for _ in range(2):
            qw.qw_kv_reset(eng.kv, -1, eng.stream)
            g = run.prefill(list(range(B)), prompts, debug=False, reserve_extra=2)
            d = run.decode(list(range(B)), g["next"].tolist(), debug=False)
            res.append(d["logits"])
    finally:
        qw.qw_set_option(eng.model, qw.QW_OPT_DECODE_STEP_KERNEL, 0)
    np.testing.assert_array_equal(res[0], res[1])


class _PeakyQK:
    """The seeded weights with every QK-norm weight set to 2.0. Normalised q and k then have
    RMS 2 per component, the attention logits q.k / sqrt(128) a standard deviation near 4, and
    each query's softmax mass sits on a few keys: a stale or wrong key/value tile changes the
    attention output by O(1) instead of averaging out as it does with near-uniform weights."""

    def __init__(self, base):
        self.base = base
        self.shape = base.shape

    @property
    def embed(self):
        return self.base.embed

    @property
    def final_norm(self):
        return self.base.final_norm

    def layer(self, i):
        d = dict(self.base.layer(i))
        for name in ("self_attn.q_norm.weight", "self_attn.k_norm.weight"):
            d[name] = np.full_like(d[name], 0x4000)  # bf16 bits of 2.0
        return d

    def named(self):
        yield "model.embed_tokens.weight", self.embed
        for i in range(self.shape.n_layers):
            for name, arr in self.layer(i).items():
                yield f"model.layers.{i}.{name}", arr
        yield "model.norm.weight", self.final_norm


ATTN_REL = 2e-2  # ||o_gpu - o_oracle|| / ||o_oracle|| per token (fp16 q, k, v, P; peaky softmax)


@pytest.mark.parametrize("lens", [(300, 129, 64, 17), (1000,)])
def test_prefill_attention_peaky(qw, lens):
    """Prefill attention output of every token against the oracle's, with sharply peaked
    softmax rows; sequences span many 64-key tiles and end mid-tile and mid-page."""
    import torch
    w = _PeakyQK(weights(S1))
    om = oracle.Model(w)
    names = [n for n, _ in synth.Weights(S1).named()]
    wd = dict(w.named())
    assert sorted(wd) == sorted(names)
    eng = qw.qw.Engine(S1, wd, max_tokens=1024, max_batch=8, max_context=1024, kv_pages=256, max_seqs=8)
    try:
        run = Run(qw, eng)
        prompts = [synth.make_tokens(S1.vocab, n, 900 + i).tolist() for i, n in enumerate(lens)]
        T = sum(lens)
        attn = torch.zeros((S1.n_layers, T, S1.n_heads * S1.head_dim), dtype=torch.float16, device="cuda")
        qw.qw.qw_debug_set_attn(eng.model, attn.data_ptr())
        try:
            g = run.prefill(list(range(len(lens))), prompts)
        finally:
            qw.qw.qw_debug_set_attn(eng.model, 0)
        assert g["status"] == 0
        a = attn.float().cpu().numpy()
        row = 0
        for b, p in enumerate(prompts):
            taps = {}
            o = oracle.forward(om, p, oracle.SeqCache(S1.n_layers), taps=taps)
            want = taps["attn"][0]
            got = a[0, row:row + len(p)]
            err = np.linalg.norm(got - want, axis=1) / np.linalg.norm(want, axis=1)
            worst = int(np.argmax(err))
            assert err[worst] <= ATTN_REL, f"sequence {b}, token {worst}: {err[worst]:.3e}"
            check_hidden(g["hidden"][:, row:row + len(p)], o["hidden"])
            check_logits(g["logits"][b], o["logits"])
            row += len(p)
    finally:
        eng.close()


def _chunked_run(om, run, plan, s, taps_check=None):
    """plan: list of calls, each a list of (seq, n_tokens). Every call's hidden states, last
    logits, positions and slots against the oracle continuing each sequence's own cache."""
    caches, fed = {}, {}
    mirror = oracle.PagedKVMirror(run.qw.qw_kv_pool_ptrs(run.eng.kv)[2], 16, 16)
    total = {}
    for call in plan:
        for sq, n in call:
            total[sq] = total.get(sq, 0) + n
    run.qw.qw_kv_reset(run.eng.kv, -1, run.eng.stream)
    for sq in sorted(total):
        run.qw.qw_kv_reserve(run.eng.kv, sq, total[sq], run.eng.stream)
        mirror.reserve(sq, total[sq])
    for ci, call in enumerate(plan):
        seqs = [sq for sq, _ in call]
        prompts = [synth.make_tokens(s.vocab, n, 3000 + 31 * ci + sq).tolist() for sq, n in call]
        T = sum(len(p) for p in prompts)
        attn = None
        if taps_check is not None:
            import torch
            attn = torch.zeros((s.n_layers, T, s.n_heads * s.head_dim), dtype=torch.float16, device="cuda")
            run.qw.qw_debug_set_attn(run.eng.model, attn.data_ptr())
        try:
            g = run.prefill(seqs, prompts, reserve=False)
        finally:
            if attn is not None:
                run.qw.qw_debug_set_attn(run.eng.model, 0)
        assert g["status"] == 0
        row = 0
        for b, (sq, p) in enumerate(zip(seqs, prompts)):
            c = caches.setdefault(sq, oracle.SeqCache(s.n_layers))
            start = fed.get(sq, 0)
            np.testing.assert_array_equal(g["pos"][row:row + len(p)], np.arange(start, start + len(p)))
            np.testing.assert_array_equal(g["slot"][row:row + len(p)], mirror.slots(sq, range(start, start + len(p))))
            taps = {}
            o = oracle.forward(om, p, c, taps=taps)
            check_hidden(g["hidden"][:, row:row + len(p)], o["hidden"])
            check_logits(g["logits"][b], o["logits"])
            check_token(g["next"][b], o["logits"])
            if taps_check is not None:
                taps_check(attn.float().cpu().numpy()[0, row:row + len(p)], taps["attn"][0], (ci, sq))
            fed[sq] = start + len(p)
            row += len(p)


def test_chunked_prefill_tensor_core_path(blk):
    """Prompts fed in chunks that continue each sequence's cache (positions after the cached
    prefix, attention over it): chunks of several sequences share calls, start and end
    mid-page and mid-tile, and one call is small enough for the small-batch path."""
    run, om = blk
    plan = [[(0, 300), (1, 77)], [(0, 200), (1, 50), (2, 9)], [(1, 129), (2, 140)], [(2, 5), (0, 3)]]
    _chunked_run(om, run, plan, S1)


def test_chunked_prefill_peaked_attention(qw):
    """The same with sharply peaked attention (QK-norm weights 2.0): every token's attention
    output over the cached prefix within 2e-2 of the oracle's."""
    w = _PeakyQK(weights(S1))
    om = oracle.Model(w)
    eng = qw.qw.Engine(S1, dict(w.named()), max_tokens=1024, max_batch=8, max_context=1024, kv_pages=256,
                       max_seqs=8)

    def check(got, want, where):
        err = np.linalg.norm(got - want, axis=1) / np.linalg.norm(want, axis=1)
        assert err.max() <= ATTN_REL, f"{where}: token {int(np.argmax(err))}: {err.max():.3e}"

    try:
        plan = [[(0, 333), (1, 64)], [(0, 420), (1, 191)], [(1, 17)]]
        _chunked_run(om, Run(qw, eng), plan, S1, taps_check=check)
    finally:
        eng.close()
