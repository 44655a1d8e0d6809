"""GPU parity, small-batch path (<= 8 token rows per call: the GEMV family + paged attention).

Each test drives libqw through its C ABI and compares with the fp64 oracle on the same
seeded bf16 weights: positions and KV slots bit-exact, hidden state per layer and token
within 5e-3 normwise, logits within 5e-2, greedy ids equal when the oracle's top-2 gap
exceeds 1e-2.
"""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, check_hidden, check_logits, check_token, engine, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def one_block(qw):
    eng = engine(qw, synth.ONE_BLOCK, max_tokens=64, max_batch=16, max_context=512, kv_pages=256,
                 max_seqs=16)
    yield Run(qw, eng), oracle.Model(weights(synth.ONE_BLOCK))
    eng.close()


def _n_pages(run):
    return run.qw.qw_kv_pool_ptrs(run.eng.kv)[2]


def _greedy_parity(run, om, prompt, n_decode, graph_steps=()):
    """Prefill + n_decode greedy steps on sequence 0; the oracle runs its own greedy loop.
    Comparison stops at the first legitimate divergence (ids differ where the top-2 gap is
    within tolerance)."""
    s = run.s
    qw, eng = run.qw, run.eng
    qw.qw_kv_reset(eng.kv, -1, eng.stream)
    mirror = oracle.PagedKVMirror(_n_pages(run), 16, 16)
    mirror.reserve(0, len(prompt) + n_decode)
    cache = oracle.SeqCache(s.n_layers)
    o = oracle.forward(om, prompt, cache)
    g = run.prefill([0], [prompt], reserve_extra=n_decode)
    assert g["status"] == 0
    np.testing.assert_array_equal(g["pos"], np.arange(len(prompt)))
    np.testing.assert_array_equal(g["slot"], mirror.slots(0, range(len(prompt))))
    np.testing.assert_array_equal(qw.qw_kv_page_table(eng.kv, 0), mirror.tables[0])
    check_hidden(g["hidden"], o["hidden"])
    check_logits(g["logits"][0], o["logits"])
    same = check_token(g["next"][0], o["logits"])
    tok = int(g["next"][0])
    compared = 0
    for step in range(n_decode):
        if not same:
            break
        pos = len(prompt) + step
        o = oracle.forward(om, [tok], cache)
        dbg = step not in graph_steps
        g = run.decode([0], [tok], debug=dbg)
        assert g["status"] == 0
        if dbg:
            assert g["pos"][0] == pos
            assert g["slot"][0] == mirror.slots(0, [pos])[0]
            check_hidden(g["hidden"], o["hidden"])
        check_logits(g["logits"][0], o["logits"])
        same = check_token(g["next"][0], o["logits"])
        tok = int(g["next"][0])
        compared += 1
    return compared


def test_config0_random_prompt_greedy(one_block):
    run, om = one_block
    prompt = synth.make_tokens(synth.ONE_BLOCK.vocab, 5, 1000).tolist()
    n = _greedy_parity(run, om, prompt, 16, graph_steps=range(8, 16))
    assert n >= 8


def test_config0_page_prompt_greedy(one_block):
    run, om = one_block
    n = _greedy_parity(run, om, list(synth.PAGE_PROMPT), 16)
    assert n >= 8


def test_graph_replay_bit_identical_to_direct(one_block):
    run, _ = one_block
    qw, eng = run.qw, run.eng
    prompt = synth.make_tokens(synth.ONE_BLOCK.vocab, 7, 77).tolist()
    outs = []
    for dbg in (True, False, False):
        qw.qw_kv_reset(eng.kv, -1, eng.stream)
        g = run.prefill([3], [prompt], debug=False, reserve_extra=4)
        tok = int(g["next"][0])
        steps = []
        for _ in range(3):
            d = run.decode([3], [tok], debug=dbg)
            steps.append(d["logits"][0])
            tok = int(d["next"][0])
        outs.append(np.stack(steps))
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[1], outs[2])


def test_ragged_small_batch_slots_and_values(one_block):
    """Three sequences with interleaved reservations, prefilled together (6 tokens)."""
    run, om = one_block
    s = synth.ONE_BLOCK
    qw, eng = run.qw, run.eng
    qw.qw_kv_reset(eng.kv, -1, eng.stream)
    mirror = oracle.PagedKVMirror(_n_pages(run), 16, 16)
    for seq, n in ((2, 20), (0, 7), (2, 40), (5, 3)):
        qw.qw_kv_reserve(eng.kv, seq, n, eng.stream)
        mirror.reserve(seq, n)
    seqs = [2, 0, 5]
    prompts = [synth.make_tokens(s.vocab, n, 300 + i).tolist() for i, n in enumerate((3, 2, 1))]
    g = run.prefill(seqs, prompts)
    assert g["status"] == 0
    want_pos = np.concatenate([np.arange(len(p)) for p in prompts])
    want_slot = np.concatenate([mirror.slots(sq, range(len(p))) for sq, p in zip(seqs, prompts)])
    np.testing.assert_array_equal(g["pos"], want_pos)
    np.testing.assert_array_equal(g["slot"], want_slot)
    for sq in (0, 2, 5):
        np.testing.assert_array_equal(qw.qw_kv_page_table(eng.kv, sq), mirror.tables[sq])
    # per-sequence oracle: hidden states and last-position logits; K rows at their slots
    kptr, _, n_pages = qw.qw_kv_pool_ptrs(eng.kv)
    import torch
    off = kptr - eng.pool.data_ptr()
    nk = n_pages * s.n_kv_heads * 16 * s.head_dim
    k0 = eng.pool[off:off + 2 * nk].view(torch.float16).float().cpu().numpy()
    k0 = k0.reshape(n_pages, s.n_kv_heads, 16, s.head_dim)
    row = 0
    for b, (sq, p) in enumerate(zip(seqs, prompts)):
        taps = {}
        o = oracle.forward(om, p, oracle.SeqCache(1), taps=taps)
        check_hidden(g["hidden"][:, row:row + len(p)], o["hidden"])
        check_logits(g["logits"][b], o["logits"])
        check_token(g["next"][b], o["logits"])
        for j in range(len(p)):
            slot = int(want_slot[row + j])
            got = k0[slot // 16, :, slot % 16, :]            # [n_kv, head_dim]
            want = taps["k"][0][:, j, :]                      # layer 0, after QK-norm + RoPE
            err = np.linalg.norm(got - want) / np.linalg.norm(want)
            assert err < 1e-2, (sq, j, err)
        row += len(p)


def test_error_paths_leave_state(one_block):
    run, _ = one_block
    qw, eng = run.qw, run.eng
    qw.qw_kv_reset(eng.kv, -1, eng.stream)
    free = qw.qw_kv_free_pages(eng.kv)
    per_seq = 512 // 16
    n_full = free // per_seq
    for sq in range(n_full):
        qw.qw_kv_reserve(eng.kv, sq, 512, eng.stream)
    left = qw.qw_kv_free_pages(eng.kv)
    with pytest.raises(qw.QwError) as e:
        qw.qw_kv_reserve(eng.kv, n_full, 16 * (left + 1), eng.stream)
    assert e.value.status == -2
    assert qw.qw_kv_free_pages(eng.kv) == left       # nothing was taken
    qw.qw_kv_reset(eng.kv, -1, eng.stream)
    assert qw.qw_kv_free_pages(eng.kv) == free
    # prefill beyond the reservation
    qw.qw_kv_reserve(eng.kv, 1, 4, eng.stream)
    with pytest.raises(qw.QwError) as e:
        run.prefill([1], [[1] * 20], debug=False, reserve=False)
    assert e.value.status == -2
    assert qw.qw_kv_length(eng.kv, 1) == 0
    # a prompt continues a non-empty sequence (chunked prefill) within its reservation only
    g = run.prefill([1], [[1, 2, 3]], debug=False)
    assert g["status"] == 0
    g = run.prefill([1], [[4]], debug=False, reserve=False)
    assert g["status"] == 0
    assert qw.qw_kv_length(eng.kv, 1) == 4
    pages = len(qw.qw_kv_page_table(eng.kv, 1))
    with pytest.raises(qw.QwError) as e:
        run.prefill([1], [[5] * (16 * pages - 3)], debug=False, reserve=False)
    assert e.value.status == -2
    assert qw.qw_kv_length(eng.kv, 1) == 4
    # a token id outside the vocabulary is reported through the status word
    qw.qw_kv_reserve(eng.kv, 4, 8, eng.stream)
    g = run.prefill([4], [[5, synth.ONE_BLOCK.vocab + 3]], debug=False, check=False)
    assert g["status"] == -5
    assert qw.qw_sync_status(eng.model, eng.stream) == 0  # the word was cleared


def test_degenerate_calls_are_rejected(one_block):
    """Empty batches, empty prompts, repeated or unknown sequence ids and batches beyond
    max_batch are refused on the host (QW_ERR_INVALID_ARG) before any launch, and leave the
    cache untouched."""
    import torch
    run, _ = one_block
    qw, eng = run.qw, run.eng
    qw.qw_kv_reset(eng.kv, -1, eng.stream)
    qw.qw_kv_reserve(eng.kv, 0, 32, eng.stream)
    qw.qw_kv_reserve(eng.kv, 1, 32, eng.stream)
    tok = torch.ones(64, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(32, dtype=torch.int32, device="cuda")
    t, n = tok.data_ptr(), nxt.data_ptr()
    calls = [
        lambda: qw.qw_prefill(eng.model, eng.kv, [], [], t, 0, n, eng.stream),            # no sequence
        lambda: qw.qw_prefill(eng.model, eng.kv, [0], [0], t, 0, n, eng.stream),          # empty prompt
        lambda: qw.qw_prefill(eng.model, eng.kv, [0, 1], [2, 0], t, 0, n, eng.stream),   # one empty prompt
        lambda: qw.qw_prefill(eng.model, eng.kv, [0, 0], [2, 2], t, 0, n, eng.stream),   # repeated id
        lambda: qw.qw_prefill(eng.model, eng.kv, [10 ** 6], [2], t, 0, n, eng.stream),   # unknown id
        lambda: qw.qw_prefill(eng.model, eng.kv, [-1], [2], t, 0, n, eng.stream),        # negative id
        lambda: qw.qw_prefill(eng.model, eng.kv, list(range(17)), [1] * 17, t, 0, n, eng.stream),  # > max_batch
        lambda: qw.qw_decode_step(eng.model, eng.kv, [], t, 0, n, eng.stream),           # no sequence
        lambda: qw.qw_decode_step(eng.model, eng.kv, [1, 1], t, 0, n, eng.stream),       # repeated id
        lambda: qw.qw_decode_step(eng.model, eng.kv, list(range(17)), t, 0, n, eng.stream),  # > max_batch
    ]
    # generate: prompt + decode steps beyond max_context (512) are refused before any work,
    # although the reserved pages hold them
    qw.qw_kv_reserve(eng.kv, 2, 512, eng.stream)
    h_prompt = np.ones(8, np.int32)
    h_out = np.zeros((1, 506), np.int32)
    calls.append(lambda: qw.qw_generate(eng.model, eng.kv, [2], [8], h_prompt, 505, h_out, eng.stream))
    for call in calls:
        with pytest.raises(qw.QwError) as e:
            call()
        assert e.value.status == -1
        assert qw.qw_kv_length(eng.kv, 0) == 0 and qw.qw_kv_length(eng.kv, 1) == 0
        assert qw.qw_kv_length(eng.kv, 2) == 0
    qw.qw_kv_reset(eng.kv, -1, eng.stream)


@pytest.fixture(scope="module")
def full_model(qw):
    eng = engine(qw, synth.QWEN3_0_6B, max_tokens=64, max_batch=8, max_context=256, kv_pages=64,
                 max_seqs=8)
    yield Run(qw, eng), oracle.Model(weights(synth.QWEN3_0_6B))
    eng.close()


def test_config1_greedy_28_layers(full_model):
    """28 layers, batch 1, 5-token prompt, 64 greedy decode steps (graph replays except a few
    steps that also dump hidden states)."""
    run, om = full_model
    prompt = synth.make_tokens(synth.QWEN3_0_6B.vocab, 5, 1001).tolist()
    graph = [i for i in range(64) if i not in (0, 31, 63)]
    n = _greedy_parity(run, om, prompt, 64, graph_steps=graph)
    assert n >= 32


@pytest.fixture(scope="module")
def one_block_long(qw):
    eng = engine(qw, synth.ONE_BLOCK, max_tokens=64, max_batch=8, max_context=8192, kv_pages=1300,
                 max_seqs=8)
    yield Run(qw, eng), oracle.Model(weights(synth.ONE_BLOCK))
    eng.close()


@pytest.fixture(scope="module")
def one_block_long_batch(qw):
    eng = engine(qw, synth.ONE_BLOCK, max_tokens=64, max_batch=16, max_context=8192, kv_pages=3000,
                 max_seqs=16)
    yield Run(qw, eng), oracle.Model(weights(synth.ONE_BLOCK))
    eng.close()


@pytest.mark.parametrize("lens", [(5000, 17, 4100, 300, 6001, 2, 4097, 900, 33, 5555),
                                  (5000, 17, 4100, 300, 6001, 2, 4097, 900, 33, 5555, 1, 64, 65, 2000, 16, 7000)])
def test_injected_long_cache_batched_decode(one_block_long_batch, lens):
    """More than 8 sequences (tensor-core projections) with caches longer than 4096 keys: 10
    sequences take the evenly split decode attention behind the q|k|v epilogue; 16 run both
    through the launch-per-phase path and through the decode-step kernel (ragged caches from
    1 to 7000 keys)."""
    run = one_block_long_batch[0]
    modes = (0, 1) if len(lens) >= 16 else (0,)
    try:
        for mode in modes:
            run.qw.qw_set_option(run.eng.model, run.qw.QW_OPT_DECODE_STEP_KERNEL, mode)
            test_injected_long_cache_forced_decode(one_block_long_batch, lens)
    finally:
        run.qw.qw_set_option(run.eng.model, run.qw.QW_OPT_DECODE_STEP_KERNEL, 0)


@pytest.mark.parametrize("lens", [(2047, 3001), (1, 300, 4000), (5000, 700, 6100)])
def test_injected_long_cache_forced_decode(one_block_long, lens):
    """KV caches filled by the counter-based generator (bit-identical on both sides), then
    forced decode steps; the oracle reads the same injected prefix. The last case is long
    enough (tokens x keys) for the evenly split decode attention."""
    run, om = one_block_long
    s = synth.ONE_BLOCK
    qw, eng = run.qw, run.eng
    qw.qw_kv_reset(eng.kv, -1, eng.stream)
    seed = 2024
    seqs = list(range(len(lens)))
    for sq, n in zip(seqs, lens):
        qw.qw_kv_reserve(eng.kv, sq, n + 3, eng.stream)
        qw.qw_kv_fill_synthetic(eng.kv, sq, n, seed, eng.stream)
    # the pool holds exactly the generator's values at the reserved slots
    eng.stream.synchronize()  # the fills ran on the engine's stream
    kptr, vptr, n_pages = qw.qw_kv_pool_ptrs(eng.kv)
    import torch
    off = kptr - eng.pool.data_ptr()
    nk = n_pages * s.n_kv_heads * 16 * s.head_dim
    k0 = eng.pool[off:off + 2 * nk].view(torch.float16).float().cpu().numpy().reshape(n_pages, s.n_kv_heads, 16, 128)
    pt = qw.qw_kv_page_table(eng.kv, seqs[-1])
    want = synth.kv_fill_values(seed, 0, 0, np.arange(32), s.n_kv_heads, s.head_dim)
    got = np.concatenate([k0[pt[0]], k0[pt[1]]], axis=1)
    np.testing.assert_array_equal(got, want)

    def prior_for(n):
        def prior(layer):
            pos = np.arange(n)
            return (synth.kv_fill_values(seed, layer, 0, pos, s.n_kv_heads, s.head_dim).astype(np.float64),
                    synth.kv_fill_values(seed, layer, 1, pos, s.n_kv_heads, s.head_dim).astype(np.float64))
        return prior
    caches = [oracle.SeqCache(1, prior=prior_for(n), prior_len=n) for n in lens]
    forced = synth.make_tokens(s.vocab, 2 * len(lens), 77).reshape(2, len(lens))
    for step in range(2):
        d = run.decode(seqs, forced[step].tolist(), debug=True)
        assert d["status"] == 0
        for b, n in enumerate(lens):
            o = oracle.forward(om, [int(forced[step, b])], caches[b])
            assert d["pos"][b] == n + step
            check_hidden(d["hidden"][:, b:b + 1], o["hidden"])
            check_logits(d["logits"][b], o["logits"])
            check_token(d["next"][b], o["logits"])


def test_generate_eos_stop(one_block):
    """Paso 9's EOS stop over a batch: each row equals the no-stop run cut after its first EOS
    (then -1), each cache holds exactly the tokens fed (the EOS is never fed), and a stopped
    sequence continues from its cache as the oracle's does."""
    run, om = one_block
    qw, eng = run.qw, run.eng
    s = synth.ONE_BLOCK
    lens, nd = [5, 9, 3, 7], 20
    prompts = [synth.make_tokens(s.vocab, n, 600 + n).tolist() for n in lens]
    flat = np.ascontiguousarray(np.concatenate(prompts).astype(np.int32))
    seqs = [0, 1, 2, 3]

    def fresh():
        qw.qw_kv_reset(eng.kv, -1, eng.stream)
        for sq, n in zip(seqs, lens):
            qw.qw_kv_reserve(eng.kv, sq, n + nd, eng.stream)

    fresh()
    full = np.zeros((4, nd + 1), np.int32)
    qw.qw_generate(eng.model, eng.kv, seqs, lens, flat, nd, full, eng.stream)
    eos = int(full[1, 4])  # appears in row 1 by index 4; maybe elsewhere, maybe not
    fresh()
    out = np.zeros((4, nd + 1), np.int32)
    counts = np.zeros(4, np.int32)
    qw.qw_generate_eos(eng.model, eng.kv, seqs, lens, flat, nd, eos, out, counts, eng.stream)
    stopped = []
    for b in range(4):
        hits = np.flatnonzero(full[b] == eos)
        n = int(hits[0]) + 1 if hits.size else nd + 1
        assert counts[b] == n, (b, counts[b], n)
        np.testing.assert_array_equal(out[b, :n], full[b, :n])
        assert np.all(out[b, n:] == -1)
        if hits.size:
            stopped.append(b)
            assert qw.qw_kv_length(eng.kv, seqs[b]) == lens[b] + n - 1
    assert 1 in stopped
    if len(stopped) == 4:  # every row stopped: the loop ended at the last stop
        last = max(int(counts[b]) for b in range(4)) - 1
    else:
        last = nd
    for b in range(4):
        if b not in stopped:
            assert qw.qw_kv_length(eng.kv, seqs[b]) == lens[b] + last
    # row 1 continues from its cache, fed token 17: the oracle is given the same tokens the
    # GPU fed (the prompt and the picks before the EOS; greedy paths of the two may part on
    # near ties, so the GPU's picks are forced)
    c = oracle.SeqCache(s.n_layers)
    oracle.forward(om, prompts[1] + out[1, :counts[1] - 1].tolist(), c)
    assert c.length == qw.qw_kv_length(eng.kv, 1)
    o = oracle.forward(om, [17], c)
    d = run.decode([1], [17], debug=False)
    check_logits(d["logits"][0], o["logits"])
    check_token(d["next"][0], o["logits"])
