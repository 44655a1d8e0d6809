"""qw_decode_steps: n greedy decode steps (the generation loop of "Dentro de un LLM", Paso 9)
replayed from one CUDA graph. Its picks, the cache it leaves and the next step's logits are
bit-identical to n calls of qw_decode_step, on the batch-1 cluster path (28 layers), the
small-batch GEMV path and the two-stream tensor-core path; the first picks also match the
oracle. Out-of-range step counts and unreserved positions are refused before anything runs."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, check_token, engine, weights

pytestmark = pytest.mark.gpu

S = synth.QWEN3_0_6B
S1 = synth.ONE_BLOCK


@pytest.fixture(scope="module")
def full(qw):
    eng = engine(qw, S, max_tokens=256, max_batch=24, max_context=256, kv_pages=24 * 16 + 8, max_seqs=24)
    yield Run(qw, eng)
    eng.close()


def _steps_vs_single(run, B, P, n, seed):
    """Prefill B prompts of P tokens, then n steps through qw_decode_steps and again through
    n qw_decode_step calls; returns both pick arrays [n, B], both next-step logits and the
    prompts."""
    import torch
    qw, eng = run.qw, run.eng
    prompts = [synth.make_tokens(run.s.vocab, P, seed + b).tolist() for b in range(B)]
    seqs = list(range(B))
    res = []
    for multi in (True, False):
        qw.qw_kv_reset(eng.kv, -1, eng.stream)
        g = run.prefill(seqs, prompts, debug=False, logits=False, reserve_extra=n + 1)
        first = torch.tensor(g["next"], dtype=torch.int32, device="cuda")
        out = torch.full((n, B), -7, dtype=torch.int32, device="cuda")
        if multi:
            qw.qw_decode_steps(eng.model, eng.kv, seqs, n, first.data_ptr(), out.data_ptr(), eng.stream)
        else:
            for i in range(n):
                src = first if i == 0 else out[i - 1]
                qw.qw_decode_step(eng.model, eng.kv, seqs, src.data_ptr(), 0, out[i].data_ptr(), eng.stream)
        assert qw.qw_sync_status(eng.model, eng.stream) == 0, qw.qw_last_error()
        for b in seqs:
            assert qw.qw_kv_length(eng.kv, b) == P + n
        d = run.decode(seqs, out[n - 1].cpu().numpy(), debug=False)
        res.append((out.cpu().numpy(), d["logits"], g["next"]))
    (m_ids, m_lg, m_first), (s_ids, s_lg, s_first) = res
    assert np.array_equal(m_first, s_first)
    assert np.array_equal(m_ids, s_ids)
    assert np.array_equal(m_lg, s_lg)
    return m_ids, m_first, prompts


def test_batch1_cluster_path_matches_single_steps_and_oracle(full):
    """B=1, 28 layers (two cluster kernels per layer): 12 steps in one graph."""
    run = full
    run.qw.qw_set_option(run.eng.model, run.qw.QW_OPT_BATCH1_CLUSTERS, 1)
    ids, first, prompts = _steps_vs_single(run, 1, 5, 12, 7100)
    om = oracle.Model(weights(S))
    c = oracle.SeqCache(S.n_layers)
    o = oracle.forward(om, prompts[0], c)
    check_token(first[0], o["logits"])
    tok = int(first[0])
    for i in range(3):   # the first picks against the oracle fed the same ids
        o = oracle.forward(om, [tok], c)
        check_token(ids[i, 0], o["logits"])
        tok = int(ids[i, 0])


@pytest.mark.parametrize("B", [3, 20])
def test_batched_paths_match_single_steps(full, B):
    """B=3 (GEMV family) and B=20 (tensor-core GEMMs, the batch as two streams): 6 steps."""
    _steps_vs_single(full, B, 9, 6, 7200 + B)


def test_refusals_leave_the_cache_untouched(qw):
    import torch
    eng = engine(qw, S1, max_tokens=16, max_batch=4, max_context=64, kv_pages=16, max_seqs=4)
    try:
        run = Run(qw, eng)
        g = run.prefill([0], [[5, 6, 7]], debug=False, logits=False, reserve_extra=4)   # one 16-slot page
        first = torch.tensor(g["next"], dtype=torch.int32, device="cuda")
        out = torch.zeros((qw.qw.QW_MAX_GRAPH_STEPS + 1, 1), dtype=torch.int32, device="cuda")
        for n in (0, -1, qw.qw.QW_MAX_GRAPH_STEPS + 1, 14):   # 14 > the 13 reserved free slots
            with pytest.raises(qw.qw.QwError):
                qw.qw.qw_decode_steps(eng.model, eng.kv, [0], n, first.data_ptr(), out.data_ptr(), eng.stream)
            assert qw.qw.qw_kv_length(eng.kv, 0) == 3
        qw.qw.qw_decode_steps(eng.model, eng.kv, [0], 13, first.data_ptr(), out.data_ptr(), eng.stream)
        assert qw.qw.qw_sync_status(eng.model, eng.stream) == 0
        assert qw.qw.qw_kv_length(eng.kv, 0) == 16
    finally:
        eng.close()
