"""GPU parity of temperature + top-p sampling (Paso 8) through qw_sample_top_p: the token of
each row against the oracle's on the same fp32 logits and the same uniform u.

Where the oracle's running sums pass within 1e-5 of top_p or of u, the two sides may
legitimately round to different sides of the boundary (the GPU sums fp32 probabilities in
2^-40 fixed point, the oracle in fp64); there the GPU token must be valid: inside the oracle's
nucleus for top_p + 1e-5, with u inside its CDF interval widened by 1e-5. Everywhere else the
tokens must be equal."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, engine, weights

pytestmark = pytest.mark.gpu

V_FULL = synth.QWEN3_0_6B.vocab
TOL = 1e-5


def _gpu_sample(qw, logits, temperature, top_p, u):
    import torch
    lg = torch.tensor(np.ascontiguousarray(logits, np.float32), device="cuda")
    uu = torch.tensor(np.asarray(u, np.float32), device="cuda")
    nx = torch.full((lg.shape[0],), -1, dtype=torch.int32, device="cuda")
    qw.qw.qw_sample_top_p(lg.shape[0], lg.shape[1], lg.data_ptr(), lg.shape[1], temperature, top_p,
                          uu.data_ptr(), nx.data_ptr(), torch.cuda.current_stream())
    torch.cuda.synchronize()
    return nx.cpu().numpy()


def _check_row(logits, T, top_p, u, got):
    """True if compared exactly; asserts validity otherwise."""
    lg = np.asarray(logits, np.float64)
    want = oracle.sample_top_p(lg, T, top_p, float(u))
    p = oracle.softmax_t(lg, T)
    order = np.lexsort((np.arange(p.size), -p))
    cs = np.cumsum(p[order])
    ids, c = oracle.kept_cdf(lg, T, top_p)
    margin = min(np.min(np.abs(cs - top_p)), np.min(np.abs(c - u)))
    if margin > TOL:
        assert got == want, (got, want, margin)
        return True
    wide, _ = oracle.nucleus(p, top_p + TOL)
    assert got in set(wide.tolist()), (got, want)
    ids_w, c_w = oracle.kept_cdf(lg, T, min(1.0, top_p + TOL))
    k = int(np.flatnonzero(ids_w == got)[0])
    lo = c_w[k - 1] if k else 0.0
    assert lo - TOL <= u <= c_w[k] + TOL, (got, want, u, lo, c_w[k])
    return False


def test_greedy_rows_with_ties(qw):
    rng = np.random.default_rng(11)
    lg = rng.normal(0, 1, (5, V_FULL)).astype(np.float32)
    lg[2, [7, 90000, 151000]] = 9.0  # tie: the lowest index wins
    got = _gpu_sample(qw, lg, 0.0, 0.95, np.zeros(5))
    want = [int(np.flatnonzero(r == r.max())[0]) for r in lg]
    np.testing.assert_array_equal(got, want)


def _rows(kind, B, rng):
    if kind == "head":  # 20 tokens well above a Gaussian bulk: a short nucleus, wide CDF steps
        lg = rng.normal(0, 1, (B, V_FULL))
        for r in lg:
            r[rng.choice(V_FULL, 20, replace=False)] = 12.0 + 2.0 * rng.normal(0, 1, 20)
        return lg.astype(np.float32)
    return rng.normal(0, float(kind), (B, V_FULL)).astype(np.float32)


@pytest.mark.parametrize("kind,T,top_p", [("head", 1.0, 0.9), ("head", 0.5, 0.5), ("head", 0.7, 0.95),
                                          ("4.0", 1.0, 0.9), ("2.0", 0.7, 0.95), ("1.0", 1.0, 1.0),
                                          ("0.1", 1.0, 0.95), ("3.0", 1.3, 0.3)])
def test_rows_against_oracle(qw, kind, T, top_p):
    rng = np.random.default_rng(len(kind) * 1000 + int(T * 10 + top_p * 100))
    B = 12
    lg = _rows(kind, B, rng)
    u = rng.random(B)
    got = _gpu_sample(qw, lg, T, top_p, u)
    exact = sum(_check_row(lg[b], T, top_p, u[b], int(got[b])) for b in range(B))
    if kind == "head":
        assert exact >= B - 2  # short nucleus: nearly every draw is compared exactly


def test_ties_and_small_vocabularies(qw):
    rng = np.random.default_rng(5)
    for V in (17, 1000, 8191):
        # logits on a coarse grid: many exactly equal probabilities at the nucleus edge
        lg = (np.round(rng.normal(0, 2, (6, V)) * 2) / 2).astype(np.float32)
        u = rng.random(6)
        for top_p in (0.5, 0.9):
            got = _gpu_sample(qw, lg, 1.0, top_p, u)
            for b in range(6):
                _check_row(lg[b], 1.0, top_p, u[b], int(got[b]))


def test_stratified_draws_match_the_nucleus_distribution(qw):
    V, N = 5000, 4096
    rng = np.random.default_rng(9)
    row = rng.normal(0, 3, V).astype(np.float32)
    T, top_p = 0.8, 0.9
    u = (np.arange(N) + 0.5) / N
    got = _gpu_sample(qw, np.tile(row, (N, 1)), T, top_p, u)
    p = oracle.softmax_t(row.astype(np.float64), T)
    kept, _ = oracle.nucleus(p, top_p)
    want = np.zeros(V)
    want[kept] = p[kept] / p[kept].sum()
    freq = np.bincount(got, minlength=V) / N
    np.testing.assert_allclose(freq, want, rtol=0, atol=1.0 / N + 1e-4)


def test_deterministic_and_batch_independent(qw):
    rng = np.random.default_rng(21)
    lg = rng.normal(0, 1.5, (64, V_FULL)).astype(np.float32)
    u = rng.random(64)
    a = _gpu_sample(qw, lg, 0.9, 0.95, u)
    b = _gpu_sample(qw, lg, 0.9, 0.95, u)
    np.testing.assert_array_equal(a, b)
    c = np.array([_gpu_sample(qw, lg[i:i + 1], 0.9, 0.95, u[i:i + 1])[0] for i in (0, 31, 63)])
    np.testing.assert_array_equal(c, a[[0, 31, 63]])


def test_model_logits(qw):
    """Logits of a prefill (one block + tied head), then sampling as the page's loop does."""
    s = synth.ONE_BLOCK
    eng = engine(qw, s, max_tokens=64, max_batch=8, max_context=256, kv_pages=64, max_seqs=8)
    try:
        run = Run(qw, eng)
        prompts = [synth.make_tokens(s.vocab, n, 40 + n).tolist() for n in (5, 9, 3, 12)]
        g = run.prefill(list(range(4)), prompts, debug=False)
        lg = g["logits"].astype(np.float32)
        u = np.random.default_rng(4).random(4)
        for T, top_p in ((0.7, 0.9), (0.05, 0.95)):
            got = _gpu_sample(qw, lg, T, top_p, u)
            for b in range(4):
                _check_row(lg[b], T, top_p, u[b], int(got[b]))
    finally:
        eng.close()


def test_argument_errors(qw):
    import torch
    lg = torch.zeros((2, 10), device="cuda")
    u = torch.zeros(2, device="cuda")
    nx = torch.zeros(2, dtype=torch.int32, device="cuda")
    for args in ((0, 10, 10, 1.0, 0.9), (2, 10, 5, 1.0, 0.9), (2, 10, 10, -1.0, 0.9), (2, 10, 10, 1.0, 0.0),
                 (2, 10, 10, 1.0, 1.5), (2, 10, 10, float("nan"), 0.9)):
        B, V, ld, T, tp = args
        with pytest.raises(qw.qw.QwError):
            qw.qw.qw_sample_top_p(B, V, lg.data_ptr(), ld, T, tp, u.data_ptr(), nx.data_ptr())
