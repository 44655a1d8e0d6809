"""The LM-head entry point that allocates nothing (its argmax scratch is a static device
array) gives the same logits and greedy ids as the decode step it mirrors.

It exists for callers that cannot call cudaMalloc where they need the result (a fixed
device budget owned by another framework, a serving loop that never allocates after
start-up). This file is collected last so a failure here stops a -x run only after every
other test has run."""

import numpy as np
import pytest

import synth
from gpu_util import Run, check_logits, engine

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [3, 1])
def test_noalloc_lm_head_matches_decode_step(qw, B):
    import torch
    s = synth.ONE_BLOCK
    eng = engine(qw, s, max_tokens=64, max_batch=8, max_context=256, kv_pages=64, max_seqs=8)
    try:
        run = Run(qw, eng)
        seqs = list(range(B))
        prompts = [synth.make_tokens(s.vocab, 2 + b, 4100 + b).tolist() for b in range(B)]
        g = run.prefill(seqs, prompts, debug=False, reserve_extra=2)
        d = run.decode(seqs, g["next"].tolist(), debug=True)   # existing entry point
        assert d["status"] == 0
        x_last = torch.tensor(d["hidden"][-1], dtype=torch.float32, device="cuda").contiguous()
        for _ in range(2):                                        # two calls in a row
            logits = torch.empty((B, s.vocab), dtype=torch.float32, device="cuda")
            nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
            qw.qw.qw_lm_head_argmax_noalloc(eng.model, B, x_last.data_ptr(), logits.data_ptr(), nxt.data_ptr(),
                                            eng.stream)
            eng.stream.synchronize()
            check_logits(logits.cpu().numpy().astype(np.float64), d["logits"])
            np.testing.assert_array_equal(nxt.cpu().numpy(), d["next"])
        with pytest.raises(qw.qw.QwError):
            qw.qw.qw_lm_head_argmax_noalloc(eng.model, 9, x_last.data_ptr(), 0, nxt.data_ptr(), eng.stream)
    finally:
        eng.close()
