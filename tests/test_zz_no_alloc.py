"""The LM-head entry point that allocates nothing (its argmax scratch is a static device
array) against the oracle and against the decode step it mirrors.

It exists for callers that cannot call cudaMalloc where they need the result (a fixed
device budget owned by another framework, a serving loop that never allocates after
start-up). This file is collected last so a failure here stops a -x run only after every
other test has run.

For 1-3 rows the decode step's LM head is the same GEMV kernel on the same rows, so the two
must agree bit for bit; from 4 rows the decode step's head runs on the tensor cores (fp16
operands) and the two agree within the logits tolerance. B = 8 fills the whole static
array."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, check_logits, check_token, engine, weights

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [3, 1, 8])
def test_noalloc_lm_head_matches_oracle_and_decode_step(qw, B):
    import torch
    s = synth.ONE_BLOCK
    eng = engine(qw, s, max_tokens=64, max_batch=8, max_context=256, kv_pages=64, max_seqs=8)
    try:
        run = Run(qw, eng)
        om = oracle.Model(weights(s))
        fin = synth.bf16_bits_to_f32(weights(s).final_norm).astype(np.float64)
        seqs = list(range(B))
        prompts = [synth.make_tokens(s.vocab, 2 + b, 4100 + b).tolist() for b in range(B)]
        g = run.prefill(seqs, prompts, debug=False, reserve_extra=2)
        d = run.decode(seqs, g["next"].tolist(), debug=True)   # existing entry point
        assert d["status"] == 0
        x_np = d["hidden"][-1]                                    # residual rows after the last layer
        want = om.lm_head(oracle.rms_norm(x_np, fin, s.rms_eps))  # oracle on the same rows
        x_last = torch.tensor(x_np, dtype=torch.float32, device="cuda").contiguous()
        for _ in range(2):                                        # two calls in a row
            logits = torch.empty((B, s.vocab), dtype=torch.float32, device="cuda")
            nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
            qw.qw.qw_lm_head_argmax_noalloc(eng.model, B, x_last.data_ptr(), logits.data_ptr(), nxt.data_ptr(),
                                            eng.stream)
            eng.stream.synchronize()
            lg = logits.cpu().numpy().astype(np.float64)
            ids = nxt.cpu().numpy()
            for b in range(B):
                check_logits(lg[b], want[b])
                check_token(ids[b], want[b])
            if B < 4:
                np.testing.assert_array_equal(lg, d["logits"])
                np.testing.assert_array_equal(ids, d["next"])
            else:
                for b in range(B):
                    check_logits(lg[b], d["logits"][b])
        with pytest.raises(qw.qw.QwError):
            qw.qw.qw_lm_head_argmax_noalloc(eng.model, 9, x_last.data_ptr(), 0, nxt.data_ptr(), eng.stream)
    finally:
        eng.close()
