"""GPU parity of the weight-only grouped affine quantization ("Lo que omite el script": 4- and
8-bit weights) on one Qwen3-0.6B-shaped block: the codes and the fp16 (scale, bias) words of
qw_quantize_weights bit-exact against the oracle's quantizer, and the quantized model (the
GEMV path reading codes, the tensor-core path using the dequantized weights) against the
oracle over the dequantized weights, under the usual tolerances."""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import Run, check_hidden, check_logits, check_token, weights
from oracle import quant

pytestmark = pytest.mark.gpu

S1 = synth.ONE_BLOCK


def _align(n, a=256):
    return (n + a - 1) // a * a


def _layer0_mats(w):
    d = w.layer(0)
    qkv = np.concatenate([d["self_attn.q_proj.weight"], d["self_attn.k_proj.weight"], d["self_attn.v_proj.weight"]])
    return [qkv, d["self_attn.o_proj.weight"], d["mlp.gate_proj.weight"], d["mlp.up_proj.weight"],
            d["mlp.down_proj.weight"]]


def _engine(qw, bits):
    eng = qw.qw.Engine(S1, dict(weights(S1).named()), max_tokens=256, max_batch=8, max_context=512,
                       kv_pages=128, max_seqs=8)
    eng.quantize(bits)
    return eng


@pytest.mark.parametrize("bits", [8, 4])
def test_codes_and_scales_bit_exact(qw, bits):
    eng = _engine(qw, bits)
    try:
        buf = eng.qbuf.cpu().numpy()
        off = 0
        for m in _layer0_mats(weights(S1)):
            rows, k = m.shape
            nc, ns = rows * k * bits // 8, rows * (k // 64) * 4
            codes = buf[off:off + nc]
            off = _align(off + nc)
            sb = buf[off:off + ns].view(np.uint32).reshape(rows, k // 64)
            off = _align(off + ns)
            want_q, want_s, want_b = quant.quantize(m, bits)
            if bits == 4:
                codes = np.stack([codes & 0xF, codes >> 4], axis=1).reshape(-1)
            np.testing.assert_array_equal(codes.reshape(rows, k), want_q)
            np.testing.assert_array_equal((sb & 0xFFFF).astype(np.uint16), want_s.view(np.uint16))
            np.testing.assert_array_equal((sb >> 16).astype(np.uint16), want_b.view(np.uint16))
    finally:
        eng.close()


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_model_parity(qw, bits):
    om = oracle.Model(quant.QuantizedWeights(weights(S1), bits))
    eng = _engine(qw, bits)
    try:
        run = Run(qw, eng)
        # small-batch path (GEMVs over the codes): prefill 5 tokens, then greedy decode
        prompt = synth.make_tokens(S1.vocab, 5, 4100 + bits).tolist()
        run.qw.qw_kv_reserve(eng.kv, 0, 5 + 6, eng.stream)
        cache = oracle.SeqCache(S1.n_layers)
        g = run.prefill([0], [prompt], reserve=False)
        o = oracle.forward(om, prompt, cache)
        check_hidden(g["hidden"], o["hidden"])
        check_logits(g["logits"][0], o["logits"])
        tok = int(g["next"][0])
        same = check_token(tok, o["logits"])
        for _ in range(6):
            if not same:
                break
            o = oracle.forward(om, [tok], cache)
            d = run.decode([0], [tok])
            check_hidden(d["hidden"], o["hidden"])
            check_logits(d["logits"][0], o["logits"])
            same = check_token(d["next"][0], o["logits"])
            tok = int(d["next"][0])
        # tensor-core path (the dequantized fp16 weights): a 150-token prefill
        p2 = synth.make_tokens(S1.vocab, 150, 4200 + bits).tolist()
        g = run.prefill([1], [p2])
        o = oracle.forward(om, p2, oracle.SeqCache(S1.n_layers))
        check_hidden(g["hidden"], o["hidden"])
        check_logits(g["logits"][0], o["logits"])
        check_token(g["next"][0], o["logits"])
    finally:
        eng.close()


def test_quantize_errors(qw):
    eng = _engine(qw, 8)
    try:
        with pytest.raises(qw.qw.QwError):  # already quantized
            qw.qw.qw_quantize_weights(eng.model, 4, eng.qbuf.data_ptr(), eng.qbuf.numel())
        assert qw.qw.qw_quantize_bytes(eng.model, 5) == 0
    finally:
        eng.close()
