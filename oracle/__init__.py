"""CPU oracle for the Qwen3-style decoder forward pass (prefill + greedy decode) and for
temperature + top-p sampling.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, fp64 NumPy restatement of the
computation described on the page "Dentro de un LLM: Inferencia en Python puro para
Qwen3-0.6B en MLX" (Pasos 2-9). It exists to check the CUDA library against. Only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import or run it. The CUDA library never imports it and shares no code,
tables or constants with it; the two meet only through the seeded inputs of ``synth``.
"""

from .qwen3 import (  # noqa: F401
    Model,
    SeqCache,
    PagedKVMirror,
    rms_norm,
    rope_angles,
    apply_rope,
    silu,
    gqa_attention,
    ffn,
    decoder_layer,
    forward,
    generate,
    argmax_lowest,
)
from .sampling import (  # noqa: F401
    softmax_t,
    nucleus,
    kept_cdf,
    sample as sample_top_p,
)
from . import quant  # noqa: F401
