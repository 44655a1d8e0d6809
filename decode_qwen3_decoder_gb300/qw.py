"""ctypes binding of libqw (include/qw.h): argument marshalling only.

Every function here has the name of the C entry point it calls and forwards plain device
pointers, sizes and the stream handle. All arithmetic runs in the library's CUDA kernels;
there is no Python or CPU path. ``load()`` raises if the library is missing.

``Engine`` is a convenience owner of the device memory (torch tensors) that the library
borrows: the workspace, the weights and the KV pool.
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

from . import _build

QW_OK = 0
STATUS_NAMES = {0: "QW_OK", -1: "QW_ERR_INVALID_ARG", -2: "QW_ERR_KV_FULL", -3: "QW_ERR_BAD_STATE",
                -4: "QW_ERR_CUDA", -5: "QW_ERR_BAD_TOKEN", -6: "QW_ERR_TIMEOUT",
                -7: "QW_ERR_UNSUPPORTED", -8: "QW_ERR_BAD_POS", -9: "QW_ERR_RANGE"}


class QwError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class qw_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("inter", ctypes.c_int),
                ("vocab", ctypes.c_int), ("page_size", ctypes.c_int), ("tie_embed", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
                ("max_tokens", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("max_context", ctypes.c_int)]


LAYER_FIELDS = ("input_layernorm", "q_proj", "k_proj", "v_proj", "o_proj", "q_norm", "k_norm",
                "post_attention_layernorm", "gate_proj", "up_proj", "down_proj")


class qw_layer_ptrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_FIELDS]


class qw_weight_ptrs(ctypes.Structure):
    _fields_ = [("embed_tokens", ctypes.c_void_p), ("norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(qw_layer_ptrs))]


_LIB: Optional[ctypes.CDLL] = None
_VP, _I, _SZ, _P = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER

# name -> (restype, argtypes); mirrors include/qw.h
SIGNATURES = {
    "qw_model_workspace_bytes": (_SZ, [_P(qw_config)]),
    "qw_init_weights": (_I, [_P(qw_config), _P(qw_weight_ptrs), _VP, _SZ, _VP, _P(_VP)]),
    "qw_kv_pool_bytes": (_SZ, [_VP, _I, _I]),
    "qw_kv_alloc": (_I, [_VP, _VP, _SZ, _I, _VP, _P(_VP)]),
    "qw_kv_reserve": (_I, [_VP, _I, _I, _VP]),
    "qw_kv_reset": (_I, [_VP, _I, _VP]),
    "qw_kv_free_pages": (_I, [_VP]),
    "qw_kv_truncate": (_I, [_VP, _I, _I, _VP]),
    "qw_kv_length": (_I, [_VP, _I]),
    "qw_prefill": (_I, [_VP, _VP, _I, _P(_I), _P(_I), _VP, _VP, _VP, _VP]),
    "qw_decode_step": (_I, [_VP, _VP, _I, _P(_I), _VP, _VP, _VP, _VP]),
    "qw_decode_steps": (_I, [_VP, _VP, _I, _P(_I), _I, _VP, _VP, _VP]),
    "qw_generate": (_I, [_VP, _VP, _I, _P(_I), _P(_I), _P(ctypes.c_int32), _I,
                         _P(ctypes.c_int32), _VP]),
    "qw_generate_eos": (_I, [_VP, _VP, _I, _P(_I), _P(_I), _P(ctypes.c_int32), _I, _I,
                             _P(ctypes.c_int32), _P(ctypes.c_int32), _VP]),
    "qw_sync_status": (_I, [_VP, _VP]),
    "qw_last_error": (ctypes.c_char_p, []),
    "qw_free_model": (None, [_VP]),
    "qw_free_kv": (None, [_VP]),
    "qw_debug_set": (_I, [_VP, _VP, _VP, _VP]),
    "qw_quantize_bytes": (_SZ, [_VP, _I]),
    "qw_quantize_weights": (_I, [_VP, _I, _VP, _SZ, _VP]),
    "qw_sample_top_p": (_I, [_I, _I, _VP, _SZ, ctypes.c_float, ctypes.c_float, _VP, _VP, _VP]),
    "qw_debug_set_attn": (_I, [_VP, _VP]),
    "qw_kv_page_table": (_I, [_VP, _I, _P(ctypes.c_int32), _I]),
    "qw_kv_pool_ptrs": (_I, [_VP, _P(_VP), _P(_VP), _P(_I)]),
    "qw_kv_fill_synthetic": (_I, [_VP, _I, _I, ctypes.c_uint64, _VP]),
    "qw_last_launch_count": (_I, [_VP]),
    "qw_profile_set": (_I, [_VP, _I, _P(_VP), _I]),
    "qw_set_option": (_I, [_VP, _I, _I]),
    "qw_trace_set": (_I, [_VP, _VP, _I]),
    "qw_lm_head_argmax_noalloc": (_I, [_VP, _I, _VP, _VP, _VP, _VP]),
}


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libqw.so (built in-tree). Raises if it does not exist: there is no fallback."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libqw.so not found at {path}: run decode_qwen3_decoder_gb300.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == _build.LIB:
        _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != QW_OK:
        raise QwError(status, load().qw_last_error().decode())


def _ints(vals: Sequence[int]):
    arr = (ctypes.c_int * len(vals))(*[int(v) for v in vals])
    return arr


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


# ---- thin wrappers with the C names ---------------------------------------------------

def qw_model_workspace_bytes(cfg: qw_config) -> int:
    return load().qw_model_workspace_bytes(ctypes.byref(cfg))


def qw_init_weights(cfg: qw_config, w: qw_weight_ptrs, workspace_ptr: int, ws_bytes: int,
                    stream=None) -> int:
    out = ctypes.c_void_p()
    _check(load().qw_init_weights(ctypes.byref(cfg), ctypes.byref(w), workspace_ptr, ws_bytes,
                                  _stream(stream), ctypes.byref(out)))
    return out.value


def qw_kv_pool_bytes(model: int, n_pages: int, max_seqs: int) -> int:
    return load().qw_kv_pool_bytes(model, n_pages, max_seqs)


def qw_kv_alloc(model: int, pool_ptr: int, pool_bytes: int, max_seqs: int, stream=None) -> int:
    out = ctypes.c_void_p()
    _check(load().qw_kv_alloc(model, pool_ptr, pool_bytes, max_seqs, _stream(stream), ctypes.byref(out)))
    return out.value


def qw_kv_reserve(kv: int, seq_id: int, total_tokens: int, stream=None) -> None:
    _check(load().qw_kv_reserve(kv, seq_id, total_tokens, _stream(stream)))


def qw_kv_reset(kv: int, seq_id: int, stream=None) -> None:
    _check(load().qw_kv_reset(kv, seq_id, _stream(stream)))


def qw_kv_truncate(kv: int, seq_id: int, n_tokens: int, stream=None) -> None:
    _check(load().qw_kv_truncate(kv, seq_id, n_tokens, _stream(stream)))


def qw_kv_free_pages(kv: int) -> int:
    return load().qw_kv_free_pages(kv)


def qw_kv_length(kv: int, seq_id: int) -> int:
    return load().qw_kv_length(kv, seq_id)


def qw_prefill(model: int, kv: int, seq_ids: Sequence[int], lens: Sequence[int], tokens_ptr: int,
               logits_ptr: int, next_ptr: int, stream=None) -> None:
    _check(load().qw_prefill(model, kv, len(seq_ids), _ints(seq_ids), _ints(lens), tokens_ptr,
                             logits_ptr or None, next_ptr, _stream(stream)))


def qw_decode_step(model: int, kv: int, seq_ids: Sequence[int], tokens_ptr: int, logits_ptr: int,
                   next_ptr: int, stream=None) -> None:
    _check(load().qw_decode_step(model, kv, len(seq_ids), _ints(seq_ids), tokens_ptr,
                                 logits_ptr or None, next_ptr, _stream(stream)))


def qw_decode_steps(model: int, kv: int, seq_ids: Sequence[int], n_steps: int, tokens_ptr: int, out_ptr: int,
                    stream=None) -> None:
    _check(load().qw_decode_steps(model, kv, len(seq_ids), _ints(seq_ids), n_steps, tokens_ptr, out_ptr,
                                  _stream(stream)))


def qw_generate(model: int, kv: int, seq_ids: Sequence[int], lens: Sequence[int], host_prompt,
                n_decode: int, host_out, stream=None) -> None:
    """host_prompt / host_out: contiguous int32 numpy arrays (sum(lens)) / (B, n_decode + 1)."""
    import numpy as np
    assert host_prompt.dtype == np.int32 and host_prompt.flags.c_contiguous
    assert host_out.dtype == np.int32 and host_out.flags.c_contiguous
    _check(load().qw_generate(model, kv, len(seq_ids), _ints(seq_ids), _ints(lens),
                              host_prompt.ctypes.data_as(_P(ctypes.c_int32)), n_decode,
                              host_out.ctypes.data_as(_P(ctypes.c_int32)), _stream(stream)))


def qw_generate_eos(model: int, kv: int, seq_ids: Sequence[int], lens: Sequence[int], host_prompt,
                    n_decode: int, eos_id: int, host_out, host_counts, stream=None) -> None:
    """As qw_generate with an EOS stop; host_counts: int32 numpy array (B)."""
    import numpy as np
    for a in (host_prompt, host_out, host_counts):
        assert a.dtype == np.int32 and a.flags.c_contiguous
    _check(load().qw_generate_eos(model, kv, len(seq_ids), _ints(seq_ids), _ints(lens),
                                  host_prompt.ctypes.data_as(_P(ctypes.c_int32)), n_decode, eos_id,
                                  host_out.ctypes.data_as(_P(ctypes.c_int32)),
                                  host_counts.ctypes.data_as(_P(ctypes.c_int32)), _stream(stream)))


def qw_sync_status(model: int, stream=None) -> int:
    return load().qw_sync_status(model, _stream(stream))


def qw_last_error() -> str:
    return load().qw_last_error().decode()


def qw_free_model(model: int) -> None:
    load().qw_free_model(model)


def qw_free_kv(kv: int) -> None:
    load().qw_free_kv(kv)


def qw_debug_set(model: int, hidden_ptr: int, pos_ptr: int, slot_ptr: int) -> None:
    _check(load().qw_debug_set(model, hidden_ptr or None, pos_ptr or None, slot_ptr or None))


def qw_debug_set_attn(model: int, attn_ptr: int) -> None:
    _check(load().qw_debug_set_attn(model, attn_ptr or None))


def qw_quantize_bytes(model: int, bits: int) -> int:
    return load().qw_quantize_bytes(model, bits)


def qw_quantize_weights(model: int, bits: int, buf_ptr: int, nbytes: int, stream=None) -> None:
    _check(load().qw_quantize_weights(model, bits, buf_ptr, nbytes, _stream(stream)))


def qw_sample_top_p(B: int, vocab: int, logits_ptr: int, ld: int, temperature: float, top_p: float,
                    uniform_ptr: int, next_ptr: int, stream=None) -> None:
    _check(load().qw_sample_top_p(B, vocab, logits_ptr, ld, temperature, top_p, uniform_ptr or None, next_ptr,
                                  _stream(stream)))


def qw_kv_page_table(kv: int, seq_id: int, max_pages: int = 1 << 16):
    import numpy as np
    out = np.zeros(max_pages, np.int32)
    n = load().qw_kv_page_table(kv, seq_id, out.ctypes.data_as(_P(ctypes.c_int32)), max_pages)
    if n < 0:
        _check(n)
    return out[:n].copy()


def qw_kv_pool_ptrs(kv: int):
    k, v, n = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int()
    _check(load().qw_kv_pool_ptrs(kv, ctypes.byref(k), ctypes.byref(v), ctypes.byref(n)))
    return k.value, v.value, n.value


def qw_kv_fill_synthetic(kv: int, seq_id: int, n_tokens: int, seed: int, stream=None) -> None:
    _check(load().qw_kv_fill_synthetic(kv, seq_id, n_tokens, seed, _stream(stream)))


def qw_last_launch_count(model: int) -> int:
    return load().qw_last_launch_count(model)


def qw_lm_head_argmax_noalloc(model: int, B: int, x_ptr: int, logits_ptr: int, next_ptr: int,
                              stream=None) -> None:
    """LM head + argmax over B residual rows with no device allocation (scratch is a static
    device array of QW_NOALLOC_MAX_ROWS keys); see include/qw.h."""
    _check(load().qw_lm_head_argmax_noalloc(model, B, x_ptr, logits_ptr or None, next_ptr, _stream(stream)))


QW_OPT_PDL = 2
QW_OPT_SPLIT_DECODE = 3
QW_OPT_DECODE_STEP_KERNEL = 4
QW_OPT_STEP_PROJ_CTAS = 5
QW_OPT_TEST_WAIT_LIMIT_US = 6
QW_OPT_TEST_EXTRA_ARRIVALS = 7
QW_OPT_BATCH1_CLUSTERS = 8

QW_MAX_GRAPH_STEPS = 64   # most decode steps of one qw_decode_steps call


def qw_set_option(model: int, option: int, value: int) -> None:
    _check(load().qw_set_option(model, option, value))


def qw_trace_set(model: int, buf_ptr: int, per_cta: int) -> None:
    _check(load().qw_trace_set(model, buf_ptr or None, per_cta))


def qw_profile_set(model: int, kind: int, events, n_events: int) -> None:
    """events: a ctypes array of cudaEvent_t handles (or None to turn profiling off)."""
    _check(load().qw_profile_set(model, kind, events, n_events))


# ---- owner of the borrowed device memory ----------------------------------------------

def make_config(shape, max_tokens: int, max_batch: int, max_context: int) -> qw_config:
    return qw_config(n_layers=shape.n_layers, hidden=shape.hidden, n_heads=shape.n_heads,
                     n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, inter=shape.inter,
                     vocab=shape.vocab, page_size=shape.page_size, tie_embed=1,
                     rms_eps=shape.rms_eps, rope_theta=shape.rope_theta, max_tokens=max_tokens,
                     max_batch=max_batch, max_context=max_context)


class Engine:
    """Allocates (torch) the workspace, weights and KV pool that libqw borrows.

    ``weights`` maps HF tensor names to bf16 tensors already on the device (or to uint16
    numpy arrays of bf16 bits, which are uploaded)."""

    def __init__(self, shape, weights: Dict[str, object], max_tokens: int, max_batch: int,
                 max_context: int, kv_pages: int, max_seqs: int, stream=None):
        import numpy as np
        import torch
        self.shape = shape
        self.dev = torch.device("cuda")
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.cfg = make_config(shape, max_tokens, max_batch, max_context)
        ws = qw_model_workspace_bytes(self.cfg)
        if ws == 0:
            raise QwError(-1, "configuration rejected by qw_model_workspace_bytes")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.dev)
        self._w: Dict[str, object] = {}
        with torch.cuda.stream(self.stream):
            for name, t in weights.items():
                if isinstance(t, np.ndarray):
                    t = torch.from_numpy(t.view(np.int16)).to(self.dev, non_blocking=False).view(torch.bfloat16)
                self._w[name] = t
        torch.cuda.synchronize()
        layers = (qw_layer_ptrs * shape.n_layers)()
        for i in range(shape.n_layers):
            for f in LAYER_FIELDS:
                key = f"model.layers.{i}.{self._hf_suffix(f)}"
                setattr(layers[i], f, self._w[key].data_ptr())
        self._layers = layers
        wp = qw_weight_ptrs(embed_tokens=self._w["model.embed_tokens.weight"].data_ptr(),
                            norm=self._w["model.norm.weight"].data_ptr(), layers=layers)
        self.model = qw_init_weights(self.cfg, wp, self.workspace.data_ptr(), ws, self.stream)
        # the packed copies are done once the stream passes them; keep only the embedding
        self.stream.synchronize()
        self.embed = self._w["model.embed_tokens.weight"]
        self._w = {"model.embed_tokens.weight": self.embed}
        pool = qw_kv_pool_bytes(self.model, kv_pages, max_seqs)
        self.pool = torch.empty(pool, dtype=torch.uint8, device=self.dev)
        self.kv = qw_kv_alloc(self.model, self.pool.data_ptr(), pool, max_seqs, self.stream)
        self.stream.synchronize()

    @staticmethod
    def _hf_suffix(field: str) -> str:
        if field in ("input_layernorm", "post_attention_layernorm"):
            return f"{field}.weight"
        if field in ("q_proj", "k_proj", "v_proj", "o_proj", "q_norm", "k_norm"):
            return f"self_attn.{field}.weight"
        return f"mlp.{field}.weight"

    def quantize(self, bits: int) -> None:
        """Quantize the layers' projections (qw_quantize_weights) into a buffer this engine
        keeps alive."""
        import torch
        n = qw_quantize_bytes(self.model, bits)
        if n == 0:
            raise ValueError("bits must be 8 or 4")
        self.qbuf = torch.empty(n, dtype=torch.uint8, device=self.dev)
        qw_quantize_weights(self.model, bits, self.qbuf.data_ptr(), n, self.stream)
        self.stream.synchronize()

    def close(self) -> None:
        if getattr(self, "kv", None):
            qw_free_kv(self.kv)
            self.kv = None
        if getattr(self, "model", None):
            qw_free_model(self.model)
            self.model = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
