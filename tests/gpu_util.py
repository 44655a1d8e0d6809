"""Helpers shared by the GPU parity tests: build an engine from seeded weights, run the
library through its C ABI, and compare with the oracle under the stated tolerances."""

from __future__ import annotations

import functools

import numpy as np

import synth

# Tolerances of the GPU-vs-oracle comparison.
HIDDEN_REL = 5e-3   # ||x_gpu - x_oracle|| / ||x_oracle|| per layer and token
LOGITS_ABS = 5e-2   # max |logit_gpu - logit_oracle|
TOP2_GAP = 1e-2     # greedy ids must agree when the oracle's top-2 gap exceeds this


@functools.lru_cache(maxsize=4)
def weights(shape: synth.Shape, seed: int = 0) -> synth.Weights:
    w = synth.Weights(shape, seed)
    for _ in w.named():
        pass
    return w


def engine(pkg, shape, max_tokens=64, max_batch=8, max_context=1024, kv_pages=512, max_seqs=16,
           seed=0):
    return pkg.qw.Engine(shape, dict(weights(shape, seed).named()), max_tokens=max_tokens,
                         max_batch=max_batch, max_context=max_context, kv_pages=kv_pages,
                         max_seqs=max_seqs)


class Run:
    """Drives one engine through the C ABI with torch buffers on the engine's stream."""

    def __init__(self, pkg, eng):
        import torch
        self.torch = torch
        self.qw = pkg.qw
        self.eng = eng
        self.s = eng.shape

    def _t(self, arr, dtype):
        return self.torch.tensor(np.asarray(arr), dtype=dtype, device="cuda")

    def prefill(self, seq_ids, prompts, debug=True, logits=True, reserve_extra=0, reserve=True, check=True):
        torch, qw, eng = self.torch, self.qw, self.eng
        lens = [len(p) for p in prompts]
        if reserve:
            for s, n in zip(seq_ids, lens):
                qw.qw_kv_reserve(eng.kv, s, n + reserve_extra, eng.stream)
        T = sum(lens)
        toks = self._t(np.concatenate([np.asarray(p, np.int32) for p in prompts]), torch.int32)
        return self._step(lambda lg, nx: qw.qw_prefill(eng.model, eng.kv, seq_ids, lens, toks.data_ptr(), lg, nx,
                                                        eng.stream), len(seq_ids), T, debug, logits, check)

    def decode(self, seq_ids, tokens, debug=True, logits=True, check=True):
        torch, qw, eng = self.torch, self.qw, self.eng
        toks = self._t(np.asarray(tokens, np.int32), torch.int32)
        return self._step(lambda lg, nx: qw.qw_decode_step(eng.model, eng.kv, seq_ids, toks.data_ptr(), lg, nx,
                                                            eng.stream), len(seq_ids), len(seq_ids), debug, logits,
                          check)

    def _step(self, call, B, T, debug, logits, check=True):
        torch, qw, eng, s = self.torch, self.qw, self.eng, self.s
        lg = torch.empty((B, s.vocab), dtype=torch.float32, device="cuda") if logits else None
        nx = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        out = {}
        if debug:
            hid = torch.empty((s.n_layers, T, s.hidden), dtype=torch.float32, device="cuda")
            pos = torch.full((T,), -1, dtype=torch.int32, device="cuda")
            slot = torch.full((T,), -1, dtype=torch.int32, device="cuda")
            qw.qw_debug_set(eng.model, hid.data_ptr(), pos.data_ptr(), slot.data_ptr())
        try:
            call(lg.data_ptr() if lg is not None else 0, nx.data_ptr())
        finally:
            if debug:
                qw.qw_debug_set(eng.model, 0, 0, 0)
        st = qw.qw_sync_status(eng.model, eng.stream)
        if check:
            assert st == 0, f"device status {st}: {qw.qw_last_error()}"
        out["status"] = st
        out["next"] = nx.cpu().numpy()
        if lg is not None:
            out["logits"] = lg.cpu().numpy().astype(np.float64)
        if debug:
            out["hidden"] = hid.cpu().numpy().astype(np.float64)
            out["pos"] = pos.cpu().numpy()
            out["slot"] = slot.cpu().numpy()
        return out


def rel_err(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def check_hidden(gpu_h, orc_h, tol=HIDDEN_REL):
    """gpu_h, orc_h: [L, n, D]. Normwise error per layer and token."""
    assert gpu_h.shape == orc_h.shape, (gpu_h.shape, orc_h.shape)
    worst = 0.0
    for l in range(orc_h.shape[0]):
        for t in range(orc_h.shape[1]):
            e = rel_err(gpu_h[l, t], orc_h[l, t])
            worst = max(worst, e)
            assert e <= tol, f"layer {l} token {t}: ||dx||/||x|| = {e:.3e} > {tol}"
    return worst


def check_logits(gpu_l, orc_l, tol=LOGITS_ABS):
    err = float(np.max(np.abs(gpu_l - orc_l)))
    assert err <= tol, f"max |dlogit| = {err:.3e} > {tol}"
    return err


def top2_gap(logits):
    top = np.partition(logits, -2)[-2:]
    return float(top[1] - top[0])


def check_token(gpu_id, orc_logits):
    """Greedy ids must agree whenever the oracle's top-2 gap exceeds TOP2_GAP. Returns True if
    the ids agree."""
    want = int(np.argmax(orc_logits))
    if top2_gap(orc_logits) > TOP2_GAP:
        assert int(gpu_id) == want, f"greedy id {gpu_id} != oracle {want} (gap {top2_gap(orc_logits):.3e})"
    return int(gpu_id) == want
