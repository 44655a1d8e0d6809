"""Host logic of bench.py's roofline accounting, on the CPU: the per-launch algorithmic bytes
of every kernel a batch-1 decode step launches (cluster path and launch-per-phase path) add
up to the step's own byte count up to the activation vectors, so the two views the bench
reports describe the same work; the ncu traffic figure follows its source file (edited or
missing: none)."""

import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

S = synth.QWEN3_0_6B


def _act_bound(s, B):
    """A generous bound on the non-weight, non-KV bytes of one decode step: every activation
    vector a layer passes between launches (x, partial sums, q|k|v, the SwiGLU activation,
    logits-free), in fp32, 64 of them per layer and token."""
    return s.n_layers * B * 64 * max(s.hidden, s.inter) * 4


@pytest.mark.parametrize("ctx", [0.0, 37.0, 100.0])
def test_cluster_path_launches_add_up_to_the_step(ctx):
    """Per layer one attention-side and one MLP-side cluster launch, then the LM head: the
    weights and the KV bytes of the launches equal the step's; the rest is activations."""
    L = S.n_layers
    per_step = L * (bench.kernel_bytes(3, S, 1, 1, ctx, clusters=True) +
                    bench.kernel_bytes(5, S, 1, 1, ctx, clusters=True)) + bench.kernel_bytes(7, S, 1, 1)
    step = bench.step_bytes(S, 1, ctx)
    assert per_step >= step - S.hidden * 2 - 1          # every weight and K/V byte is counted
    assert per_step - step <= _act_bound(S, 1)           # the excess is activations only
    assert (per_step - step) / step < 5e-3


@pytest.mark.parametrize("ctx", [0.0, 37.0, 100.0])
def test_launch_per_phase_launches_add_up_to_the_step(ctx):
    """q|k|v, attention fused with o_proj, gate/up and down per layer, then the LM head (one
    token): the same weight and K/V bytes as the step; the step's new K/V and embedding row
    are the only bytes the launches do not count."""
    L = S.n_layers
    per_layer = sum(bench.kernel_bytes(k, S, 1, 1, ctx) for k in (1, 3, 5, 6))
    per_step = L * per_layer + bench.kernel_bytes(7, S, 1, 1)
    step = bench.step_bytes(S, 1, ctx)
    new_kv_and_embedding = L * 2 * S.n_kv_heads * S.head_dim * 2 + S.hidden * 2
    assert per_step >= step - new_kv_and_embedding
    assert per_step - step <= _act_bound(S, 1)
    assert (per_step - step) / step < 5e-3


def test_step_bytes_of_the_default_workload():
    """1.196 GB per batch-1 step at the bench's mean cache (5 + 32 keys): the figure the
    step roofline divides."""
    b = bench.step_bytes(S, 1, 5 + 64 / 2)
    w = S.n_layers * ((S.n_heads * 128 + 2 * S.n_kv_heads * 128) * S.hidden + S.hidden * S.n_heads * 128 +
                      3 * S.inter * S.hidden) * 2 + S.vocab * S.hidden * 2
    assert w < b < w * 1.01
    assert b == pytest.approx(1.19633e9, rel=1e-4)


def test_ncu_traffic_follows_the_source(tmp_path, monkeypatch):
    """The traffic of an entry is reported while its source file hashes to the captured
    sha256 and is None once the file differs or is missing."""
    src = tmp_path / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    table = {(9, "k"): (1234, str(src), sha), (9, "gone"): (5, str(tmp_path / "none.cu"), sha)}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", table)
    assert bench.ncu_traffic(9, "k") == 1234
    assert bench.ncu_traffic(9, "gone") is None
    assert bench.ncu_traffic(9, "other") is None
    src.write_bytes(b"__global__ void k() { }\n")
    assert bench.ncu_traffic(9, "k") is None


def test_traffic_entries_name_existing_sources():
    for (cfg, name), (nbytes, src, sha) in bench.NCU_TRAFFIC.items():
        assert cfg in bench.CONFIGS
        assert os.path.exists(os.path.join(ROOT, src)), src
