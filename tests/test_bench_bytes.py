"""The roofline numerator of bench.py (bytes a decode step must move), checked on CPU
against quantities computed another way: the byte size of the weight tensors the seeded
generator actually makes, and the increments one more cached key or one more routed
expert must add."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

TINY_MOE = synth.ModelConfig("tiny-moe", n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2,
                             head_dim=64, ffn_dim=0, vocab=4096, n_experts=8, top_k=2,
                             expert_ffn_dim=128, max_positions=512)


def _tensor_bytes(W):
    n = sum(t.numel() * t.element_size() for k, t in W.items() if k != "layers")
    for L in W["layers"]:
        n += sum(t.numel() * t.element_size() for t in L.values())
    return n


@pytest.mark.parametrize("B", [1, 3])
def test_dense_weight_bytes_are_the_tensors_read(B):
    """With nothing cached (lo = pos = 0) the bytes are: every weight tensor except the
    embedding table, B embedding rows, the B new K/V rows per layer and the fp32 logits."""
    cfg = synth.TINY
    W = synth.make_weights(cfg, 1)
    got = bench.algorithmic_bytes(cfg, B, [[0] * B for _ in range(cfg.n_layers)], [0] * B)
    embed = W["embed"].numel() * 2
    row_bytes = 2 * cfg.n_kv_heads * cfg.head_dim * 2
    want = (_tensor_bytes(W) - embed + B * cfg.d_model * 2 + cfg.n_layers * B * row_bytes
            + B * cfg.vocab * 4)
    assert got == want


def test_each_cached_key_adds_one_kv_row_per_layer():
    cfg = synth.TINY
    L = cfg.n_layers
    lo = [[0, 0] for _ in range(L)]
    a = bench.algorithmic_bytes(cfg, 2, lo, [100, 37])
    b = bench.algorithmic_bytes(cfg, 2, lo, [101, 37])
    assert b - a == L * 2 * cfg.n_kv_heads * cfg.head_dim * 2
    # a sliding window's lower bound removes the keys below it on that layer only
    lo_w = [[0, 0], [40, 0]]
    c = bench.algorithmic_bytes(cfg, 2, lo_w, [100, 37])
    assert a - c == 40 * 2 * cfg.n_kv_heads * cfg.head_dim * 2


def test_shared_prefix_override_counts_the_rows_given():
    cfg = synth.TINY
    lo = [[0, 0] for _ in range(cfg.n_layers)]
    full = bench.algorithmic_bytes(cfg, 2, lo, [100, 100])
    once = bench.algorithmic_bytes(cfg, 2, lo, [100, 100], kv_rows=cfg.n_layers * (100 + 36))
    assert full - once == cfg.n_layers * 64 * 2 * cfg.n_kv_heads * cfg.head_dim * 2


def test_moe_counts_the_routed_union_and_the_router():
    cfg = TINY_MOE
    W = synth.make_weights(cfg, 2)
    lo = [[0] for _ in range(cfg.n_layers)]
    all_e = bench.algorithmic_bytes(cfg, 1, lo, [0], moe_union=[cfg.n_experts] * cfg.n_layers)
    want = (_tensor_bytes(W) - W["embed"].numel() * 2 + cfg.d_model * 2
            + cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * 2 + cfg.vocab * 4)
    assert all_e == want  # every expert routed: every tensor is read
    one_less = bench.algorithmic_bytes(cfg, 1, lo, [0], moe_union=[cfg.n_experts - 1, cfg.n_experts])
    expert = sum(W["layers"][0][k][0].numel() * 2 for k in ("exp_gate", "exp_up", "exp_down"))
    assert all_e - one_less == expert
