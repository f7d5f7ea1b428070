"""The benchmark's workloads against the configurations they stand for: launch
counts, weight bytes per step, shapes, and the MoE routing.  The byte counts
are the configurations' own: 8B-dense decode token 7,973,699,584 B in Q8_0 and
4,221,370,368 B in Q4_0 (32 layers of q, k, v, o 4096/1024 x 4096, gate, up
14336 x 4096, down 4096 x 14336, plus the 128256 x 4096 lm_head); the
Qwen3-0.6B layer set 633,233,408 B (28 layers plus the tied 151936 x 1024
lm_head); an MoE expert matrix of 768 x 2048 Q8_0 is 1,671,168 B; an int8
matrix of 1024 x 3072 is 3,145,728 B."""
import numpy as np
import pytest

import bench


def total_weight_bytes(ops):
    return sum(op.weight_bytes() for op in ops)


@pytest.mark.parametrize("workload,launches,weight_bytes", [
    ("8b-q8_0", 129, 7_973_699_584),
    ("8b-q8_0-unfused", 225, 7_973_699_584),
    ("8b-q4_0", 129, 4_221_370_368),
    ("8b-q4_0-unfused", 225, 4_221_370_368),
    ("8b-q4_k", 129, 4_221_370_368),
    ("qwen3-0.6b-q8_0", 113, 633_233_408),
    ("qwen3-0.6b-q8_0-unfused", 197, 633_233_408),
])
def test_dense_tokens_match_the_configurations(workload, launches, weight_bytes):
    model, fmt, ops = bench.workload_ops(workload, 1)
    assert len(ops) == launches
    assert total_weight_bytes(ops) == weight_bytes
    for op in ops:
        assert op.kind == "dense" and op.cols % 256 == 0          # every launch takes the TMA-staged kernel
        assert op.lora_rank == 0


def test_qlora_token_adapts_every_projection_but_the_lm_head():
    _, _, ops = bench.workload_ops("8b-q8_0-lora", 1)
    _, _, plain = bench.workload_ops("8b-q8_0", 1)
    assert len(ops) == 129
    for op, p in zip(ops, plain):
        assert (op.rows, op.cols) == (p.rows, p.cols)
        assert op.lora_rank == (0 if op.name == "lm_head" else 16)
        assert op.weight_bytes() == p.weight_bytes() + 2 * op.lora_rank * (op.rows + op.cols)


@pytest.mark.parametrize("n_vec", [1, 4])
def test_moe_layers_route_eight_distinct_experts_per_token(n_vec):
    _, fmt, ops = bench.workload_ops("moe-q8_0", n_vec)
    assert fmt == "q8_0" and len(ops) == 2 * bench.MOE_LAYERS
    expert_bytes = 768 * (2048 // 32) * 34
    assert expert_bytes == 1_671_168
    for gate_up, down in zip(ops[0::2], ops[1::2]):
        assert (gate_up.rows, gate_up.cols, gate_up.x_per_slot) == (1536, 2048, 0)    # gate and up fused
        assert (down.rows, down.cols, down.x_per_slot) == (2048, 768, 1)
        ids = gate_up.ids
        assert ids.shape == (n_vec, 8) and np.array_equal(ids, down.ids)
        assert ids.min() >= 0 and ids.max() < 128
        for t in range(n_vec):
            assert len(set(ids[t].tolist())) == 8                    # drawn without replacement
        distinct = len(np.unique(ids))
        assert gate_up.weight_bytes() == distinct * 2 * expert_bytes
        assert down.weight_bytes() == distinct * expert_bytes


def test_int8_step_is_96_copies_of_both_matrices():
    _, fmt, ops = bench.workload_ops("int8-requant", 1)
    assert fmt == "i8" and len(ops) == 192
    shapes = sorted({(op.rows, op.cols) for op in ops})
    assert shapes == [(1024, 3072), (3072, 1024)]
    assert all(op.rows * op.cols == 3_145_728 for op in ops)
    assert total_weight_bytes(ops) == 192 * 3_145_728 + sum(8 * op.rows for op in ops)
