"""The seeded generators are deterministic and have the workloads' structure."""
import numpy as np

import synth


def test_deterministic_and_block_addressable():
    spec = synth.WORKLOADS["multi_lane"]
    k1, v1 = synth.context_chunk(spec, 3, 100, 200)
    k2, v2 = synth.context_chunk(spec, 3, 0, 400)
    assert np.array_equal(k1, k2[100:300]) and np.array_equal(v1, v2[100:300])
    assert k1.shape == (200, 4, 128) and k1.dtype == np.uint16


def test_context_lengths_in_range():
    for name in ("multi_lane", "int4_12slot"):
        spec = synth.WORKLOADS[name]
        L = synth.context_lengths(spec)
        assert len(L) == spec.num_lanes and L.min() >= spec.ctx_lo and L.max() <= spec.ctx_hi
        assert np.array_equal(L, synth.context_lengths(spec))


def test_permuted_page_table_is_a_permutation():
    spec = synth.WORKLOADS["multi_lane"]
    L = synth.context_lengths(spec)
    table, total = synth.page_table_for(spec, L, spec.window)
    used = np.concatenate([table[b, :(L[b] + spec.window + 63) // 64] for b in range(len(L))])
    assert np.array_equal(np.sort(used), np.arange(total))
    assert not np.array_equal(used, np.arange(total))


def test_outlier_channels():
    spec = synth.WORKLOADS["plain_decode"]
    m = synth.outlier_channels(spec)
    assert ((m == 8.0).sum(1) == 4).all()
    k, _ = synth.context_chunk(spec, 0, 0, 4096)
    x = synth.bf16_to_f32(k)
    big = np.abs(x[:, 0, m[0] == 8.0]).mean()
    small = np.abs(x[:, 0, m[0] == 1.0]).mean()
    assert 6 < big / small < 10


def test_acceptance_inputs_plant_the_target():
    spec = synth.WORKLOADS["tiny"]
    logits, drafts, targets = synth.acceptance_inputs(spec, 5, 4, 4096, 0.7)
    assert (logits.argmax(-1) == targets).all()
    assert drafts.shape == (5, 3) and drafts.min() >= 0 and drafts.max() < 4096


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38], np.float32)
    bits = synth.to_bf16_bits(x)
    back = synth.bf16_to_f32(bits)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.015625 and back[3] == -2.5
