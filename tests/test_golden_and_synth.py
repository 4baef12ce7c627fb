"""The stored oracle fixture, and the seeded generator against its own definition."""
import json
import os

import numpy as np

import oracle
from speculative_decoding_mla_gb300 import synth
from tests.golden import make_fixtures

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_stored_fixture():
    data = json.load(open(os.path.join(HERE, "golden", "oracle_small.json")))
    for name, entry in data["cases"].items():
        case = make_fixtures.make(entry["spec"])
        o, l = oracle.verify(case)
        np.testing.assert_allclose(l, np.array(entry["lse"]), atol=1e-9, rtol=0)
        np.testing.assert_allclose(o[:, :, data["dims"]], np.array(entry["out_dims"]), atol=1e-9, rtol=0)


def test_generator_c_matches_numpy_definition():
    for seed, tag, n, off in [(1, 2, 1000, 0), (123456789, 7, 333, 17), (2 ** 63 + 5, 1, 10, 3)]:
        assert np.array_equal(synth.words(seed, tag, n, off), synth.words_numpy(seed, tag, n, off))
    a = synth.normals(9, 1, 1001)
    b = synth.normals_numpy(9, 1, 1001)
    np.testing.assert_allclose(a, b, atol=1e-15, rtol=0)
    x = synth.bf16_normals(9, 1, 1001, 0.5)
    y = synth.f32_to_bf16_bits((b * 0.5).astype(np.float32))
    assert np.array_equal(x, y)


def test_splitmix64_reference_value():
    # splitmix64's published first output for state 0 (one increment, then the finaliser)
    z = synth._mix(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF


def test_bf16_rounding_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], dtype=np.float32)
    got = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(vals))
    assert list(got) == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0]


def test_workload_shapes():
    s = synth.workload_sizes("sweep_q4")
    assert len(s["prefixes"]) == 32 and all(2048 <= p <= 131072 for p in s["prefixes"])
    c = synth.workload("contiguous_1k")
    assert c.q.shape == (16, 64, 576) and c.kv_pool.shape == (1040, 576)
    assert np.array_equal(c.kv_indices, np.arange(1040))
    par = synth.tree_parents(4, 64, 8, 0)
    depth = np.zeros(64, int)
    for i in range(1, 64):
        assert 0 <= par[i] < i
        depth[i] = depth[par[i]] + 1
    assert depth.max() <= 8
