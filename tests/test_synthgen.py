"""The seeded input generator: determinism, per-expert random access and the
value recipe (uniform 4-bit codes, E4M3 scales in [2^-8, 2^-4], bf16 normals)."""
import numpy as np

import synthgen


def test_deterministic_and_seed_sensitive():
    a = synthgen.normal_bf16(1, 2, synthgen.T_X, 0, 4096)
    b = synthgen.normal_bf16(1, 2, synthgen.T_X, 0, 4096)
    c = synthgen.normal_bf16(2, 2, synthgen.T_X, 0, 4096)
    d = synthgen.normal_bf16(1, 3, synthgen.T_X, 0, 4096)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_per_expert_generation_equals_bulk():
    w = synthgen.WORKLOADS["tiny"]
    full = synthgen.make_layer(w, 0)
    part = synthgen.make_layer(w, 0, experts=[3, 11])
    for name in ("gate", "up", "down"):
        f, p = getattr(full, name), getattr(part, name)
        for e in (3, 11):
            assert np.array_equal(f.codes[e], p.codes[e])
            assert np.array_equal(f.scales[e], p.scales[e])
        assert not p.codes[0].any()


def test_offsets_slice_the_same_stream():
    a = synthgen.codes(4, 0, synthgen.T_GATE_C, 0, 1024)
    b = synthgen.codes(4, 0, synthgen.T_GATE_C, 512, 512)
    assert np.array_equal(a[512:], b)
    s = synthgen.scales(4, 0, synthgen.T_GATE_S, 0, 300)
    t = synthgen.scales(4, 0, synthgen.T_GATE_S, 100, 200)
    assert np.array_equal(s[100:], t)


def test_value_recipe():
    c = synthgen.codes(0, 0, synthgen.T_UP_C, 0, 1 << 20)
    nib = np.concatenate([c & 15, c >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * counts.mean() and counts.max() < 1.1 * counts.mean()
    x = synthgen.bf16_to_f32(synthgen.normal_bf16(0, 0, synthgen.T_X, 0, 1 << 18)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    r = synthgen.bf16_to_f32(synthgen.normal_bf16(0, 0, synthgen.T_ROUTER_W, 0, 1 << 18, 0.0, 0.02))
    assert abs(r.std() - 0.02) < 0.001
    b = synthgen.zipf_log_prior(1.1, 256)
    assert b[0] == 0.0 and np.all(np.diff(b) < 0) and abs(b[255] + 1.1 * np.log(256)) < 1e-5
