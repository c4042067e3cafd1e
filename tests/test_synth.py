"""The seeded input generator: determinism, exact bf16 rounding, uniform grid."""
import numpy as np
import torch

from eagle_speculative_decoding_tree_gb300 import synth


def test_same_seed_same_bytes():
    w = synth.WORKLOADS["tiny"]
    sl = synth.prefix_lengths(w)
    a = synth.attn_tensors(w, 1, 1, sl, w.rows)
    b = synth.attn_tensors(w, 1, 1, sl, w.rows)
    for x, y in zip(a, b):
        assert x.tobytes() == y.tobytes()
    c = synth.attn_tensors(w, 0, 1, sl, w.rows)
    assert a[0].tobytes() != c[0].tobytes()


def test_bf16_rounding_matches_torch():
    g = synth.rng(0, 99)
    x = (g.standard_normal(100000) * 10.0 ** g.integers(-6, 6, 100000)).astype(np.float32)
    # exact halfway cases (ties to even)
    halves = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, halves, -halves])
    ours = synth.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_value(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_uniforms_on_grid():
    u = synth.uniforms(synth.rng(0, 5), (100000,))
    assert u.dtype == np.float32
    assert u.min() >= 0.0 and u.max() < 1.0
    scaled = u.astype(np.float64) * 2 ** 24
    assert np.array_equal(scaled, np.floor(scaled))


def test_static_shapes():
    par = synth.static_parents(synth.TINY_STATIC_CHOICES)
    assert par.tolist() == [-1, 0, 0, 0, 0, 1, 1, 2, 3, 5, 5]
    chain = synth.static_parents(synth.CHAIN7)
    assert chain.tolist() == [-1, 0, 1, 2, 3, 4, 5, 6]


def test_ragged_prefix_lengths():
    w = synth.WORKLOADS["concurrency"].with_(batch=32)
    sl = synth.prefix_lengths(w)
    assert sl.shape == (32,) and sl.min() >= 1024 and sl.max() <= 16384
    assert len(set(sl.tolist())) > 20
    assert np.array_equal(sl, synth.prefix_lengths(w))


def test_hash_lm_rows_are_path_functions():
    lm = synth.HashLM(100, "normal", 3.0, 0.5, "bf16")
    h = synth.child_hash(synth.root_hash(2, 0), 7)
    assert np.array_equal(lm.target_row(h), lm.target_row(h))
    assert not np.array_equal(lm.target_row(h), lm.target_row(synth.child_hash(h, 7)))
    # values are exactly bf16
    r = lm.draft_row(h)
    assert np.array_equal(synth.bf16_value(synth.bf16_bits(r)), r)


def test_zipf_row_is_exact_power_law():
    x = synth.zipf_row(synth.rng(0, 3), 1000).astype(np.float64)
    p = np.exp(x - x.max())
    p /= p.sum()
    ranks = np.argsort(-p)
    # p is proportional to rank^-1.1 (up to float32 rounding of the logits)
    expect = np.arange(1, 1001, dtype=np.float64) ** -1.1
    expect /= expect.sum()
    np.testing.assert_allclose(p[ranks], expect, rtol=1e-5)
