"""The seeded input generator: integer stream, uniforms and normals."""
import math

import torch

import synth


def test_splitmix_stream_matches_python_integers():
    seed, stream = 0, 1
    key = synth.stream_key(seed, stream)
    got = synth.raw_u64(seed, stream, 5, 8)
    for i, x in enumerate(got.tolist()):
        n = 5 + i + 1
        expect = synth._mix_int(key + n * synth.GAMMA)
        assert x % (1 << 64) == expect


def test_known_splitmix64_vector():
    # Published SplitMix64 sequence for state 0: first output 0xE220A8397B1DCDAF.
    assert synth._mix_int(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_normals_are_standard_and_reproducible():
    a = synth.normal((4, 1000), 0, 0)
    b = synth.normal((4, 1000), 0, 0)
    assert torch.equal(a, b)
    assert abs(a.mean().item()) < 0.05
    assert abs(a.std().item() - 1.0) < 0.05
    c = synth.normal((4, 1000), 0, 1)
    assert not torch.equal(a, c)


def test_elements_are_independent_of_shape():
    a = synth.normal((10,), 3, 2).view(-1)
    b = synth.normal((2, 7), 3, 2).view(-1)
    assert torch.equal(a[:10], b[:10])


def test_bf16_is_rounded_from_f32():
    f = synth.normal((257,), 0, 2, dtype=torch.float32)
    h = synth.normal((257,), 0, 2, dtype=torch.bfloat16)
    assert torch.equal(f.to(torch.bfloat16), h)


def test_empty_rows_fraction_and_distinct():
    rows = synth.empty_rows(2, 4096, 0.01, seed=0)
    assert len(rows) == round(0.01 * 2 * 4096) == 82
    assert len(set(rows)) == 82
    rb = synth.row_kv_bounds_with_empty_rows(2, 4096, 4096, 0.01, seed=0)
    empty = (rb[..., 0] > rb[..., 1]).sum().item()
    assert empty == 82


def test_alibi_slopes_geometric():
    s = synth.alibi_slopes(16)
    for h in range(16):
        assert s[h].item() == float(torch.tensor(2.0 ** (-8 * (h + 1) / 16), dtype=torch.float32))
    assert math.isclose(s[1].item() / s[0].item(), 2 ** -0.5, rel_tol=1e-6)
