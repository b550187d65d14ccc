"""CPU pins of the seeded input generators that feed both the oracle and the
CUDA path.  A mistake here would not show up as a parity failure, since both
sides would receive the same wrong inputs.  So the generators are checked
directly against the recipe they claim: bf16 by round-to-nearest-even (as
torch casts), exact widening back to float32, determinism per (seed,
stream), the kept-unit ids of the MAE mask, and the weight scale."""
import math

import numpy as np
import pytest

import synthetic as S


def test_bf16_rounding_hand_ties():
    u = 2.0 ** -7  # bf16 ulp on [1, 2)
    cases = [
        (1.0, 1.0),
        (1.0 + u / 2, 1.0),               # tie: 1.0 has the even last bit
        (1.0 + 3 * u / 2, 1.0 + 2 * u),   # tie between odd 1+u and even 1+2u
        (1.0 + u / 2 + 2.0 ** -20, 1.0 + u),
        (1.0 + u / 2 - 2.0 ** -20, 1.0),
        (-(1.0 + 3 * u / 2), -(1.0 + 2 * u)),
        (255.5, 256.0),
        (254.5, 254.0),
        (0.0, 0.0),
    ]
    x = np.array([c[0] for c in cases], np.float32)
    got = S.bf16_bits_to_f32(S.f32_to_bf16_bits(x))
    np.testing.assert_array_equal(got, np.array([c[1] for c in cases], np.float32))


def test_bf16_rounding_matches_torch_cast():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(11)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-30, 30, 20000),
                        1.0 + np.arange(1024) * 2.0 ** -10]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(S.f32_to_bf16_bits(x), ref)


def test_bf16_widening_is_exact_and_round_trips():
    bits = np.arange(0, 0x7F80, 7, dtype=np.uint16)       # finite positives
    bits = np.concatenate([bits, bits | np.uint16(0x8000)])
    f = S.bf16_bits_to_f32(bits)
    assert np.all(np.isfinite(f))
    np.testing.assert_array_equal(S.f32_to_bf16_bits(f), bits)


def test_normal_is_deterministic_per_seed_and_stream():
    a = S.normal((3, 5, 7), 4, 2)
    np.testing.assert_array_equal(a, S.normal((3, 5, 7), 4, 2))
    assert not np.array_equal(a, S.normal((3, 5, 7), 4, 3))
    assert not np.array_equal(a, S.normal((3, 5, 7), 5, 2))
    assert a.dtype == np.uint16
    f = S.normal((3, 5, 7), 4, 2, dtype="f32")
    assert f.dtype == np.float32
    # the bf16 draw is the f32 draw rounded
    np.testing.assert_array_equal(a, S.f32_to_bf16_bits(f))
    with pytest.raises(ValueError):
        S.normal((2,), 0, 0, dtype="f16")


def test_normal_moments():
    x = S.bf16_bits_to_f32(S.normal((200000,), 0, 0)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    H = 20
    w32 = S.premix_weight(H, 4, 0, 1)
    assert w32.shape == (H, 4, H) and w32.dtype == np.float32
    w = w32.astype(np.float64)
    assert abs(w.std() - 1.0 / math.sqrt(H)) < 0.03 / math.sqrt(H) * 3


def test_keep_units_are_sorted_unique_and_in_range():
    keep = S.keep_units(64, 49, 20, 3)
    assert keep.shape == (64, 20) and keep.dtype == np.int32
    assert np.all(np.diff(keep, axis=1) > 0)
    assert keep.min() >= 0 and keep.max() < 49
    np.testing.assert_array_equal(keep, S.keep_units(64, 49, 20, 3))
    # different samples draw different masks
    assert len({tuple(r) for r in keep}) > 1


def test_workload_shapes_are_the_pages():
    assert (S.LLAMA_PREMIX.B, S.LLAMA_PREMIX.N, S.LLAMA_PREMIX.H, S.LLAMA_PREMIX.P,
            S.LLAMA_PREMIX.d) == (1, 8192, 20, 4, 128)
    assert S.LLAMA_WINDOW.HP == 80 and S.LLAMA_WINDOW.N == 4096 and S.WINDOW_KEYS == 1024
    assert (S.LONG_CTX.B, S.LONG_CTX.N, S.LONG_CTX.HP) == (2, 16384, 80)
    mu = S.HIERA_MU
    assert (mu.B, mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w, mu.n_keep, mu.C) == \
        (128, 56, 56, 8, 8, 20, 96)
    assert mu.n_units == 49 and mu.unit_tokens == 64
    assert (S.TINY.B, S.TINY.N, S.TINY.H, S.TINY.P, S.TINY.d) == (1, 128, 4, 2, 32)
