"""The seeded input generator: determinism, bf16 rounding, packed layout. No GPU."""
import numpy as np

from speculative_decoding_token_temp_gb300 import synth


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -2.5, 3.0e38],
                 dtype=np.float32)
    got = synth.bf16_bits_as_f32(synth.round_to_bf16_bits(x))
    # 1+2^-8 is halfway between 1 and 1+2^-7: ties go to the even mantissa (1.0);
    # 1+3*2^-8 is halfway between 1+2^-7 and 1+2^-6: even is 1+2^-6
    assert list(got[:5]) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.5]
    assert abs(got[5] - 3.0e38) / 3.0e38 < 2 ** -8


def test_deterministic_and_per_sequence_streams():
    a = synth.make_stochastic(3, 300, synth.BF16, 0.6, seed=9, gamma=4)
    b = synth.make_stochastic(3, 300, synth.BF16, 0.6, seed=9, gamma=4)
    for k in ("target", "draft", "tokens", "u_accept", "u_sample"):
        assert np.array_equal(getattr(a, k), getattr(b, k))
    c = synth.make_stochastic(5, 300, synth.BF16, 0.6, seed=9, gamma=4)
    assert np.array_equal(a.target, c.target[:15]) and np.array_equal(a.tokens, c.tokens[:12])


def test_ragged_layout():
    w = synth.make_stochastic(7, 64, synth.BF16, 0.8, seed=4, gamma_range=(1, 16), agreement=0.7)
    assert w.cu_draft[0] == 0 and np.all(np.diff(w.cu_draft) == w.gammas)
    assert np.all((w.gammas >= 1) & (w.gammas <= 16))
    assert w.target.shape == (w.total_draft + 7, 64) and w.draft.shape == (w.total_draft, 64)
    assert np.all((w.tokens >= 0) & (w.tokens < 64))
    assert np.all((w.u_accept >= 0) & (w.u_accept < 1)) and np.all((w.u_sample >= 0) & (w.u_sample < 1))


def test_generator_shape_statistics():
    """Target rows: sd 3 noise plus +8 on one token; draft: 0.9*target-noise + N(0,1)."""
    w = synth.make_stochastic(1, 200000, synth.F32, 1.0, seed=1, gamma=2)
    t = w.target.astype(np.float64)
    d = w.draft.astype(np.float64)
    assert abs(np.std(t[0]) - 3.0) < 0.05
    resid = d[0] - 0.9 * t[0]
    resid = resid[np.abs(resid) < 6]
    assert abs(np.std(resid) - 1.0) < 0.05


def test_tree_inputs():
    w = synth.make_tree(4, 500, synth.BF16, seed=3)
    assert w.target.shape == (4 * 13, 500) and w.node_tokens.shape == (4, 12)
    assert list(w.parent) == list(synth.TREE_PARENT)
    # the three root candidates are distinct
    for b in range(4):
        assert len(set(w.node_tokens[b, :3].tolist())) == 3
