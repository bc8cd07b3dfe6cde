"""The seeded input generators: determinism, shapes, rounding and padding."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_45_gb300 import workloads


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 3, 10000), rng.normal(0, 1e-30, 100), [0.0, -0.0, np.inf, -np.inf, 1e38]])
    ours = workloads.f64_to_bf16_bits(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = workloads.bf16_bits_to_f64(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("cfg,B", [(1, None), (2, None), (3, 4), (4, 7), (5, 4)])
def test_configs_shapes_and_determinism(cfg, B):
    a = workloads.make_config(cfg, B=B)
    b = workloads.make_config(cfg, B=B)
    for f in ("target", "draft", "tokens", "num_draft", "uniforms", "temperature"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert a.target.shape == (a.B, a.gmax + 1, a.V) and a.draft.shape == (a.B, a.gmax, a.V)
    assert a.uniforms.dtype == np.float32 and np.all((a.uniforms >= 0) & (a.uniforms < 1))
    for s in range(a.B):
        g = a.num_draft[s]
        assert 0 <= g <= a.gmax
        assert np.all((a.tokens[s, :g] >= 0) & (a.tokens[s, :g] < a.V))
        assert np.all(a.tokens[s, g:] == -1)
        tail_t = workloads.logits_as_f64(a.target[s, g + 1:], a.dtype)
        tail_d = workloads.logits_as_f64(a.draft[s, g:], a.dtype)
        assert np.all(np.isposinf(tail_t)) and np.all(np.isposinf(tail_d))
        assert np.all(np.isfinite(workloads.logits_as_f64(a.target[s, : g + 1], a.dtype)))


def test_seeds_differ():
    a = workloads.make_config(3, seed=1, B=2)
    b = workloads.make_config(3, seed=2, B=2)
    assert not np.array_equal(a.target, b.target)


def test_config_parameters():
    c4 = workloads.make_config(4, B=9)
    assert set(np.unique(c4.temperature)) == {0.0, np.float32(0.6), 1.0}
    assert c4.V == 151936 and c4.gmax == 7
    c5 = workloads.make_config(5, B=6)
    assert list(c5.temperature) == [0.0, 1.0] * 3
    assert c5.V == 128256 and c5.dtype == "bf16"
    assert workloads.make_config(2, greedy=True).temperature[0] == 0.0


def test_algorithmic_bytes_config5_full():
    """B=256, gamma=4, V=128256: 1280 target rows + 512 sampled draft rows of 256,512 bytes."""
    B, g, V = 256, 4, 128256
    rows = B * (g + 1) + (B // 2) * g
    assert rows * V * 2 == 459_669_504
    assert (B * (g + 1) + B * g) * V * 2 == 591_003_648


def test_greedy_drafts_are_draft_argmax_and_sampled_drafts_follow_q():
    b = workloads.make_config(5, B=4)
    d0 = workloads.logits_as_f64(b.draft[0], b.dtype)
    assert list(b.tokens[0]) == [int(np.argmax(r)) for r in d0]
    # Gumbel-max sampling: frequencies on a tiny row follow softmax(d / T)
    rng = np.random.Generator(np.random.PCG64(5))
    d = np.array([0.0, 1.0, 2.0], np.float32)
    draws = np.array([workloads._draft_token(rng, d, "f32", 0.5) for _ in range(20000)])
    w = np.exp(d / 0.5)
    w /= w.sum()
    freq = np.bincount(draws, minlength=3) / draws.size
    assert np.all(np.abs(freq - w) < 5 * np.sqrt(w * (1 - w) / draws.size))


@pytest.mark.parametrize("seed", range(12))
def test_random_batch_is_seeded_and_poisons_padding(seed):
    a, b = workloads.random_batch(seed), workloads.random_batch(seed)
    for name in ("target", "draft", "tokens", "num_draft", "uniforms"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))
    np.testing.assert_array_equal(a.temperature.view(np.int32), b.temperature.view(np.int32))  # NaN-safe
    assert a.target.shape == (a.B, a.gmax + 1, a.V) and a.draft.shape == (a.B, a.gmax, a.V)
    assert 1 <= a.B <= 48 and 0 <= a.gmax <= 9 and a.V >= 2
    t = workloads.logits_as_f64(a.target, a.dtype)
    d = workloads.logits_as_f64(a.draft, a.dtype)
    for i in range(a.B):
        g = int(a.num_draft[i])
        if g > a.gmax:  # a planted bad count: nothing else is promised for the row
            continue
        assert np.all(np.isposinf(t[i, g + 1:])) and np.all(np.isposinf(d[i, g:]))
        assert np.all(a.tokens[i, g:] == -1)
        assert np.all(np.isfinite(t[i, : g + 1])) and np.all(np.isfinite(d[i, :g]))
    assert np.all((a.uniforms >= 0) & (a.uniforms < 1))


def test_random_batches_cover_the_sweep():
    batches = [workloads.random_batch(s) for s in range(48)]
    assert {b.dtype for b in batches} == {"bf16", "f32"}
    assert any(b.gmax == 0 for b in batches) and any(b.gmax >= 8 for b in batches)
    assert any(b.V < 64 for b in batches) and any(b.V > 5000 for b in batches)
    assert any(b.V % 8 for b in batches) and any(b.V % 8 == 0 for b in batches)
    temps = np.concatenate([b.temperature for b in batches])
    assert np.any(temps == 0) and np.any(temps > 0) and (np.any(np.isnan(temps)) or np.any(temps < 0))
