"""Pins for the sampling oracle (oracle/sampling.py): the generator, the sampler's law, and lossless
tree decoding with sampling acceptance."""
import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chisquare

from oracle import config, sampling as smp, tiny_lm


@pytest.mark.parametrize("ctr,key,want", [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
])
def test_philox_known_answers(ctr, key, want):
    """Known-answer vectors published with the Random123 generators (Philox-4x32, 10 rounds)."""
    out = smp.philox4x32_10(np.array(ctr, np.uint32)[None], np.array(key, np.uint32)[None])[0]
    assert tuple(int(x) for x in out) == want


def test_uniforms_are_open_interval_and_exact_in_float32():
    x = np.array([0, 255, 256, 0xFFFFFFFF], np.uint32)
    u = smp.uniforms(x)
    assert np.all((u > 0) & (u < 1))
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)


def test_sampler_follows_softmax_at_temperature():
    """Gumbel-max over keyed noise draws from softmax(logits / T): chi-square over 4000 draws."""
    logits = np.array([2.0, 1.0, 0.5, 0.0, -1.0, 3.0])
    T = 1.7
    counts = np.zeros(6)
    for pos in range(4000):
        counts[smp.sample_row(logits, T, 12345, 3, pos)[0]] += 1
    p = softmax(logits / T)
    assert chisquare(counts, 4000 * p).pvalue > 1e-3


def test_distinct_keys_give_distinct_streams():
    a = smp.draws(1, 0, 10, 64)
    assert not np.array_equal(a, smp.draws(2, 0, 10, 64))
    assert not np.array_equal(a, smp.draws(1, 1, 10, 64))
    assert not np.array_equal(a, smp.draws(1, 0, 11, 64))


@pytest.fixture(scope="module")
def lm():
    return tiny_lm.TinyLM(seed=0)


@pytest.mark.parametrize("T,seed", [(0.7, 1), (1.0, 2)])
def test_hybrid_sampling_equals_autoregressive_sampling(lm, T, seed):
    """Losslessness under sampling: with the same position-keyed noise, tree decoding with sampling
    acceptance emits exactly the tokens autoregressive sampling does."""
    rng = np.random.default_rng(seed)
    seg = rng.integers(0, lm.V, 5).tolist()
    prompt = rng.integers(0, lm.V, 6).tolist() + seg + seg
    cfg = config.make_config(Kmax=16, D=4, k=3, V=lm.V, W=4, tau=0.3)
    ar, _, _, gaps = tiny_lm.sample_ar(lm, prompt, 30, 200, T, seed)
    assert min(gaps) > 1e-6
    hy, _, _, steps, _ = tiny_lm.sample_hybrid(lm, prompt, 30, 200, cfg, T, seed, sharpen=4.0)
    assert hy == ar
    assert max(s["acc_len"] for s in steps) > 1
