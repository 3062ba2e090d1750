"""Token sampling on the device (repetition penalty, temperature, top-k, top-p,
inverse-CDF draw) against the oracle's sample_detail, through llama_sample.

The draw is an integer decided by floating point: the kernel sums in fp32, the
oracle in fp64. A row passes when the ids agree; where they differ, the GPU's
id must still be valid for the oracle: kept by it (or the next id in its order
when the top-k / top-p cut-off is within rounding), with the uniform inside
that id's cumulative-probability interval widened by U_TOL. At most a few rows
of a batch may fall in that band."""
import numpy as np
import pytest
import torch

from _common import f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu

U_TOL = 2e-4
L7 = synth.LLAMA2_7B.with_(n_layers=1)


def _ctx(shape, max_batch=256):
    need_gpu()
    w = {"layers": [synth.layer_weights(shape, 7, 0)]}
    return binding.Model(shape, to_dev(w), max_batch=max_batch, max_tokens=0, max_seq=64,
                         has_embed_head=False)


@pytest.fixture(scope="module")
def ctx7():
    return _ctx(L7)


def _logits(B, V, seed, std=1.3):
    g = torch.Generator()
    g.manual_seed(seed)
    z = torch.randn(B, V, generator=g) * std
    z[::5] *= 4.0  # some peaked rows
    return z


def _history(B, V, seed, max_len=300):
    g = torch.Generator()
    g.manual_seed(seed + 1)
    lens = torch.randint(0, max_len + 1, (B,), generator=g, dtype=torch.int32)
    hist = torch.randint(0, V, (B, max_len), generator=g, dtype=torch.int32)
    return hist, lens


def _uniforms(B, seed):
    g = torch.Generator()
    g.manual_seed(seed + 2)
    return torch.rand(B, generator=g)


def _run(m, z, u, params, hist=None, lens=None):
    ids = torch.full((z.shape[0],), -1, dtype=torch.int32, device="cuda")
    m.sample(z.cuda(), u.cuda(), ids, history=None if hist is None else hist.cuda(),
             history_len=None if lens is None else lens.cuda(), **params)
    m.sync()
    return ids.cpu().numpy()


def _rank_of(s, v):
    """0-based position of id v in the order s descending, lower id first."""
    return int(np.sum(s > s[v]) + np.sum((s == s[v]) & (np.arange(len(s)) < v)))


def _check(z, u, params, got, hist=None, lens=None, max_band=3):
    T, k = params.get("temperature", 1.0), params.get("top_k", 0)
    p, r = params.get("top_p", 1.0), params.get("repetition_penalty", 1.0)
    zf, band = f64(z), 0
    for b in range(len(got)):
        h = None if hist is None else hist[b, : int(lens[b])].numpy()
        d = O.sample_detail(zf[b], h, T, k, p, r, float(u[b]))
        g = int(got[b])
        if g == d["token"]:
            continue
        band += 1
        kept = list(d["kept"])
        if g in kept:
            i = kept.index(g)
            assert d["cdf_lo"][i] - U_TOL <= u[b] < d["cdf_hi"][i] + U_TOL, \
                (b, g, d["token"], float(u[b]), d["cdf_lo"][i], d["cdf_hi"][i])
        else:  # the cut-off itself must be marginal: g is the next id in the order
            s = d["z"] / T
            rank, n = _rank_of(s, g), len(kept)
            assert rank == n, (b, g, rank, n)
            if 0 < k < len(s) and n == k:
                kth = s[np.lexsort((np.arange(len(s)), -s))[k - 1]]
                assert abs(s[g] - kth) <= 1e-6 * max(1.0, abs(kth)), (b, s[g], kth)
            else:
                assert abs(d["cum_sorted"][n - 1] - p) < 1e-4 or abs(d["cum_sorted"][n - 2] - p) < 1e-4
            assert u[b] > 1.0 - 1e-3 or abs(u[b] - d["cdf_hi"][-1]) < 1e-3
    assert band <= max_band, "%d rows disagree" % band


CASES = [
    dict(temperature=1.0),
    dict(temperature=0.7, top_k=50, top_p=0.9, repetition_penalty=1.1),
    dict(temperature=0.7, top_p=0.9),
    dict(temperature=1.3, top_k=20),
    dict(temperature=0.5, top_p=0.5, repetition_penalty=1.3),
    dict(temperature=0.9, top_k=1000, top_p=0.95),
]


@pytest.mark.parametrize("params", CASES)
def test_sampling_matches_oracle(ctx7, params):
    B, V = 64, L7.vocab
    z = _logits(B, V, 301)
    u = _uniforms(B, 301)
    hist, lens = _history(B, V, 301) if params.get("repetition_penalty", 1.0) != 1.0 else (None, None)
    got = _run(ctx7, z, u, params, hist, lens)
    assert np.all((got >= 0) & (got < V))
    _check(z, u, params, got, hist, lens)


def test_temperature_zero_is_the_penalised_argmax(ctx7):
    B, V = 32, L7.vocab
    z = _logits(B, V, 302)
    hist, lens = _history(B, V, 302, max_len=2000)
    u = _uniforms(B, 302)
    got = _run(ctx7, z, u, dict(temperature=0.0, repetition_penalty=1.5), hist, lens)
    zf = f64(z)
    want = [O.sample_detail(zf[b], hist[b, : int(lens[b])].numpy(), 0.0, 0, 1.0, 1.5, 0.5)["token"]
            for b in range(B)]
    np.testing.assert_array_equal(got, want)
    plain = _run(ctx7, z, u, dict(temperature=0.0))
    np.testing.assert_array_equal(plain, O.greedy(zf))


def test_top_k_one_and_tiny_top_p_give_the_argmax(ctx7):
    B, V = 48, L7.vocab
    z = _logits(B, V, 303)
    u = torch.linspace(0.0, 0.99999, B)
    want = O.greedy(f64(z))
    np.testing.assert_array_equal(_run(ctx7, z, u, dict(temperature=0.8, top_k=1)), want)
    np.testing.assert_array_equal(_run(ctx7, z, u, dict(temperature=1.0, top_p=1e-6)), want)


def test_draws_are_reproducible_and_follow_the_distribution(ctx7):
    # one row repeated with a grid of uniforms: the ids walk the CDF in id order
    B, V = 256, L7.vocab
    row = _logits(1, V, 304, std=3.0)
    z = row.repeat(B, 1)
    u = (torch.arange(B, dtype=torch.float32) + 0.5) / B
    params = dict(temperature=0.8, top_p=0.9)
    a = _run(ctx7, z, u, params)
    b = _run(ctx7, z, u, params)
    np.testing.assert_array_equal(a, b)
    assert np.all(np.diff(a) >= 0)  # a growing uniform never moves back in id order
    _check(z, u, params, a, max_band=4)


def test_small_vocabulary_and_history_outside_the_vocabulary():
    shape = synth.TINY.with_(n_layers=1)
    m = _ctx(shape, max_batch=16)
    B, V = 12, shape.vocab
    z = _logits(B, V, 305)
    u = _uniforms(B, 305)
    hist, lens = _history(B, V, 305, max_len=40)
    params = dict(temperature=0.9, top_k=30, top_p=0.8, repetition_penalty=1.2)
    got = _run(m, z, u, params, hist, lens)
    _check(z, u, params, got, hist, lens, max_band=1)
    hist[0, 0] = V + 5  # outside the vocabulary: skipped and flagged
    lens[0] = max(int(lens[0]), 1)
    again = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    m.sample(z.cuda(), u.cuda(), again, history=hist.cuda(), history_len=lens.cuda(), **params)
    rc, flags = m.sync_status()
    assert rc == 5 and flags & binding.FLAG_TOKEN_RANGE
    _check(z, u, params, again.cpu().numpy(), hist, lens, max_band=1)


def test_invalid_parameters_are_rejected(ctx7):
    z = torch.zeros(2, L7.vocab, device="cuda")
    u = torch.zeros(2, device="cuda")
    ids = torch.zeros(2, dtype=torch.int32, device="cuda")
    for bad in (dict(temperature=-1.0), dict(top_p=0.0), dict(top_p=1.5),
                dict(repetition_penalty=0.0), dict(temperature=float("nan"))):
        with pytest.raises(RuntimeError, match="INVALID_ARG"):
            ctx7.sample(z, u, ids, **bad)


def test_ties_at_the_thresholds_follow_the_index_order(ctx7):
    # rows with long runs of equal logits: every entry tied (the radix search
    # never shrinks the candidates), and a plateau straddling the top-k cut
    B, V = 8, L7.vocab
    z = torch.zeros(B, V)
    z[1] = 0.25
    z[2, ::3] = 1.0
    z[3, 1000:1100] = 2.0
    z[3, 5000:5040] = 3.0
    z[4:] = torch.round(_logits(4, V, 306) * 2.0) / 2.0  # few distinct values
    u = _uniforms(B, 306)
    for params in (dict(temperature=1.0, top_k=50), dict(temperature=0.8, top_k=70, top_p=0.5),
                   dict(temperature=1.0, top_p=0.3), dict(temperature=1.0, top_k=5000)):
        got = _run(ctx7, z, u, params)
        _check(z, u, params, got, max_band=1)
