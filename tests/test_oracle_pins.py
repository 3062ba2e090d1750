"""Pins of the CPU oracle to facts other than itself: closed forms, invariants
the pages state, library routines on special cases, brute force on tiny
inputs and the numbers the pages print. CPU only."""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import llama_oracle as O
from llama2_decoder_forward_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(7)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_uniform_gamma_closed_form():
    # gamma == c everywhere: RMS(y) = c * sqrt(ms / (ms + eps)).
    x = rng.standard_normal((5, 64)) * 3.0
    c, eps = 1.7, 1e-5
    y = O.rmsnorm(x, np.full(64, c), eps)
    ms = np.mean(x * x, axis=-1)
    rms_y = np.sqrt(np.mean(y * y, axis=-1))
    np.testing.assert_allclose(rms_y, c * np.sqrt(ms / (ms + eps)), rtol=1e-13)


def test_rmsnorm_eps_inside_root_and_scale_invariance():
    x = np.array([[3.0, 4.0]])            # mean(x^2) = 12.5
    y = O.rmsnorm(x, np.ones(2), 0.5)
    np.testing.assert_allclose(y, x / math.sqrt(13.0), rtol=1e-15)
    # Scaling x by a leaves y unchanged up to eps: y(a z) / y(z) = sqrt((ms + eps) / (ms + eps / a^2)).
    z = rng.standard_normal((3, 32))
    ms = np.mean(z * z, axis=-1, keepdims=True)
    ratio = O.rmsnorm(1e3 * z, np.ones(32), 1e-5) / O.rmsnorm(z, np.ones(32), 1e-5)
    np.testing.assert_allclose(ratio, np.broadcast_to(np.sqrt((ms + 1e-5) / (ms + 1e-11)), ratio.shape),
                               rtol=1e-13)


def test_rmsnorm_matches_library_and_is_per_token():
    x = rng.standard_normal((4, 48))
    g = 1 + 0.1 * rng.standard_normal(48)
    ref = F.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(g), eps=1e-5).numpy()
    np.testing.assert_allclose(O.rmsnorm(x, g, 1e-5), ref, rtol=1e-13, atol=1e-14)
    x2 = x.copy()
    x2[1:] *= 5.0  # other tokens must not change token 0's output
    np.testing.assert_array_equal(O.rmsnorm(x2, g, 1e-5)[0], O.rmsnorm(x, g, 1e-5)[0])


# ---------------------------------------------------------------- RoPE

def test_rope_hand_angles():
    # d = 4, base 10000: theta_0 = 1, theta_1 = 10000^(-1/2) = 0.01.
    np.testing.assert_allclose(O.rope_frequencies(4, 10000.0), [1.0, 0.01], rtol=1e-15)
    e0 = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    y = O.rope(e0, [1], 10000.0)[0, 0]
    np.testing.assert_allclose(y, [math.cos(1.0), math.sin(1.0), 0, 0], atol=1e-15)
    e2 = np.array([[[0.0, 0.0, 1.0, 0.0]]])
    y = O.rope(e2, [100], 10000.0)[0, 0]          # pair 1 turns by 100 * 0.01 = 1 rad
    np.testing.assert_allclose(y, [0, 0, math.cos(1.0), math.sin(1.0)], atol=1e-14)
    e1 = np.array([[[0.0, 1.0, 0.0, 0.0]]])       # (a, b) = (0, 1) -> (-sin, cos)
    y = O.rope(e1, [2], 10000.0)[0, 0]
    np.testing.assert_allclose(y[:2], [-math.sin(2.0), math.cos(2.0)], atol=1e-15)


def test_rope_position_zero_is_identity_and_norm_preserved():
    x = rng.standard_normal((6, 3, 64))
    np.testing.assert_array_equal(O.rope(x, np.zeros(6), 10000.0), x)
    y = O.rope(x, np.arange(6) * 517, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_relative_position_invariant():
    # <R_m q, R_n k> depends only on m - n (§1.4).
    d = 128
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    for delta in (0, 1, 7, 300):
        vals = []
        for n in (0, 5, 1000, 4000):
            a = O.rope(q, [n + delta], 10000.0)[0, 0]
            b = O.rope(k, [n], 10000.0)[0, 0]
            vals.append(a @ b)
        ref = O.rope(q, [delta], 10000.0)[0, 0] @ k[0, 0]
        np.testing.assert_allclose(vals, ref, rtol=1e-9, atol=1e-9)


def test_rope_matches_complex_form():
    # f(q, m) = q * e^{i m theta}: pairs as complex numbers, via torch.polar.
    d, T = 64, 9
    x = torch.from_numpy(rng.standard_normal((T, 2, d)))
    pos = torch.arange(T, dtype=torch.float64) * 37
    freqs = 10000.0 ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones(T, d // 2, dtype=torch.float64), pos[:, None] * freqs[None])
    xc = torch.view_as_complex(x.reshape(T, 2, d // 2, 2).contiguous())
    ref = torch.view_as_real(xc * rot[:, None, :]).reshape(T, 2, d).numpy()
    np.testing.assert_allclose(O.rope(x.numpy(), pos.numpy(), 10000.0), ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- softmax / attention

def test_softmax_rows_sum_to_one_and_shift_invariant():
    s = rng.standard_normal((7, 33)) * 10
    p = O.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.softmax(s + 123.0), p, rtol=1e-12)
    np.testing.assert_allclose(p, scipy.special.softmax(s, axis=-1), rtol=1e-13)
    big = O.softmax(np.array([[1000.0, 1000.0, 999.0]]))   # no overflow
    e = math.exp(-1)
    np.testing.assert_allclose(big[0], [1 / (2 + e), 1 / (2 + e), e / (2 + e)], rtol=1e-14)


def _brute_attend(q, K, V):
    d = len(q)
    s = [sum(q[i] * K[n][i] for i in range(d)) / math.sqrt(d) for n in range(len(K))]
    mx = max(s)
    w = [math.exp(x - mx) for x in s]
    tot = sum(w)
    return [sum(w[n] * V[n][i] for n in range(len(K))) / tot for i in range(len(V[0]))]


def test_attention_brute_force_tiny():
    q = rng.standard_normal(4)
    K = rng.standard_normal((5, 4))
    V = rng.standard_normal((5, 4))
    np.testing.assert_allclose(O.attend(q, K, V), _brute_attend(q, K, V), rtol=1e-13)


def test_attention_special_cases():
    K = rng.standard_normal((6, 8))
    V = rng.standard_normal((6, 8))
    np.testing.assert_allclose(O.attend(np.zeros(8), K, V), V.mean(0), rtol=1e-13)
    np.testing.assert_allclose(O.attend(rng.standard_normal(8), K[:1], V[:1]), V[0], rtol=1e-15)


def test_gqa_group_one_is_mha_and_repeat_equivalence():
    n_q, n_kv, S, d = 8, 2, 11, 16
    q = rng.standard_normal((n_q, d))
    K = rng.standard_normal((n_kv, S, d))
    V = rng.standard_normal((n_kv, S, d))
    g = O.gqa_attention(q, K, V, 9)
    Kr, Vr = np.repeat(K, n_q // n_kv, 0), np.repeat(V, n_q // n_kv, 0)
    mha = O.gqa_attention(q, Kr, Vr, 9)          # G = 1
    np.testing.assert_allclose(g, mha, rtol=1e-14)
    per_head = np.stack([O.attend(q[h], Kr[h, :9], Vr[h, :9]) for h in range(n_q)])
    np.testing.assert_allclose(mha, per_head, rtol=1e-14)


def test_causal_attention_matches_library_sdpa():
    # All rows of a prompt vs torch's causal scaled_dot_product_attention.
    n_q, n_kv, T, d = 4, 2, 7, 8
    q = rng.standard_normal((n_q, T, d))
    K = rng.standard_normal((n_kv, T, d))
    V = rng.standard_normal((n_kv, T, d))
    ours = np.stack([O.gqa_attention(q[:, t], K, V, t + 1) for t in range(T)], 1)
    Kr = torch.from_numpy(np.repeat(K, 2, 0))
    Vr = torch.from_numpy(np.repeat(V, 2, 0))
    ref = F.scaled_dot_product_attention(torch.from_numpy(q), Kr, Vr, is_causal=True).numpy()
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- SwiGLU

def test_silu_closed_form():
    assert O.silu(np.array(0.0)) == 0.0
    np.testing.assert_allclose(O.silu(np.array(1.0)), math.e / (1 + math.e), rtol=1e-15)
    z = rng.standard_normal(100) * 6
    np.testing.assert_allclose(O.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-13, atol=1e-15)


def test_swiglu_gate_zero_and_orientation():
    H, I = 6, 10
    u = rng.standard_normal((3, H))
    wu, wd = rng.standard_normal((I, H)), rng.standard_normal((H, I))
    assert np.all(O.swiglu_ffn(u, np.zeros((I, H)), wu, wd) == 0.0)
    # W stored [out, in]: a single 1 at W[o, i] copies input i to output o.
    w = np.zeros((I, H))
    w[3, 5] = 1.0
    np.testing.assert_array_equal(O.linear(u, w)[:, 3], u[:, 5])
    wg = rng.standard_normal((I, H))
    a = F.silu(torch.from_numpy(u @ wg.T)).numpy() * (u @ wu.T)
    np.testing.assert_allclose(O.swiglu_ffn(u, wg, wu, wd), a @ wd.T, rtol=1e-13)


# ---------------------------------------------------------------- whole layer vs library composition

def _torch_layer_prefill(x, lw, shape):
    """The layer built from torch library routines (rms_norm, linear, complex
    RoPE, causal SDPA with repeated K/V heads, silu) in fp64."""
    T = x.shape[0]
    nq, nkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    t = {k: torch.from_numpy(v) for k, v in lw.items()}
    xt = torch.from_numpy(x)
    u = F.rms_norm(xt, (shape.hidden,), t["attn_norm"], eps=shape.rms_eps)
    qkv = F.linear(u, t["wqkv"])
    q = qkv[:, : nq * d].reshape(T, nq, d)
    k = qkv[:, nq * d: (nq + nkv) * d].reshape(T, nkv, d)
    v = qkv[:, (nq + nkv) * d:].reshape(T, nkv, d)
    freqs = shape.rope_theta ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones(T, d // 2, dtype=torch.float64),
                      torch.arange(T, dtype=torch.float64)[:, None] * freqs[None])

    def rope(z):
        zc = torch.view_as_complex(z.reshape(T, z.shape[1], d // 2, 2).contiguous())
        return torch.view_as_real(zc * rot[:, None]).reshape(T, z.shape[1], d)

    q, k = rope(q), rope(k)
    G = nq // nkv
    o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1).repeat_interleave(G, 0),
                                       v.transpose(0, 1).repeat_interleave(G, 0), is_causal=True)
    h = xt + F.linear(o.transpose(0, 1).reshape(T, nq * d), t["wo"])
    u2 = F.rms_norm(h, (shape.hidden,), t["ffn_norm"], eps=shape.rms_eps)
    ff = F.linear(F.silu(F.linear(u2, t["w_gate"])) * F.linear(u2, t["w_up"]), t["w_down"])
    return (h + ff).numpy()


@pytest.mark.parametrize("nq,nkv", [(4, 4), (4, 2), (8, 1)])
def test_layer_matches_library_composition(nq, nkv):
    shape = synth.Shape(1, 48, nq, nkv, 8, 40, 64, dtype="f32")   # n_q*d != hidden: no square weights
    w = {k: O.as64(v) for k, v in synth.layer_weights(shape, 5, 0, std=0.2).items()}
    x = rng.standard_normal((1, 9, 48))
    K = np.zeros((1, nkv, 16, 8))
    V = np.zeros((1, nkv, 16, 8))
    ours = O.layer_prefill(x, w, shape, K, V, cache_dtype="f64")[0]
    np.testing.assert_allclose(ours, _torch_layer_prefill(x[0], w, shape), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- KV cache semantics

def test_decode_step_equals_prefill_row():
    # The cache only removes recompute (§2.4): decoding token t after a prefill
    # of tokens 0..t-1 gives prefill row t.
    shape = synth.TINY
    w = synth.model_weights(shape, 1001)
    toks = synth.token_ids(2, 10, shape.vocab, 1001).numpy()
    full = O.Model(shape, w, 2, 16).prefill(toks)
    m = O.Model(shape, w, 2, 16)
    m.prefill(toks[:, :7])
    for t in range(7, 10):
        lg = m.decode(toks[:, t], np.full(2, t))
        np.testing.assert_allclose(lg, full[:, t], rtol=1e-10, atol=1e-12)


def test_paged_equals_contiguous():
    shape = synth.Shape(1, 32, 4, 2, 8, 24, 16, dtype="f32")
    lw = {k: O.as64(v) for k, v in synth.layer_weights(shape, 3, 0, std=0.3).items()}
    P, B = 4, 3
    lens = np.array([5, 9, 2])
    x = rng.standard_normal((B, 32))
    Kc = rng.standard_normal((B, 2, 16, 8))
    Vc = rng.standard_normal((B, 2, 16, 8))
    n_pages = [int(math.ceil((L + 1) / P)) for L in lens]
    table, total = synth.page_table(n_pages, 4, 3)
    table = table.numpy()
    Kp = np.zeros((total, 2, P, 8))
    Vp = np.zeros((total, 2, P, 8))
    for b in range(B):
        for m in range(lens[b]):
            Kp[table[b, m // P], :, m % P] = Kc[b, :, m]
            Vp[table[b, m // P], :, m % P] = Vc[b, :, m]
    contig = O.layer_decode(x, lw, shape, Kc.copy(), Vc.copy(), lens)
    paged = O.layer_decode_paged(x, lw, shape, Kp, Vp, table, lens, P)
    np.testing.assert_allclose(paged, contig, rtol=1e-13)
    contig = O.layer_decode(x, lw, shape, Kc.copy(), Vc.copy(), lens, cache_dtype="f64")
    paged = O.layer_decode_paged(x, lw, shape, Kp, Vp, table, lens, P, cache_dtype="f64")
    np.testing.assert_allclose(paged, contig, rtol=1e-13)
    for b in range(B):   # new token landed in its page slot
        m = lens[b]
        assert np.any(Kp[table[b, m // P], :, m % P] != 0)


def test_greedy_lowest_index_on_tie():
    assert list(O.greedy(np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0]]))) == [1, 0]


# ---------------------------------------------------------------- sizes the pages print

def _golden_table():
    rows = {}
    with open(os.path.join(GOLDEN, "size_table.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *vals = line.split()
                rows[k] = [float(v) for v in vals]
    return rows


def test_shapes_match_printed_size_table():
    g = _golden_table()
    for i, s in enumerate((synth.LLAMA2_7B, synth.LLAMA2_13B, synth.LLAMA2_70B)):
        assert [s.n_layers, s.hidden, s.n_q_heads, s.n_kv_heads, s.intermediate, s.vocab] == [
            g[k][i] for k in ("layers", "hidden", "heads", "kv_heads", "intermediate", "vocab")]
    assert 1 - synth.LLAMA2_70B.n_kv_heads / synth.LLAMA2_70B.n_q_heads == g["gqa_kv_saving_70b"][0]


def test_param_count_matches_printed_weight_sizes():
    g = _golden_table()
    assert O.param_count(synth.LLAMA2_7B) == 6_738_415_616          # the "7B"
    for i, s in enumerate((synth.LLAMA2_7B, synth.LLAMA2_13B, synth.LLAMA2_70B)):
        gb = O.param_count(s) * 2 / 1e9
        assert abs(gb - g["weights_fp16_gb"][i]) / g["weights_fp16_gb"][i] < 0.05


def test_kv_cache_formula_7b():
    # 7B, 4096 tokens, fp16: exactly 2 GiB, the page's "about 2GB".
    b = O.kv_cache_bytes(synth.LLAMA2_7B, 4096, 2)
    assert b == 2 * 1024 ** 3
    assert round(b / 1024 ** 3) == _golden_table()["kv_fp16_4096_gb"][0]


def test_embed_and_head_match_library():
    table = rng.standard_normal((20, 12))
    toks = np.array([3, 0, 19, 3])
    np.testing.assert_array_equal(O.embed(table, toks),
                                  F.embedding(torch.from_numpy(toks), torch.from_numpy(table)).numpy())
    h = rng.standard_normal((4, 12))
    g = 1 + 0.1 * rng.standard_normal(12)
    w = rng.standard_normal((20, 12))
    ref = F.linear(F.rms_norm(torch.from_numpy(h), (12,), torch.from_numpy(g), eps=1e-5), torch.from_numpy(w))
    np.testing.assert_allclose(O.lm_head(h, g, w, 1e-5), ref.numpy(), rtol=1e-13)


# ---------------------------------------------------------------- planted mistakes are caught

def _half_split_rope(x, positions, theta):
    d = x.shape[-1]
    phi = np.asarray(positions, dtype=np.float64)[:, None] * O.rope_frequencies(d, theta)[None, :]
    c, s = np.cos(phi)[:, None, :], np.sin(phi)[:, None, :]
    a, b = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], -1)


@pytest.mark.parametrize("mutant,pin", [
    ("rope", "test_rope_hand_angles"),
    ("rope", "test_rope_matches_complex_form"),
    ("gqa", "test_causal_attention_matches_library_sdpa"),
    ("scale", "test_attention_brute_force_tiny"),
    ("eps", "test_rmsnorm_eps_inside_root_and_scale_invariance"),
])
def test_pins_catch_planted_mistakes(monkeypatch, mutant, pin):
    if mutant == "rope":
        monkeypatch.setattr(O, "rope", _half_split_rope)
    elif mutant == "gqa":
        def wrong_gqa(q, K, V, n):
            return np.stack([O.attend(q[h], K[h % K.shape[0], :n], V[h % K.shape[0], :n])
                             for h in range(q.shape[0])])
        monkeypatch.setattr(O, "gqa_attention", wrong_gqa)
    elif mutant == "scale":
        monkeypatch.setattr(O, "attend", lambda q, K, V: O.softmax(K @ q) @ V)
    elif mutant == "eps":
        monkeypatch.setattr(O, "rmsnorm", lambda x, g, eps: x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps) * g)
    with pytest.raises(AssertionError):
        globals()[pin]()


# ---------------------------------------------------------------- KV cache storage type

def test_round_to_bf16_hand_values_and_library_cast():
    # ties go to the even significand
    assert O.round_to_bf16(np.array(1 + 2 ** -8)) == 1.0
    assert O.round_to_bf16(np.array(1 + 3 * 2 ** -8)) == 1 + 2 ** -6
    assert O.round_to_bf16(np.array(-(1 + 2 ** -7))) == -(1 + 2 ** -7)   # representable: unchanged
    assert O.round_to_bf16(np.array(0.0)) == 0.0
    x = (rng.standard_normal(100000) * 3).astype(np.float32).astype(np.float64)  # exact in fp32
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x), ref)


def test_cache_holds_storage_type_and_decode_still_equals_prefill():
    shape = synth.Shape(1, 32, 4, 2, 8, 24, 16, dtype="bf16")
    lw = {k: O.as64(v) for k, v in synth.layer_weights(shape, 8, 0, std=0.3).items()}
    x = rng.standard_normal((1, 6, 32))
    K = np.zeros((1, 2, 8, 8)); V = np.zeros_like(K)
    full = O.layer_prefill(x, lw, shape, K, V)[0]
    assert np.array_equal(K[:, :, :6], O.round_to_bf16(K[:, :, :6]))      # bf16 values only
    assert np.array_equal(V[:, :, :6], O.round_to_bf16(V[:, :, :6]))
    K2 = np.zeros_like(K); V2 = np.zeros_like(K)
    O.layer_prefill(x[:, :5], lw, shape, K2, V2)
    step = O.layer_decode(x[:, 5], lw, shape, K2, V2, [5])
    np.testing.assert_allclose(step[0], full[5], rtol=1e-12, atol=1e-12)
    # with fp64 storage the cache keeps the exact projections
    K3 = np.zeros_like(K); V3 = np.zeros_like(K)
    O.layer_prefill(x, lw, shape, K3, V3, cache_dtype="f64")
    assert not np.array_equal(K3[:, :, :6], O.round_to_bf16(K3[:, :, :6]))
    np.testing.assert_allclose(K[:, :, :6], K3[:, :, :6], rtol=2 ** -8)


# ---------------------------------------------------------------- sampling (§2.5, §3.3)

def test_sample_temperature_zero_is_greedy():
    rng = np.random.default_rng(21)
    z = rng.standard_normal(50)
    z[[3, 17]] = z.max() + 1.0  # a tie: the lower index wins
    for u in (0.0, 0.5, 0.999):
        assert O.sample_detail(z, None, 0.0, 0, 1.0, 1.0, u)["token"] == 3


def test_sample_top_k_one_is_argmax():
    rng = np.random.default_rng(22)
    z = rng.standard_normal(40)
    for T in (0.3, 1.0, 2.5):
        for u in (0.01, 0.6, 0.99):
            assert O.sample_detail(z, None, T, 1, 1.0, 1.0, u)["token"] == int(np.argmax(z))


def test_sample_draws_follow_the_library_softmax():
    # inverse-CDF draws over a uniform grid of u reproduce softmax(z / T)
    rng = np.random.default_rng(23)
    z = rng.standard_normal(7) * 2
    T, N = 0.8, 20000
    counts = np.zeros(7)
    for i in range(N):
        counts[O.sample_detail(z, None, T, 0, 1.0, 1.0, (i + 0.5) / N)["token"]] += 1
    np.testing.assert_allclose(counts / N, scipy.special.softmax(z / T), atol=1.5 / N)


def test_sample_top_k_keeps_the_k_largest_by_brute_force():
    rng = np.random.default_rng(24)
    z = np.round(rng.standard_normal(30), 1)  # rounding makes ties
    for k in (1, 3, 7, 29):
        ranked = sorted(range(30), key=lambda i: (-z[i], i))
        kept = O.sample_detail(z, None, 1.3, k, 1.0, 1.0, 0.5)["kept"]
        assert sorted(kept.tolist()) == sorted(ranked[:k])


def test_sample_top_p_hand_example():
    z = np.log(np.array([0.05, 0.5, 0.15, 0.3]))  # probabilities at T = 1
    cases = {0.45: [1], 0.7: [1, 3], 0.9: [1, 2, 3], 0.99: [0, 1, 2, 3]}
    for p, want in cases.items():
        d = O.sample_detail(z, None, 1.0, 0, p, 1.0, 0.3)
        assert d["kept"].tolist() == want, p
        np.testing.assert_allclose(d["q"].sum(), 1.0, rtol=1e-14)
    d = O.sample_detail(z, None, 1.0, 0, 0.7, 1.0, 0.3)
    np.testing.assert_allclose(d["q"], [0.5 / 0.8, 0.3 / 0.8], rtol=1e-12)


def test_sample_repetition_penalty_hand_example():
    z = np.array([2.0, -1.0, 0.5, 3.0, 1.0])
    d = O.sample_detail(z, [0, 1, 1, 3, 7, -2], 0.0, 0, 1.0, 2.0, 0.5)  # 7, -2: outside V
    np.testing.assert_array_equal(d["z"], [1.0, -2.0, 0.5, 1.5, 1.0])
    assert d["token"] == 3
    z2 = np.array([2.0, 1.9, 0.0])
    assert O.sample_detail(z2, [0], 0.0, 0, 1.0, 1.5, 0.5)["token"] == 1


def test_sample_draw_walks_the_vocabulary_in_ascending_order():
    z = np.log(np.array([0.2, 0.5, 0.3]))
    for u, want in ((0.1, 0), (0.19, 0), (0.3, 1), (0.69, 1), (0.75, 2), (0.999, 2)):
        assert O.sample_detail(z, None, 1.0, 0, 1.0, 1.0, u)["token"] == want, u


# ---------------------------------------------------------------- continuous batching (extend)

def test_extend_covers_prefill_decode_chunks_and_mixed_batches():
    # One extend step of rows (sequence, position) reproduces: a whole-prompt
    # prefill; a prompt fed in two pieces; ragged prompts in one batch; and a
    # decode token of one sequence next to a prompt piece of another.
    shape = synth.TINY
    w = synth.model_weights(shape, 1002)
    toks = synth.token_ids(2, 12, shape.vocab, 1002).numpy()
    full = O.Model(shape, w, 2, 16).prefill(toks)           # [2, 12, V]

    m = O.Model(shape, w, 2, 16)                              # whole prompts as one extend
    seq = np.repeat([0, 1], 12)
    pos = np.tile(np.arange(12), 2)
    lg = m.extend(toks.reshape(-1), seq, pos)
    np.testing.assert_allclose(lg.reshape(2, 12, -1), full, rtol=1e-10, atol=1e-12)

    m = O.Model(shape, w, 2, 16)                              # ragged: 5 and 9 tokens, then the rest
    seq = np.array([0] * 5 + [1] * 9)
    pos = np.concatenate([np.arange(5), np.arange(9)])
    lg = m.extend(np.concatenate([toks[0, :5], toks[1, :9]]), seq, pos)
    np.testing.assert_allclose(lg[:5], full[0, :5], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lg[5:], full[1, :9], rtol=1e-10, atol=1e-12)
    # mixed: sequence 1 decodes token 9 while sequence 0 feeds its prompt piece 5..11
    seq = np.array([0] * 7 + [1])
    pos = np.concatenate([np.arange(5, 12), [9]])
    lg = m.extend(np.concatenate([toks[0, 5:], toks[1, 9:10]]), seq, pos)
    np.testing.assert_allclose(lg[:7], full[0, 5:], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lg[7], full[1, 9], rtol=1e-10, atol=1e-12)
    lg = m.extend(toks[1, 10:11], np.array([1]), np.array([10]))  # sequence 1 alone continues
    np.testing.assert_allclose(lg[0], full[1, 10], rtol=1e-10, atol=1e-12)


def test_extend_of_one_token_per_sequence_is_decode():
    shape = synth.TINY
    w = synth.model_weights(shape, 1003)
    toks = synth.token_ids(3, 6, shape.vocab, 1003).numpy()
    a, b = O.Model(shape, w, 3, 8), O.Model(shape, w, 3, 8)
    a.prefill(toks[:, :5])
    b.prefill(toks[:, :5])
    want = a.decode(toks[:, 5], np.full(3, 5))
    got = b.extend(toks[:, 5], np.arange(3), np.full(3, 5))
    np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------------- FP8 (E4M3) cache storage

def test_round_to_e4m3_hand_values():
    x = np.array([0.0, 1.0625, 1.1875, 17.0, 19.0, 2.0**-9, 2.0**-10, 3 * 2.0**-11, 2.0**-6,
                  448.0, 464.0, 500.0, -500.0, -0.3])
    want = np.array([0.0, 1.0, 1.25, 16.0, 20.0, 2.0**-9, 0.0, 2.0**-9, 2.0**-6,
                     448.0, 448.0, 448.0, -448.0, -0.3125])
    np.testing.assert_array_equal(O.round_to_e4m3(x), want)


def test_round_to_e4m3_matches_library_cast():
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(50000) * 0.01])
    x = np.clip(x, -448, 448).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_e4m3(x.astype(np.float64)), lib)


def test_e4m3_cache_stores_scaled_values_and_decode_still_equals_prefill():
    shape = synth.TINY
    w = synth.model_weights(shape, 1004)
    toks = synth.token_ids(2, 9, shape.vocab, 1004).numpy()
    cdt = ("e4m3", 0.05, 0.03)
    full = O.Model(shape, w, 2, 12, cache_dtype=cdt).prefill(toks)
    m = O.Model(shape, w, 2, 12, cache_dtype=cdt)
    m.prefill(toks[:, :6])
    for t in range(6, 9):
        np.testing.assert_allclose(m.decode(toks[:, t], np.full(2, t)), full[:, t], rtol=1e-10,
                                   atol=1e-12)
    k = m.K[0][:, :, :9] / 0.05  # every stored K is an E4M3 value times the scale
    np.testing.assert_allclose(O.round_to_e4m3(k), k, rtol=1e-14, atol=0)
    assert len(np.unique(np.round(np.abs(k[k != 0]), 9))) < 250  # at most 2 x 126 finite magnitudes


# ---------------------------------------------------------------- FP8 (E4M3) weights, row scales

def test_quantize_rows_e4m3_hand_rows():
    w = np.array([[0.5, -1.0, 0.25, 0.0],
                  [0.0, 0.0, 0.0, 0.0],
                  [3.0, 0.01, -0.75, 1.5]])
    codes, s = O.quantize_rows_e4m3(w)
    np.testing.assert_array_equal(s, np.float32([1 / 448, 1.0, 3 / 448]).astype(np.float64))
    np.testing.assert_array_equal(codes[0], [224.0, -448.0, 112.0, 0.0])
    np.testing.assert_array_equal(codes[1], [0.0, 0.0, 0.0, 0.0])
    # 0.01 / (3/448) = 1.4933 -> 1.5; -0.75 / (3/448) = -112; 1.5 -> 224
    np.testing.assert_array_equal(codes[2], [448.0, 1.5, -112.0, 224.0])


def test_quantize_rows_e4m3_matches_library_cast_and_maps_row_max_to_448():
    rng = np.random.default_rng(32)
    w = (rng.standard_normal((37, 300)) * 0.02).astype(np.float32)  # non-square: rows are outputs
    w[5] *= 1000.0
    w[9] = 0.0
    codes, s = O.quantize_rows_e4m3(w)
    wt = torch.from_numpy(w)
    st = torch.where(wt.abs().amax(1) > 0, wt.abs().amax(1) / 448.0, torch.ones(37))
    lib = (wt / st[:, None]).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(s, st.double().numpy())
    np.testing.assert_array_equal(codes, lib)
    nz = np.abs(w).max(1) > 0
    np.testing.assert_array_equal(np.abs(codes[nz]).max(1), np.full(nz.sum(), 448.0))
    assert np.all(codes[9] == 0) and s[9] == 1.0


def test_dequantized_rows_are_within_half_an_e4m3_step():
    rng = np.random.default_rng(33)
    w = rng.standard_normal((64, 512)) * 0.02
    codes, s = O.quantize_rows_e4m3(w)
    deq = O.dequantize_rows(codes, s)
    # half the spacing: 2^-4 relative for normals, 2^-10 * s below 2^-6 * s
    bound = np.maximum(np.abs(w) * 2.0**-4, s[:, None] * 2.0**-10) * (1 + 1e-6)
    assert np.all(np.abs(w - deq) <= bound)
    assert np.abs(w - deq).max() > 0  # it does quantise


def test_row_scales_factor_out_of_the_projection():
    # y[n, m] = s_m * sum_k u[n, k] code[m, k]: the row scale can be applied to
    # the accumulator after the contraction
    rng = np.random.default_rng(34)
    w = rng.standard_normal((24, 40)) * 0.05
    u = rng.standard_normal((7, 40))
    codes, s = O.quantize_rows_e4m3(w)
    np.testing.assert_allclose(O.linear(u, O.dequantize_rows(codes, s)), (u @ codes.T) * s[None, :],
                               rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- generation loop (§3.4)

def test_generate_greedy_equals_prefill_of_the_extended_prompt():
    # The generation loop feeds each greedy choice back at the next position
    # ("Llama2架构与推理全解析" §3.4) and the cache only saves recompute (§2.4):
    # step s's logits are the last row of a fresh prefill of the prompt
    # followed by the first s chosen ids, and each id is its row's argmax.
    shape = synth.TINY.with_(n_layers=1)
    w = synth.model_weights(shape, 1011)
    B, T, n = 2, 9, 5
    prompt = synth.token_ids(B, T, shape.vocab, 1011).numpy()
    ids, lg = O.generate_greedy(O.Model(shape, w, B, T + n + 1), prompt, n)
    assert ids.shape == (B, n + 1) and lg.shape == (B, n + 1, shape.vocab)
    for s in range(n + 1):
        seq = np.concatenate([prompt, ids[:, :s]], axis=1)
        ref = O.Model(shape, w, B, T + n + 1).prefill(seq)[:, -1]
        np.testing.assert_allclose(lg[:, s], ref, rtol=1e-10, atol=1e-12)
        top2 = np.sort(ref, -1)[:, -2:]
        assert np.all(top2[:, 1] - top2[:, 0] > 1e-9)  # the choice is unambiguous
        np.testing.assert_array_equal(ids[:, s], np.argmax(ref, -1))


def _generate_position_off_by_one(model, prompt, n_steps):
    prompt = np.asarray(prompt)
    B, T = prompt.shape
    lg = model.prefill(prompt)[:, -1]
    ids, logits = [O.greedy(lg)], [lg]
    for s in range(n_steps):
        lg = model.decode(ids[-1], np.full(B, T + s + 1))
        ids.append(O.greedy(lg))
        logits.append(lg)
    return np.stack(ids, 1), np.stack(logits, 1)


def _generate_feeds_first_choice(model, prompt, n_steps):
    prompt = np.asarray(prompt)
    B, T = prompt.shape
    lg = model.prefill(prompt)[:, -1]
    ids, logits = [O.greedy(lg)], [lg]
    for s in range(n_steps):
        lg = model.decode(ids[0], np.full(B, T + s))
        ids.append(O.greedy(lg))
        logits.append(lg)
    return np.stack(ids, 1), np.stack(logits, 1)


@pytest.mark.parametrize("mutant", [_generate_position_off_by_one, _generate_feeds_first_choice])
def test_generate_greedy_pin_catches_planted_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(O, "generate_greedy", mutant)
    with pytest.raises(AssertionError):
        test_generate_greedy_equals_prefill_of_the_extended_prompt()
