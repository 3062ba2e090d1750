"""FP8 E4M3 KV cache (one byte per value, times a per-tensor scale) against the
oracle's scaled E4M3 cache: the cache writes of the RoPE/append kernel and of
the fused decode epilogue, the E4M3 flash-decode kernel (contiguous and paged,
MHA and GQA), a 7B layer decode step, and prefill + decode of a small model."""
import math

import numpy as np
import pytest
import torch

from _common import BF16_TOL, assert_close, f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu

L7 = synth.LLAMA2_7B.with_(n_layers=1)
KS, VS = 0.02, 0.015  # cache scales (not powers of two, so the scaling is exercised)


def _e4m3_values(cache_u8):
    """Stored bytes -> E4M3 values (float64), by the library cast of the bytes."""
    return cache_u8.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _quantise(x, scale):
    """E4M3 bytes of x / scale, by the oracle's rounding (checked against
    torch's cast in the oracle pins)."""
    q = O.round_to_e4m3(np.asarray(x, np.float64) / scale)
    return torch.from_numpy(q).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def _near(got, want, scale):
    """Within one E4M3 step of the oracle's stored value (fp32 on the GPU and
    fp64 in the oracle may land on the two sides of a rounding boundary)."""
    w = np.abs(np.asarray(want) / scale)
    ex = np.maximum(np.floor(np.log2(np.maximum(w, 2.0**-9))), -6).astype(np.int64) - 3
    step = np.ldexp(1.0, ex) * scale
    bad = np.abs(np.asarray(got) - np.asarray(want)) > step * 1.0001
    assert bad.mean() < 0.01 and not np.any(np.abs(np.asarray(got) - np.asarray(want)) > 2.0001 * step)


def _ctx(shape, B, max_seq, max_tokens=0, seed=5):
    need_gpu()
    w = {"layers": [synth.layer_weights(shape, seed, 0)]}
    return binding.Model(shape, to_dev(w), max_batch=B, max_tokens=max_tokens, max_seq=max_seq,
                         has_embed_head=False)


@pytest.mark.parametrize("paged", [False, True])
def test_rope_append_writes_e4m3(paged):
    shape = L7
    m = _ctx(shape, 8, 1040)
    B, nq, nkv, d = 6, shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    pos = torch.tensor([0, 1, 15, 16, 100, 1023], dtype=torch.int32)
    g = torch.Generator().manual_seed(61)
    qkv = torch.randn(B, shape.qkv_rows, generator=g) * 1.5
    if paged:
        n_pages = [int(p) // 16 + 1 for p in pos]
        table, total = synth.page_table(n_pages, max(n_pages), 61)
        kv = binding.KVCache(shape, n_pages=total, page_size=16, page_table=table.cuda(),
                             e4m3=(KS, VS))
    else:
        kv = binding.KVCache(shape, batch=B, capacity=1040, e4m3=(KS, VS))
    q_out = torch.empty(B, nq * d, dtype=torch.bfloat16, device="cuda")
    m.op_rope_append(qkv.cuda(), 1, pos.cuda(), 0, kv, q_out)
    m.sync()
    x = f64(qkv)
    k = O.rope(x[:, nq * d:(nq + nkv) * d].reshape(B, nkv, d), pos.numpy(), 1e4)
    v = x[:, (nq + nkv) * d:].reshape(B, nkv, d)
    K, V = _e4m3_values(kv.k)[0] * KS, _e4m3_values(kv.v)[0] * VS
    for b in range(B):
        p = int(pos[b])
        if paged:
            kk, vv = K[int(table[b, p // 16]), :, p % 16], V[int(table[b, p // 16]), :, p % 16]
        else:
            kk, vv = K[b, :, p], V[b, :, p]
        _near(kk, O.cache_store(k[b], "e4m3", KS), KS)
        _near(vv, O.cache_store(v[b], "e4m3", VS), VS)
    assert int((kv.k != 0).sum()) <= B * nkv * d


@pytest.mark.parametrize("nq,nkv", [(32, 32), (32, 8)])
@pytest.mark.parametrize("page_size", [0, 16, 64])
def test_decode_attention_e4m3(nq, nkv, page_size):
    shape = L7.with_(n_q_heads=nq, n_kv_heads=nkv)
    positions = [0, 14, 15, 16, 63, 64, 65, 1024, 2047, 333]
    B, d = len(positions), shape.head_dim
    m = _ctx(shape, B, 2112)
    g = torch.Generator().manual_seed(62)
    q = (torch.randn(B, nq, d, generator=g)).to(torch.bfloat16)
    lens = [p + 1 for p in positions]
    if page_size:
        n_pages = [math.ceil(L / page_size) for L in lens]
        table, total = synth.page_table(n_pages, max(n_pages), 62)
        kf = torch.randn(1, total, nkv, page_size, d, generator=g).numpy()
        vf = torch.randn(1, total, nkv, page_size, d, generator=g).numpy()
        kv = binding.KVCache(shape, n_pages=total, page_size=page_size, page_table=table.cuda(),
                             k=_quantise(kf, KS).cuda(), v=_quantise(vf, VS).cuda(), e4m3=(KS, VS))
        logical = lambda pool, b, n: O.gather_paged(pool, table[b].numpy(), n, page_size)
    else:
        cap = max(lens) + 16
        kf = torch.randn(1, B, nkv, cap, d, generator=g).numpy()
        vf = torch.randn(1, B, nkv, cap, d, generator=g).numpy()
        kv = binding.KVCache(shape, batch=B, capacity=cap, k=_quantise(kf, KS).cuda(),
                             v=_quantise(vf, VS).cuda(), e4m3=(KS, VS))
        logical = lambda pool, b, n: pool[b, :, :n]
    Kf, Vf = _e4m3_values(kv.k)[0] * KS, _e4m3_values(kv.v)[0] * VS
    out = torch.empty(B, nq * d, dtype=torch.bfloat16, device="cuda")
    m.op_attention_decode(q.cuda(), torch.tensor(positions, dtype=torch.int32).cuda(), 0, kv, out)
    m.sync()
    qf = f64(q)
    for b, n in enumerate(lens):
        ref = O.gqa_attention(qf[b], logical(Kf, b, n), logical(Vf, b, n), n)
        assert_close(out[b].view(nq, d), ref, BF16_TOL, "e4m3 decode attention b=%d n=%d" % (b, n))


def test_layer_decode_7b_e4m3_cache():
    need_gpu()
    shape, B, S, seed = L7, 32, 1024, 2101
    lw = synth.layer_weights(shape, seed, 0, std=0.02)
    nkv, d = shape.n_kv_heads, shape.head_dim
    cap = S + 16
    g = torch.Generator().manual_seed(seed)
    kf = torch.randn(1, B, nkv, cap, d, generator=g).numpy() * 2
    vf = torch.randn(1, B, nkv, cap, d, generator=g).numpy()
    kf[:, :, :, S:] = 0
    vf[:, :, :, S:] = 0
    kv = binding.KVCache(shape, batch=B, capacity=cap, k=_quantise(kf, KS).cuda(),
                         v=_quantise(vf, VS).cuda(), e4m3=(KS, VS))
    K, V = _e4m3_values(kv.k)[0] * KS, _e4m3_values(kv.v)[0] * VS
    x = synth.hidden_input(B, shape.hidden, seed)
    m = binding.Model(shape, to_dev({"layers": [lw]}), max_batch=B, max_tokens=0, max_seq=cap,
                      has_embed_head=False)
    pos = torch.full((B,), S, dtype=torch.int32)
    h = x.cuda()
    m.decode_hidden(h, pos.cuda(), kv)
    m.sync()
    lw64 = {k: f64(v) for k, v in lw.items()}
    ref = O.layer_decode(f64(x), lw64, shape, K, V, pos.numpy(), cache_dtype=("e4m3", KS, VS))
    assert_close(h, ref, BF16_TOL, "layer output over an e4m3 cache")
    got = _e4m3_values(kv.k)[0][np.arange(B), :, S] * KS
    _near(got, K[np.arange(B), :, S], KS)


def test_layer_prefill_7b_e4m3_cache_token_major_gemms():
    # 640 prompt rows: the Q/K/V projection (with RoPE and the E4M3 append in
    # its epilogue) and gate/up run on the persistent token-major GEMM, the O
    # and down projections (80 tiles) on the other one
    need_gpu()
    shape, B, T, seed = L7, 2, 320, 2103
    lw = synth.layer_weights(shape, seed, 0, std=0.02)
    kv = binding.KVCache(shape, batch=B, capacity=T, e4m3=(KS, VS))
    x = synth.hidden_input(B * T, shape.hidden, seed)
    m = binding.Model(shape, to_dev({"layers": [lw]}), max_batch=B, max_tokens=B * T, max_seq=T,
                      has_embed_head=False)
    h = x.cuda()
    m.prefill_hidden(h, B, T, kv)
    m.sync()
    rows = [0, 1, 127, 128, 255, 319]
    K = np.zeros((B, shape.n_kv_heads, T, shape.head_dim))
    V = np.zeros_like(K)
    lw64 = {k: f64(v) for k, v in lw.items()}
    ref = O.layer_prefill(f64(x).reshape(B, T, -1), lw64, shape, K, V, rows=rows,
                          cache_dtype=("e4m3", KS, VS))
    assert_close(f64(h).reshape(B, T, -1)[:, rows], ref, BF16_TOL, "prefill rows, e4m3 cache")
    for t in (0, 200, 319):
        _near(_e4m3_values(kv.k)[0][:, :, t] * KS, K[:, :, t], KS)
        _near(_e4m3_values(kv.v)[0][:, :, t] * VS, V[:, :, t], VS)


def test_prefill_then_decode_small_model_e4m3():
    need_gpu()
    shape = synth.Shape(2, 256, 4, 2, 128, 512, 512, dtype="bf16")
    B, T, cap, seed = 2, 24, 32, 2102
    w = synth.model_weights(shape, seed)
    toks = synth.token_ids(B, T + 3, shape.vocab, seed)
    m = binding.Model(shape, to_dev(w), max_batch=B, max_tokens=B * T, max_seq=cap)
    kv = binding.KVCache(shape, batch=B, capacity=cap, e4m3=(0.05, 0.03))
    ref = O.Model(shape, w, B, cap, cache_dtype=("e4m3", 0.05, 0.03))
    lg = torch.empty(B, shape.vocab, device="cuda")
    m.prefill(toks[:, :T].contiguous().cuda(), kv, lg)
    m.sync()
    want = ref.prefill(toks[:, :T].numpy())[:, -1]
    assert_close(lg, want, BF16_TOL, "prefill logits over an e4m3 cache")
    for t in range(T, T + 3):
        pos = torch.full((B,), t, dtype=torch.int32)
        m.decode_step(toks[:, t].contiguous().cuda(), pos.cuda(), kv, lg)
        m.sync()
        assert_close(lg, ref.decode(toks[:, t].numpy(), pos.numpy()), BF16_TOL,
                     "decode logits over an e4m3 cache, step %d" % t)


def test_e4m3_host_checks():
    need_gpu()
    shape = synth.Shape(1, 256, 4, 2, 128, 512, 512, dtype="bf16")
    m = binding.Model(shape, to_dev(synth.model_weights(shape, 3)), max_batch=2, max_tokens=16,
                      max_seq=32)
    lg = torch.empty(2, shape.vocab, device="cuda")
    tok = torch.zeros(2, dtype=torch.int32, device="cuda")
    pos = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.LlamaError, match="INVALID_ARG"):
        m.decode_step(tok, pos, binding.KVCache(shape, batch=2, capacity=32, e4m3=(0.0, 1.0)), lg)
    kv = binding.KVCache(shape, batch=2, capacity=32, e4m3=(1.0, 1.0))
    cu = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    with pytest.raises(binding.LlamaError, match="UNSUPPORTED"):
        m.extend(tok, cu, pos, kv, lg, max_rows=1)
    tiny = synth.TINY.with_(n_layers=1)
    mf = binding.Model(tiny, to_dev(synth.model_weights(tiny, 3)), max_batch=2, max_tokens=16,
                       max_seq=32)
    with pytest.raises(binding.LlamaError, match="UNSUPPORTED"):
        mf.decode_step(tok, pos, binding.KVCache(tiny, batch=2, capacity=32, e4m3=(1.0, 1.0)),
                       torch.empty(2, tiny.vocab, device="cuda"))
