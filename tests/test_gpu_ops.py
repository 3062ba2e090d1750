"""Each kernel of the forward pass against the CPU oracle, through the C ABI's
single-operation entry points, on seeded inputs spanning several tiles and a
ragged tail."""
import math

import numpy as np
import pytest
import torch

from _common import BF16_TOL, F32_TOL, assert_close, f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu

# fp32-accumulated GEMM outputs: K <= 11008 bf16 products of magnitude < 0.2
# summed in fp32 stay within 1e-3 of the exact sum.
GEMM_F32_TOL = (2e-3, 1e-3)

L7 = synth.LLAMA2_7B.with_(n_layers=1)


def ctx_for(shape, max_batch=64, max_tokens=4096, max_seq=4608, embed=False, seed=5, n_layers=1):
    need_gpu()
    shape = shape.with_(n_layers=n_layers)
    w = synth.model_weights(shape, seed) if embed else \
        {"layers": [synth.layer_weights(shape, seed, l) for l in range(n_layers)]}
    wd = to_dev(w)
    m = binding.Model(shape, wd, max_batch=max_batch, max_tokens=max_tokens, max_seq=max_seq,
                      has_embed_head=embed)
    return m, w


@pytest.fixture(scope="module")
def ctx7():
    return ctx_for(L7)[0]


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _randn(shape, std, dtype, seed):
    return (torch.randn(*shape, generator=_gen(seed)) * std).to(dtype)


# --------------------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("rows,stride,offset", [(37, 1, 0), (4, 5, 4), (1, 1, 0)])
def test_rmsnorm_bf16(ctx7, rows, stride, offset):
    H = L7.hidden
    x = _randn((rows * stride, H), 2.0, torch.float32, 11)
    gamma = (1 + 0.1 * torch.randn(H, generator=_gen(12))).to(torch.bfloat16)
    out = torch.empty(rows, H, dtype=torch.bfloat16, device="cuda")
    ctx7.op_rmsnorm(x.cuda(), gamma.cuda(), out, rows=rows, stride=stride, offset=offset)
    ctx7.sync()
    xs = f64(x)[offset::stride][:rows]
    assert_close(out, O.rmsnorm(xs, f64(gamma), 1e-5), BF16_TOL, "rmsnorm")


def test_rmsnorm_f32():
    m, _ = ctx_for(synth.TINY, max_batch=4, max_tokens=16, max_seq=32)
    x = _randn((9, 256), 1.0, torch.float32, 13)
    gamma = 1 + 0.1 * torch.randn(256, generator=_gen(14))
    out = torch.empty(9, 256, device="cuda")
    m.op_rmsnorm(x.cuda(), gamma.cuda(), out)
    m.sync()
    assert_close(out, O.rmsnorm(f64(x), f64(gamma), 1e-5), F32_TOL, "rmsnorm f32")


# --------------------------------------------------------------------------- linear (tcgen05)
EPIS = {"store_f32": binding.EPI_STORE_F32, "resid": binding.EPI_RESID_F32,
        "store_t": binding.EPI_STORE_T, "swiglu": binding.EPI_SWIGLU}


@pytest.mark.parametrize("M,N,K,epi", [
    (12288, 32, 4096, "store_f32"),   # decode Q/K/V, split K
    (4096, 32, 4096, "resid"),        # decode output projection + residual
    (11008, 32, 4096, "swiglu"),      # decode gate/up + SiLU*up
    (4096, 32, 11008, "resid"),       # decode down projection + residual
    (32000, 8, 4096, "store_f32"),    # LM head, 8 sequences (N padded to 16)
    (4096, 1, 4096, "store_t"),       # one row
    (640, 300, 4104, "store_t"),      # ragged N (two tiles) and ragged K
    (200, 64, 256, "store_f32"),      # ragged M
    (4096, 4096, 4096, "resid"),      # prefill-sized tile grid
    (1024, 1000, 512, "swiglu"),      # prefill SwiGLU, ragged N
])
def test_linear_bf16(ctx7, M, N, K, epi):
    x = _randn((N, K), 1.0, torch.bfloat16, 21)
    w = _randn((M, K), 0.02, torch.bfloat16, 22)
    wu = _randn((M, K), 0.02, torch.bfloat16, 23) if epi == "swiglu" else None
    xd, wd = x.cuda(), w.cuda()
    wud = wu.cuda() if wu is not None else None
    ref = O.linear(f64(x), f64(w))
    if epi == "swiglu":
        ref = O.silu(ref) * O.linear(f64(x), f64(wu))
    if epi in ("store_t", "swiglu"):
        out = torch.empty(N, M, dtype=torch.bfloat16, device="cuda")
        tol = BF16_TOL
    else:
        out = torch.empty(N, M, dtype=torch.float32, device="cuda")
        tol = GEMM_F32_TOL
    if epi == "resid":
        base = _randn((N, M), 1.0, torch.float32, 24)
        out.copy_(base)
        ref = ref + f64(base)
    for _ in range(2):  # second call reuses the split-K counters
        if epi == "resid":
            out.copy_(base)
        ctx7.op_linear(xd, wd, out, EPIS[epi], w_up=wud)
        ctx7.sync()
        assert_close(out, ref, tol, "linear %s M=%d N=%d K=%d" % (epi, M, N, K))


def _pair(x):
    """hi/lo bf16 pair layout of fp32 rows: [hi rows, pad, lo rows, pad]."""
    n, K = x.shape
    L = (n + 15) // 16 * 16
    hi = x.to(torch.bfloat16)
    lo = (x - hi.float()).to(torch.bfloat16)
    out = torch.zeros(2 * L, K, dtype=torch.bfloat16)
    out[:n] = hi
    out[L:L + n] = lo
    return out, L


@pytest.mark.parametrize("M,N,K,epi", [
    (12288, 32, 4096, "store_f32"),
    (11008, 32, 4096, "swiglu"),
    (4096, 100, 11008, "resid"),
    (32000, 8, 4096, "store_f32"),
    (1024, 1, 256, "store_t"),
    # at least one 128-row x 256-feature tile per SM: the persistent kernel
    # with the activation rows on the MMA's M side (ragged rows, features, K)
    (12288, 1000, 4096, "store_f32"),
    (4000, 1300, 4104, "resid"),
    (2816, 1200, 4096, "swiglu"),
    (4096, 1200, 1024, "store_t"),
    (2900, 1200, 4096, "swiglu"),      # ragged features with gate and up halves
    (12200, 1000, 4096, "store_f32"),  # M % 16 != 0: unaligned rows, element stores
    (4096, 1100, 4096, "resid"),       # 144 tiles: one round on fewer CTAs than SMs
])
def test_linear_bf16_pair_operands(ctx7, M, N, K, epi):
    # fp32 activations carried as bf16 hi + lo: the product tracks the fp32 values
    x = _randn((N, K), 1.0, torch.float32, 25)
    w = _randn((M, K), 0.02, torch.bfloat16, 26)
    wu = _randn((M, K), 0.02, torch.bfloat16, 27) if epi == "swiglu" else None
    xp, L = _pair(x)
    ref = O.linear(f64(x), f64(w))
    if epi == "swiglu":
        ref = O.silu(ref) * O.linear(f64(x), f64(wu))
    if epi in ("store_t", "swiglu"):
        out = torch.zeros(2 * L, M, dtype=torch.bfloat16, device="cuda")
    else:
        out = torch.zeros(N, M, dtype=torch.float32, device="cuda")
    if epi == "resid":
        base = _randn((N, M), 1.0, torch.float32, 28)
        out.copy_(base)
        ref = ref + f64(base)
    ctx7.op_linear(xp.cuda(), w.cuda(), out, EPIS[epi] | binding.EPI_SPLIT_X,
                   w_up=wu.cuda() if wu is not None else None, n_rows=N)
    ctx7.sync()
    got = f64(out[:N]) + f64(out[L:L + N]) if epi in ("store_t", "swiglu") else f64(out)
    assert_close(got, ref, GEMM_F32_TOL, "pair-operand linear %s" % epi)


@pytest.mark.parametrize("epi", list(EPIS))
def test_linear_f32(epi):
    m, _ = ctx_for(synth.TINY, max_batch=4, max_tokens=16, max_seq=32)
    M, N, K = 688, 16, 256
    x = _randn((N, K), 1.0, torch.float32, 31)
    w = _randn((M, K), 0.02, torch.float32, 32)
    wu = _randn((M, K), 0.02, torch.float32, 33)
    ref = O.linear(f64(x), f64(w))
    if epi == "swiglu":
        ref = O.silu(ref) * O.linear(f64(x), f64(wu))
    out = torch.zeros(N, M, device="cuda")
    m.op_linear(x.cuda(), w.cuda(), out, EPIS[epi], w_up=wu.cuda())
    m.sync()
    assert_close(out, ref, F32_TOL, "linear f32 " + epi)


# --------------------------------------------------------------------------- RoPE + append
def _paged_setup(lengths, n_kv, d, page, seed, dtype, n_layers=1, extra_slot=True):
    n_pages = [math.ceil((L + (1 if extra_slot else 0)) / page) for L in lengths]
    maxp = max(n_pages)
    table, total = synth.page_table(n_pages, maxp, seed)
    return table, total


@pytest.mark.parametrize("paged", [False, True])
def test_rope_append_bf16(ctx7, paged):
    shape = L7
    B = 6
    nq, nkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    pos = torch.tensor([0, 1, 15, 16, 100, 1023], dtype=torch.int32)
    qkv = _randn((B, shape.qkv_rows), 1.5, torch.float32, 41)
    if paged:
        table, total = _paged_setup([int(p) for p in pos], nkv, d, 16, 41, torch.bfloat16)
        kv = binding.KVCache(shape, n_pages=total, page_size=16, page_table=table.cuda())
    else:
        kv = binding.KVCache(shape, batch=B, capacity=1040)
    q_out = torch.empty(B, nq * d, dtype=torch.bfloat16, device="cuda")
    ctx7.op_rope_append(qkv.cuda(), 1, pos.cuda(), 0, kv, q_out)
    ctx7.sync()
    q, k, v = (f64(qkv)[:, : nq * d].reshape(B, nq, d), f64(qkv)[:, nq * d:(nq + nkv) * d].reshape(B, nkv, d),
               f64(qkv)[:, (nq + nkv) * d:].reshape(B, nkv, d))
    assert_close(q_out.view(B, nq, d), O.rope(q, pos.numpy(), 1e4), BF16_TOL, "rotated q")
    kref = O.rope(k, pos.numpy(), 1e4)
    K, V = f64(kv.k)[0], f64(kv.v)[0]
    for b in range(B):
        m = int(pos[b])
        if paged:
            page = int(table[b, m // 16])
            kk, vv = K[page, :, m % 16], V[page, :, m % 16]
        else:
            kk, vv = K[b, :, m], V[b, :, m]
        assert_close(kk, kref[b], BF16_TOL, "cached k")
        assert_close(vv, v[b], BF16_TOL, "cached v")
    # nothing else in the cache was written
    assert int((kv.k != 0).sum()) == B * nkv * d
    assert int((kv.v != 0).sum()) == B * nkv * d


# --------------------------------------------------------------------------- decode attention
def _decode_case(nq, nkv, positions, paged, seed, cap=None):
    """paged: False (contiguous cache) or the page size in keys."""
    shape = L7.with_(n_q_heads=nq, n_kv_heads=nkv)
    m, _ = ctx_for(shape, max_batch=len(positions), max_tokens=0, max_seq=4608)
    B, d = len(positions), shape.head_dim
    pos = torch.tensor(positions, dtype=torch.int32)
    q = _randn((B, nq, d), 1.0, torch.bfloat16, seed)
    if paged:
        ps = int(paged)
        table, total = _paged_setup(positions, nkv, d, ps, seed, torch.bfloat16)
        k = synth.cache_values((1, total, nkv, ps, d), seed, torch.bfloat16, stream=0)
        v = synth.cache_values((1, total, nkv, ps, d), seed, torch.bfloat16, stream=1)
        kv = binding.KVCache(shape, n_pages=total, page_size=ps, page_table=table.cuda(),
                             k=k.cuda(), v=v.cuda())
        Kf, Vf = f64(k)[0], f64(v)[0]
        logical = lambda pool, b, n: O.gather_paged(pool, table[b].numpy(), n, ps)
    else:
        cap = cap or (max(positions) + 1 + 15) // 16 * 16
        k = synth.cache_values((1, B, nkv, cap, d), seed, torch.bfloat16, stream=0)
        v = synth.cache_values((1, B, nkv, cap, d), seed, torch.bfloat16, stream=1)
        kv = binding.KVCache(shape, batch=B, capacity=cap, k=k.cuda(), v=v.cuda())
        Kf, Vf = f64(k)[0], f64(v)[0]
        logical = lambda pool, b, n: pool[b, :, :n]
    out = torch.empty(B, nq * d, dtype=torch.bfloat16, device="cuda")
    m.op_attention_decode(q.cuda(), pos.cuda(), 0, kv, out)
    m.sync()
    qf = f64(q)
    for b in range(B):
        n = int(pos[b]) + 1
        ref = O.gqa_attention(qf[b], logical(Kf, b, n), logical(Vf, b, n), n)
        assert_close(out[b].view(nq, d), ref, BF16_TOL, "decode attention b=%d n=%d" % (b, n))


@pytest.mark.parametrize("nq,nkv", [(32, 32), (32, 8), (16, 4), (16, 8)])
@pytest.mark.parametrize("paged", [False, 16, 64])
def test_attention_decode_bf16(nq, nkv, paged):
    positions = [0, 14, 15, 16, 17, 63, 64, 65, 1024, 2047, 4095, 333]
    _decode_case(nq, nkv, positions, paged, 51)


def test_attention_decode_full_capacity():
    # the key range ends exactly at the cache capacity (last slot in use)
    _decode_case(8, 8, [1039, 1039, 0], False, 52, cap=1040)


def test_attention_decode_many_splits():
    # few (sequence, head) pairs and long context: several key splits merged
    _decode_case(64, 8, [4096, 3000], False, 53)


def test_attention_decode_positions_outside_the_planned_keys_are_flagged():
    # max_seq 256 against a 1024-slot cache: the split plan covers 256 keys, so
    # position 600 is flagged; a negative position gives zero rows and a flag;
    # an in-range sequence of the same launch is unaffected
    shape = L7.with_(n_q_heads=8, n_kv_heads=8)
    m, _ = ctx_for(shape, max_batch=3, max_tokens=0, max_seq=256)
    B, nq, d, cap = 3, 8, 128, 1024
    positions = [100, -1, 600]
    pos = torch.tensor(positions, dtype=torch.int32)
    q = _randn((B, nq, d), 1.0, torch.bfloat16, 55)
    k = synth.cache_values((1, B, 8, cap, d), 55, torch.bfloat16, stream=0)
    v = synth.cache_values((1, B, 8, cap, d), 55, torch.bfloat16, stream=1)
    kv = binding.KVCache(shape, batch=B, capacity=cap, k=k.cuda(), v=v.cuda())
    out = torch.full((B, nq * d), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.op_attention_decode(q.cuda(), pos.cuda(), 0, kv, out)
    rc, flags = m.sync_status()
    assert rc == 5 and flags & binding.FLAG_POS_RANGE
    ref = O.gqa_attention(f64(q)[0], f64(k)[0, 0], f64(v)[0, 0], 101)
    assert_close(out[0].view(nq, d), ref, BF16_TOL, "in-range sequence beside flagged ones")
    assert torch.all(out[1] == 0)


def test_attention_decode_f32():
    shape = synth.TINY
    m, _ = ctx_for(shape, max_batch=3, max_tokens=16, max_seq=64, n_layers=2)
    B, nq, nkv, d = 3, 4, 2, 64
    pos = torch.tensor([0, 17, 40], dtype=torch.int32)
    q = _randn((B, nq, d), 1.0, torch.float32, 54)
    k = synth.cache_values((2, B, nkv, 48, d), 54, torch.float32, stream=0)
    v = synth.cache_values((2, B, nkv, 48, d), 54, torch.float32, stream=1)
    kv = binding.KVCache(shape, batch=B, capacity=48, k=k.cuda(), v=v.cuda())
    out = torch.empty(B, nq * d, device="cuda")
    m.op_attention_decode(q.cuda(), pos.cuda(), 1, kv, out)
    m.sync()
    for b in range(B):
        n = int(pos[b]) + 1
        ref = O.gqa_attention(f64(q)[b], f64(k)[1, b], f64(v)[1, b], n)
        assert_close(out[b].view(nq, d), ref, F32_TOL, "decode attention f32")


# --------------------------------------------------------------------------- prefill attention
@pytest.mark.parametrize("T", [1, 17, 64, 130])
@pytest.mark.parametrize("nq,nkv", [(8, 8), (16, 2)])
def test_attention_prefill_bf16(T, nq, nkv):
    shape = L7.with_(n_q_heads=nq, n_kv_heads=nkv)
    B, d = 2, 128
    m, _ = ctx_for(shape, max_batch=B, max_tokens=B * T, max_seq=256)
    q = _randn((B * T, nq, d), 1.0, torch.bfloat16, 61)
    k = _randn((B * T, nkv, d), 1.0, torch.bfloat16, 62)
    v = _randn((B * T, nkv, d), 1.0, torch.bfloat16, 63)
    out = torch.empty(B * T, nq * d, dtype=torch.bfloat16, device="cuda")
    m.op_attention_prefill(q.cuda(), k.cuda(), v.cuda(), B, T, out)
    m.sync()
    qf, kf, vf = f64(q), f64(k), f64(v)
    for b in range(B):
        K = kf[b * T:(b + 1) * T].transpose(1, 0, 2)
        V = vf[b * T:(b + 1) * T].transpose(1, 0, 2)
        ref = np.stack([O.gqa_attention(qf[b * T + t], K, V, t + 1) for t in range(T)])
        assert_close(out[b * T:(b + 1) * T].view(T, nq, d), ref, BF16_TOL, "prefill b=%d" % b)


# --------------------------------------------------------------------------- embedding, argmax
def test_embed_and_argmax():
    shape = synth.LLAMA2_7B.with_(n_layers=1, vocab=1000)
    m, w = ctx_for(shape, max_batch=8, max_tokens=8, max_seq=64, embed=True)
    toks = torch.tensor([0, 999, 5, 5, 123], dtype=torch.int32)
    out = torch.empty(5, shape.hidden, device="cuda")
    m.op_embed(toks.cuda(), out)
    m.sync()
    np.testing.assert_array_equal(f64(out), O.embed(f64(w["embed"]), toks.numpy()))
    logits = _randn((4, 32000), 1.0, torch.float32, 71)
    logits[1, 7] = logits[1, 31000] = 50.0       # tie: lowest index wins
    logits[2] = 0.0                              # all equal
    logits[3, 31999] = 60.0                      # last column
    ids = torch.empty(4, dtype=torch.int32, device="cuda")
    m.op_argmax(logits.cuda(), ids)
    m.sync()
    np.testing.assert_array_equal(ids.cpu().numpy(), O.greedy(f64(logits)))
