"""Continuous-batching extend step (llama_extend / llama_extend_hidden) against
the oracle's layer_extend / Model.extend: packed rows of several sequences,
each a whole prompt, a piece of a prompt after cached positions, or a single
decode token, in one call; contiguous and paged caches; MHA and GQA."""
import math

import numpy as np
import pytest
import torch

from _common import BF16_TOL, assert_close, f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu

L7 = synth.LLAMA2_7B.with_(n_layers=1)


def _rows(starts, counts):
    seq = np.concatenate([np.full(n, b) for b, n in enumerate(counts)]).astype(np.int64)
    pos = np.concatenate([np.arange(s, s + n) for s, n in zip(starts, counts)]).astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return seq, pos, cu


def _layer_case(shape, starts, counts, seed, page_size=0, n_kv_variant=None):
    need_gpu()
    lw = synth.layer_weights(shape, seed, 0, std=0.02)
    if n_kv_variant:
        lw = synth.gqa_variant(lw, shape, n_kv_variant)
        shape = shape.with_(n_kv_heads=n_kv_variant)
    B, nkv, d, H = len(starts), shape.n_kv_heads, shape.head_dim, shape.hidden
    seq, pos, cu = _rows(starts, counts)
    R = len(seq)
    ends = [s + n for s, n in zip(starts, counts)]
    cap = (max(ends) + 15) // 16 * 16
    # logical cache: positions below start hold N(0, 1) values, the rest zeros
    Kl = f64(synth.cache_values((B, nkv, cap, d), seed, torch.bfloat16, stream=0))
    Vl = f64(synth.cache_values((B, nkv, cap, d), seed, torch.bfloat16, stream=1))
    for b, s in enumerate(starts):
        Kl[b, :, s:] = 0
        Vl[b, :, s:] = 0
    if page_size == 0:
        kv = binding.KVCache(shape, batch=B, capacity=cap,
                             k=torch.from_numpy(Kl[None]).to(torch.bfloat16).cuda(),
                             v=torch.from_numpy(Vl[None]).to(torch.bfloat16).cuda())
        table = None
    else:
        n_pages = [math.ceil(e / page_size) for e in ends]
        table, total = synth.page_table(n_pages, max(n_pages), seed)
        t = table.numpy()
        Kp = np.zeros((total, nkv, page_size, d))
        Vp = np.zeros_like(Kp)
        for b in range(B):
            for m in range(starts[b]):
                Kp[t[b, m // page_size], :, m % page_size] = Kl[b, :, m]
                Vp[t[b, m // page_size], :, m % page_size] = Vl[b, :, m]
        kv = binding.KVCache(shape, n_pages=total, page_size=page_size, page_table=table.cuda(),
                             k=torch.from_numpy(Kp[None]).to(torch.bfloat16).cuda(),
                             v=torch.from_numpy(Vp[None]).to(torch.bfloat16).cuda())
    x = synth.hidden_input(R, H, seed)
    m = binding.Model(shape, to_dev({"layers": [lw]}), max_batch=max(B, 8), max_tokens=R,
                      max_seq=cap, has_embed_head=False)
    h = x.cuda()
    cu_d = torch.from_numpy(cu).cuda()
    st_d = torch.tensor(starts, dtype=torch.int32).cuda()
    m.extend_hidden(h, cu_d, st_d, kv, max_rows=max(counts))
    m.sync()
    lw64 = {k: f64(v) for k, v in lw.items()}
    ref = O.layer_extend(f64(x), lw64, shape, Kl, Vl, seq, pos)
    assert_close(h, ref, BF16_TOL, "extend layer output")
    # the appended keys landed in their slots
    if page_size == 0:
        got_k = f64(kv.k)[0][seq, :, pos]
    else:
        t = table.numpy()
        got_k = f64(kv.k)[0][t[seq, pos // page_size], :, pos % page_size]
    assert_close(got_k, Kl[seq, :, pos], BF16_TOL, "appended K")


# a fresh prompt spanning three query tiles, a decode token, a 64-row piece
# after 37 cached positions, a ragged piece after 300
STARTS, COUNTS = [0, 100, 37, 300], [130, 1, 64, 17]


@pytest.mark.parametrize("page_size", [0, 16, 64])
def test_extend_layer_mixed_batch_7b(page_size):
    _layer_case(L7, STARTS, COUNTS, 2001, page_size)


def test_extend_layer_gqa_paged():
    _layer_case(L7, [5, 0, 200], [60, 70, 1], 2002, page_size=16, n_kv_variant=8)


def test_extend_layer_decode_only_and_single_prompt():
    _layer_case(L7, [10, 20, 30], [1, 1, 1], 2003)
    _layer_case(L7, [0], [200], 2004)


def _small():
    return synth.Shape(2, 256, 4, 2, 128, 512, 512, dtype="bf16")


def test_extend_full_model_matches_oracle_and_prefill():
    need_gpu()
    shape = _small()
    w = synth.model_weights(shape, 2005)
    toks = synth.token_ids(3, 48, shape.vocab, 2005).numpy()
    cap = 48
    m = binding.Model(shape, to_dev(w), max_batch=4, max_tokens=128, max_seq=cap)
    kv = binding.KVCache(shape, batch=3, capacity=cap)
    ref = O.Model(shape, w, 3, cap)
    V = shape.vocab

    def step(starts, counts):
        seq, pos, cu = _rows(starts, counts)
        tk = np.concatenate([toks[b, s:s + n] for b, (s, n) in enumerate(zip(starts, counts))])
        lg = torch.empty(len(starts), V, device="cuda")
        ids = torch.empty(len(starts), dtype=torch.int32, device="cuda")
        m.extend(torch.from_numpy(tk).int().cuda(), torch.from_numpy(cu).cuda(),
                 torch.tensor(starts, dtype=torch.int32).cuda(), kv, lg, ids,
                 max_rows=max(counts))
        m.sync()
        want = ref.extend(tk, seq, pos)[cu[1:] - 1]
        assert_close(lg, want, BF16_TOL, "extend logits %s %s" % (starts, counts))
        np.testing.assert_array_equal(ids.cpu().numpy(), O.greedy(f64(lg)))
        return lg

    step([0, 0, 0], [25, 9, 40])          # ragged prompts
    step([25, 9, 40], [15, 1, 1])         # the rest of prompt 0 with two decode tokens
    last = step([40, 10, 41], [1, 20, 1])  # decode, a prompt piece, decode
    # the same three sequences through plain prefill give the same last-row logits
    kv2 = binding.KVCache(shape, batch=1, capacity=cap)
    lg2 = torch.empty(1, V, device="cuda")
    m.prefill(torch.from_numpy(toks[1:2, :30]).int().cuda(), kv2, lg2)
    m.sync()
    assert_close(last[1:2], f64(lg2), BF16_TOL, "piecewise prompt vs one-shot prefill")


def test_extend_host_checks():
    need_gpu()
    shape = _small()
    w = synth.model_weights(shape, 2006)
    m = binding.Model(shape, to_dev(w), max_batch=2, max_tokens=16, max_seq=32)
    kv = binding.KVCache(shape, batch=2, capacity=32)
    lg = torch.empty(2, shape.vocab, device="cuda")
    cu = torch.tensor([0, 3, 5], dtype=torch.int32, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    tk = torch.zeros(5, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.LlamaError, match="INVALID_ARG"):
        m.extend(tk, cu, st, kv, lg, max_rows=6)     # max_rows above n_rows
    with pytest.raises(binding.LlamaError, match="OUT_OF_RANGE"):
        m.extend(torch.zeros(17, dtype=torch.int32, device="cuda"), cu, st, kv, lg, max_rows=3)
    st[1] = 40  # position past the cache: flagged on the device
    m.extend(tk, cu, st, kv, lg, max_rows=3)
    rc, flags = m.sync_status()
    assert rc == 5 and flags & binding.FLAG_POS_RANGE


def test_prefill_fused_qkv_epilogue_writes_the_cache_of_the_separate_pass():
    # A 7B layer over 2 x 320 prompt rows. Prefill rotates Q/K and appends
    # K/V in the token-major GEMM's epilogue; an extend step of the same
    # whole prompts stores the fp32 Q/K/V sums and runs the separate RoPE
    # kernel. Both round the same sums with the same expressions, so the
    # cache (layer 0: no attention output in between) agrees bit for bit.
    # (Extend steps take bf16 caches only; the fused E4M3 append is checked
    # against the oracle in the FP8 tests.)
    need_gpu()
    shape, B, T, seed = L7, 2, 320, 2104
    lw = synth.layer_weights(shape, seed, 0, std=0.02)
    x = synth.hidden_input(B * T, shape.hidden, seed)
    m = binding.Model(shape, to_dev({"layers": [lw]}), max_batch=B, max_tokens=B * T,
                      max_seq=T, has_embed_head=False)
    kv1 = binding.KVCache(shape, batch=B, capacity=T)
    kv2 = binding.KVCache(shape, batch=B, capacity=T)
    h1 = x.cuda()
    m.prefill_hidden(h1, B, T, kv1)
    h2 = x.cuda()
    cu = torch.tensor([0, T, 2 * T], dtype=torch.int32, device="cuda")
    m.extend_hidden(h2, cu, torch.zeros(B, dtype=torch.int32, device="cuda"), kv2)
    m.sync()
    assert torch.equal(kv1.k, kv2.k) and torch.equal(kv1.v, kv2.v)
    assert_close(h1, f64(h2), BF16_TOL, "prefill and extend of the same prompts")
