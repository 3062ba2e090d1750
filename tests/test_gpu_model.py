"""Whole-model and whole-layer parity with the CPU oracle on the pages'
workloads: the tiny fp32 model (greedy ids bit-exact, logits within 1e-4),
single 7B- and 70B-shaped layers (decode and prefill) and ragged paged decode
(MHA and GQA), plus device-side range checks and the bounded-wait timeout."""
import math
import time

import numpy as np
import pytest
import torch

from _common import BF16_TOL, F32_TOL, assert_close, f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu


# --------------------------------------------------------------------------- tiny fp32 model
def test_tiny_fp32_greedy_generation():
    """Prefill 16 random ids, then 8 greedy decode steps feeding each choice
    back: 9 ids bit-exact and 9 logit rows within 1e-4 of the oracle."""
    need_gpu()
    shape = synth.TINY
    seed = 1000
    w = synth.model_weights(shape, seed)
    prompt = synth.token_ids(1, 16, shape.vocab, seed)
    steps, cap = 8, 32
    ref_ids, ref_logits = O.generate_greedy(O.Model(shape, w, 1, cap), prompt.numpy(), steps)
    # each greedy choice must be clear of the runner-up by more than the tolerance
    top2 = np.sort(ref_logits, -1)[..., -2:]
    assert np.all(top2[..., 1] - top2[..., 0] > 1e-4), "oracle margin too small for an exact id check"

    m = binding.Model(shape, to_dev(w), max_batch=1, max_tokens=16, max_seq=cap)
    kv = binding.KVCache(shape, batch=1, capacity=cap)
    logits = torch.empty(1, shape.vocab, device="cuda")
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    got_ids, got_logits = [], []
    m.prefill(prompt.cuda(), kv, logits, ids)
    got_logits.append(logits.clone())
    got_ids.append(ids.clone())
    for s in range(steps):
        pos = torch.full((1,), 16 + s, dtype=torch.int32, device="cuda")
        m.decode_step(ids.clone(), pos, kv, logits, ids)
        got_logits.append(logits.clone())
        got_ids.append(ids.clone())
    m.sync()
    gi = torch.stack(got_ids, 1).cpu().numpy()
    gl = torch.stack(got_logits, 1)
    np.testing.assert_array_equal(gi, ref_ids)
    assert_close(gl, ref_logits, F32_TOL, "tiny logits")


# --------------------------------------------------------------------------- single layers
def _layer_decode_case(shape, std, B, S, seed, paged_lengths=None, n_kv_variant=None):
    need_gpu()
    lw = synth.layer_weights(shape, seed, 0, std=std)
    if n_kv_variant:
        lw = synth.gqa_variant(lw, shape, n_kv_variant)
        shape = shape.with_(n_kv_heads=n_kv_variant)
    nkv, d = shape.n_kv_heads, shape.head_dim
    x = synth.hidden_input(B, shape.hidden, seed)
    if paged_lengths is None:
        lengths = [S] * B
        cap = (S + 1 + 15) // 16 * 16
        K = synth.cache_values((1, B, nkv, cap, d), seed, torch.bfloat16, stream=0)
        V = synth.cache_values((1, B, nkv, cap, d), seed, torch.bfloat16, stream=1)
        K[:, :, :, S:] = 0
        V[:, :, :, S:] = 0
        kv = binding.KVCache(shape, batch=B, capacity=cap, k=K.cuda(), v=V.cuda())
        max_seq = cap
    else:
        lengths = [int(v) for v in paged_lengths]
        n_pages = [math.ceil((L + 1) / 16) for L in lengths]
        table, total = synth.page_table(n_pages, max(n_pages), seed)
        K = synth.cache_values((1, total, nkv, 16, d), seed, torch.bfloat16, stream=0)
        V = synth.cache_values((1, total, nkv, 16, d), seed, torch.bfloat16, stream=1)
        kv = binding.KVCache(shape, n_pages=total, page_size=16, page_table=table.cuda(),
                             k=K.cuda(), v=V.cuda())
        max_seq = max(n_pages) * 16
    pos = torch.tensor(lengths, dtype=torch.int32)
    m = binding.Model(shape, to_dev({"layers": [lw]}), max_batch=B, max_tokens=0, max_seq=max_seq,
                      has_embed_head=False)
    h = x.cuda()
    m.decode_hidden(h, pos.cuda(), kv)
    m.sync()
    lw64 = {k: f64(v) for k, v in lw.items()}
    if paged_lengths is None:
        Kc, Vc = f64(K)[0], f64(V)[0]
        ref = O.layer_decode(f64(x), lw64, shape, Kc, Vc, pos.numpy())
        newk = f64(kv.k)[0][np.arange(B), :, pos.numpy()]
        refk = Kc[np.arange(B), :, pos.numpy()]
    else:
        Kp, Vp = f64(K)[0], f64(V)[0]
        ref = O.layer_decode_paged(f64(x), lw64, shape, Kp, Vp, table.numpy(), pos.numpy(), 16)
        t = table.numpy()
        pages = t[np.arange(B), pos.numpy() // 16]
        newk = f64(kv.k)[0][pages, :, pos.numpy() % 16]
        refk = Kp[pages, :, pos.numpy() % 16]
    assert_close(newk, refk, BF16_TOL, "appended K")
    return assert_close(h, ref, BF16_TOL, "layer output")


def test_layer_7b_decode_bs32_ctx1024():
    _layer_decode_case(synth.LLAMA2_7B.with_(n_layers=1), 0.02, 32, 1024, 1001)


def test_layer_70b_decode_bs32_ctx4096():
    _layer_decode_case(synth.LLAMA2_70B.with_(n_layers=1), 0.01, 32, 4096, 1002)


@pytest.mark.parametrize("n_kv", [None, 8])
def test_ragged_paged_decode_7b_layer(n_kv):
    lengths = synth.ragged_lengths(64, 128, 4096, 1004)
    _layer_decode_case(synth.LLAMA2_7B.with_(n_layers=1), 0.02, 64, None, 1004,
                       paged_lengths=lengths.tolist(), n_kv_variant=n_kv)


def test_layer_7b_decode_bs160_two_activation_tiles():
    # 160 sequences span two 128-row activation tiles (the last one ragged), so
    # the Q/K/V projection takes its unsplit path with RoPE in the epilogue
    _layer_decode_case(synth.LLAMA2_7B.with_(n_layers=1), 0.02, 160, 64, 1005)


def test_ragged_paged_gqa_decode_bs160():
    lengths = synth.ragged_lengths(160, 1, 300, 1006)
    _layer_decode_case(synth.LLAMA2_7B.with_(n_layers=1), 0.02, 160, None, 1006,
                       paged_lengths=lengths.tolist(), n_kv_variant=8)


def test_layer_70b_prefill_4096_sampled_rows():
    need_gpu()
    shape = synth.LLAMA2_70B.with_(n_layers=1)
    seed, T = 1002, 4096
    lw = synth.layer_weights(shape, seed, 0, std=0.01)
    x = synth.hidden_input(T, shape.hidden, seed)
    kv = binding.KVCache(shape, batch=1, capacity=T)
    m = binding.Model(shape, to_dev({"layers": [lw]}), max_batch=1, max_tokens=T, max_seq=T,
                      has_embed_head=False)
    h = x.cuda()
    m.prefill_hidden(h, 1, T, kv)
    m.sync()
    rows = [0, 1, 63, 64, 65, 1000, 2047, 4094, 4095]
    K = np.zeros((1, shape.n_kv_heads, T, shape.head_dim))
    V = np.zeros_like(K)
    lw64 = {k: f64(v) for k, v in lw.items()}
    ref = O.layer_prefill(f64(x)[None], lw64, shape, K, V, rows=rows)[0]
    assert_close(h[rows], ref, BF16_TOL, "prefill rows")
    # the whole cache was written: compare a sample of slots
    for t in (0, 777, 4095):
        assert_close(kv.k[0, 0, :, t], K[0, :, t], BF16_TOL, "cached K row %d" % t)
        assert_close(kv.v[0, 0, :, t], V[0, :, t], BF16_TOL, "cached V row %d" % t)


# --------------------------------------------------------------------------- consistency on the GPU
def _small_bf16():
    return synth.Shape(2, 256, 4, 2, 128, 512, 512, dtype="bf16")


def test_decode_continues_prefill_and_paged_matches_contiguous():
    need_gpu()
    shape = _small_bf16()
    B, T, cap = 3, 40, 64
    w = synth.model_weights(shape, 9)
    toks = synth.token_ids(B, T + 1, shape.vocab, 9)
    wd = to_dev(w)
    m = binding.Model(shape, wd, max_batch=B, max_tokens=B * (T + 1), max_seq=cap)
    # contiguous: prefill T, decode token T
    kvc = binding.KVCache(shape, batch=B, capacity=cap)
    lg_c = torch.empty(B, shape.vocab, device="cuda")
    m.prefill(toks[:, :T].contiguous().cuda(), kvc, lg_c)
    pos = torch.full((B,), T, dtype=torch.int32, device="cuda")
    m.decode_step(toks[:, T].contiguous().cuda(), pos, kvc, lg_c)
    # paged, random page permutation
    n_pages = [cap // 16] * B
    table, total = synth.page_table(n_pages, cap // 16, 9)
    kvp = binding.KVCache(shape, n_pages=total, page_size=16, page_table=table.cuda())
    lg_p = torch.empty(B, shape.vocab, device="cuda")
    m.prefill(toks[:, :T].contiguous().cuda(), kvp, lg_p)
    m.decode_step(toks[:, T].contiguous().cuda(), pos, kvp, lg_p)
    # one prefill of all T+1 tokens
    kvf = binding.KVCache(shape, batch=B, capacity=cap)
    lg_f = torch.empty(B, shape.vocab, device="cuda")
    m.prefill(toks.contiguous().cuda(), kvf, lg_f)
    m.sync()
    ref = O.Model(shape, w, B, cap).prefill(toks.numpy())[:, -1]
    assert_close(lg_c, ref, BF16_TOL, "decode after prefill")
    assert_close(lg_p, ref, BF16_TOL, "paged decode after prefill")
    assert_close(lg_f, ref, BF16_TOL, "prefill of T+1")
    np.testing.assert_array_equal(lg_p.cpu().numpy(), lg_c.cpu().numpy())  # same arithmetic


def test_host_buffer_step_matches_device_step():
    need_gpu()
    shape = _small_bf16()
    B, T, cap = 2, 8, 16
    w = to_dev(synth.model_weights(shape, 10))
    m = binding.Model(shape, w, max_batch=B, max_tokens=B * T, max_seq=cap)
    toks = synth.token_ids(B, T + 1, shape.vocab, 10)
    kv1 = binding.KVCache(shape, batch=B, capacity=cap)
    kv2 = binding.KVCache(shape, batch=B, capacity=cap)
    lg = torch.empty(B, shape.vocab, device="cuda")
    m.prefill(toks[:, :T].contiguous().cuda(), kv1, lg)
    m.prefill(toks[:, :T].contiguous().cuda(), kv2, lg)
    pos = torch.full((B,), T, dtype=torch.int32)
    ids_d = torch.empty(B, dtype=torch.int32, device="cuda")
    m.decode_step(toks[:, T].contiguous().cuda(), pos.cuda(), kv1, lg, ids_d)
    m.sync()
    lg_h = torch.empty(B, shape.vocab).pin_memory()
    ids_h = torch.empty(B, dtype=torch.int32).pin_memory()
    m.decode_step_host(toks[:, T].contiguous().pin_memory(), pos.pin_memory(), kv2, lg_h, ids_h)
    np.testing.assert_array_equal(lg_h.numpy(), lg.cpu().numpy())
    np.testing.assert_array_equal(ids_h.numpy(), ids_d.cpu().numpy())


# --------------------------------------------------------------------------- device-side checks
def test_device_range_checks_flag_and_skip():
    need_gpu()
    shape = _small_bf16()
    B, cap = 2, 32
    m = binding.Model(shape, to_dev(synth.model_weights(shape, 11)), max_batch=B, max_tokens=B * 4,
                      max_seq=64)
    kv = binding.KVCache(shape, batch=B, capacity=cap)
    lg = torch.empty(B, shape.vocab, device="cuda")
    # token id past the vocabulary
    m.decode_step(torch.tensor([1, shape.vocab + 5], dtype=torch.int32, device="cuda"),
                  torch.tensor([0, 0], dtype=torch.int32, device="cuda"), kv, lg)
    rc, flags = m.sync_status()
    assert rc == 5 and flags & binding.FLAG_TOKEN_RANGE
    # position past the cache: nothing written
    before = kv.k.clone()
    m.decode_step(torch.tensor([1, 2], dtype=torch.int32, device="cuda"),
                  torch.tensor([1, cap + 3], dtype=torch.int32, device="cuda"), kv, lg)
    rc, flags = m.sync_status()
    assert rc == 5 and flags & binding.FLAG_POS_RANGE
    assert torch.equal(kv.k[:, 1], before[:, 1])
    # page id outside the pool
    table = torch.tensor([[0, 1], [7, 2]], dtype=torch.int32, device="cuda")
    kvp = binding.KVCache(shape, n_pages=3, page_size=16, page_table=table)
    m.decode_step(torch.tensor([1, 2], dtype=torch.int32, device="cuda"),
                  torch.tensor([3, 3], dtype=torch.int32, device="cuda"), kvp, lg)
    rc, flags = m.sync_status()
    assert rc == 5 and flags & binding.FLAG_PAGE_RANGE
    # the context still works and the word was cleared
    m.decode_step(torch.tensor([1, 2], dtype=torch.int32, device="cuda"),
                  torch.tensor([0, 0], dtype=torch.int32, device="cuda"), kv, lg)
    assert m.sync_status() == (0, 0)


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    # a device wait on a barrier that nothing completes: the kernel flags the
    # timeout and returns; the host reads the flag and the next step is correct
    need_gpu()
    shape = _small_bf16()
    B, T, cap = 2, 6, 32
    w = synth.model_weights(shape, 12)
    m = binding.Model(shape, to_dev(w), max_batch=B, max_tokens=B * T, max_seq=cap)
    with pytest.raises(binding.LlamaError, match="INVALID_ARG"):
        m.check_wait_timeout(0)
    with pytest.raises(binding.LlamaError, match="INVALID_ARG"):
        m.check_wait_timeout(2_000_000)
    t0 = time.perf_counter()
    m.check_wait_timeout(20_000)  # 20 ms
    rc, flags = m.sync_status()
    took = time.perf_counter() - t0
    assert rc == 5 and flags == binding.FLAG_WAIT_TIMEOUT
    assert 0.015 < took < 5.0
    toks = synth.token_ids(B, T, shape.vocab, 12)
    kv = binding.KVCache(shape, batch=B, capacity=cap)
    lg = torch.empty(B, shape.vocab, device="cuda")
    m.prefill(toks.cuda(), kv, lg)
    assert m.sync_status() == (0, 0)
    want = O.Model(shape, w, B, cap).prefill(toks.numpy())[:, -1]
    assert_close(lg, want, BF16_TOL, "prefill after a timed-out wait")


def test_host_checks_reject_bad_sizes():
    need_gpu()
    shape = _small_bf16()
    m = binding.Model(shape, to_dev(synth.model_weights(shape, 12)), max_batch=2, max_tokens=8,
                      max_seq=32)
    kv = binding.KVCache(shape, batch=2, capacity=32)
    lg = torch.empty(3, shape.vocab, device="cuda")
    with pytest.raises(binding.LlamaError) as e:
        m.decode_step(torch.zeros(3, dtype=torch.int32, device="cuda"),
                      torch.zeros(3, dtype=torch.int32, device="cuda"), kv, lg)
    assert e.value.rc == 3
    with pytest.raises(binding.LlamaError) as e:
        m.prefill(torch.zeros(2, 5, dtype=torch.int32, device="cuda"), kv, lg)
    assert e.value.rc == 3
    bad = binding.KVCache(shape, batch=1, capacity=32)
    with pytest.raises(binding.LlamaError) as e:
        m.decode_step(torch.zeros(2, dtype=torch.int32, device="cuda"),
                      torch.zeros(2, dtype=torch.int32, device="cuda"), bad, lg)
    assert e.value.rc == 1
    # empty inputs: no sequences, or prompts of no tokens
    none = torch.zeros(0, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.LlamaError) as e:
        m.decode_step(none, none, kv, lg)
    assert e.value.rc == 1
    with pytest.raises(binding.LlamaError) as e:
        m.prefill(torch.zeros(2, 0, dtype=torch.int32, device="cuda"), kv, lg)
    assert e.value.rc == 1


# --------------------------------------------------------------------------- CUDA graph replay
def test_graph_replay_matches_direct_steps_and_runs_the_greedy_loop():
    need_gpu()
    shape = _small_bf16()
    B, T, cap, steps = 3, 12, 48, 6
    w_cpu = synth.model_weights(shape, 13)
    w = to_dev(w_cpu)
    stream = torch.cuda.Stream()
    m = binding.Model(shape, w, max_batch=B, max_tokens=B * T, max_seq=cap, stream=stream)
    toks = synth.token_ids(B, T, shape.vocab, 13).cuda()
    with torch.cuda.stream(stream):
        # direct greedy loop
        kv_d = binding.KVCache(shape, batch=B, capacity=cap)
        lg = torch.empty(B, shape.vocab, device="cuda")
        ids = torch.empty(B, dtype=torch.int32, device="cuda")
        m.prefill(toks, kv_d, lg, ids)
        direct_ids, direct_lg = [ids.clone()], [lg.clone()]
        for s in range(steps):
            pos = torch.full((B,), T + s, dtype=torch.int32, device="cuda")
            m.decode_step(ids.clone(), pos, kv_d, lg, ids)
            direct_ids.append(ids.clone())
            direct_lg.append(lg.clone())
        # the same loop as graph replays: tokens are the previous step's choices
        kv_g = binding.KVCache(shape, batch=B, capacity=cap)
        lg_g = torch.empty(B, shape.vocab, device="cuda")
        ids_g = torch.empty(B, dtype=torch.int32, device="cuda")
        m.prefill(toks, kv_g, lg_g, ids_g)
        pos_g = torch.full((B,), T, dtype=torch.int32, device="cuda")
        m.capture_decode(ids_g, pos_g, kv_g, lg_g, ids_g, advance=True)
        graph_ids, graph_lg = [ids_g.clone()], [lg_g.clone()]
        for s in range(steps):
            m.graph_launch()
            graph_ids.append(ids_g.clone())
            graph_lg.append(lg_g.clone())
    m.sync()
    for a, b in zip(direct_ids, graph_ids):
        np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())
    for a, b in zip(direct_lg, graph_lg):
        np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())
    assert int(pos_g[0]) == T + steps
    # the replayed loop against the oracle, teacher-forced with the GPU's ids:
    # one fp64 prefill of the prompt and the chosen ids gives every step's row
    # (decoding a token equals the prefill row at its position, §2.4)
    gi = torch.stack(graph_ids, 1).cpu().numpy()
    seq = np.concatenate([toks.cpu().numpy(), gi[:, :steps]], axis=1)
    ref = O.Model(shape, w_cpu, B, cap).prefill(seq)[:, T - 1:]
    got = torch.stack(graph_lg, 1)
    assert_close(got, ref, BF16_TOL, "graph replay logits vs oracle")
    np.testing.assert_array_equal(gi, O.greedy(f64(got)))
    top2 = np.sort(ref, -1)[..., -2:]
    clear = top2[..., 1] - top2[..., 0] > BF16_TOL[0] + BF16_TOL[1] * np.abs(top2[..., 1])
    assert np.all(gi[clear] == O.greedy(ref)[clear])
