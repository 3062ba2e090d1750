"""The allocation-free decode attention entry point.

Some callers cannot allocate device memory when they run attention (a host
framework that owns all device memory through its own pool, a plugin inside
one, or code under CUDA-graph stream capture). For them
llama_attention_decode_noalloc keeps its key-split partial sums in a fixed
array inside the library instead of a caller workspace. This file is named so
that pytest collects it last; it passes alone in a fresh process and after the
other tests.
"""
import ctypes

import pytest
import torch

import numpy as np

from _common import BF16_TOL, assert_close, f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu


def _call_noalloc(cfg, q, pos, B, kv, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return binding.lib().llama_attention_decode_noalloc(
        ctypes.byref(cfg), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(pos.data_ptr()), B, 0,
        ctypes.byref(kv.struct()), ctypes.c_void_p(out.data_ptr()), stream)


def _oracle_attention(q, k, v, positions, table=None, page=16):
    """fp64 oracle of decode attention (§2.3, §1.5) over the cache as stored."""
    qs, kc, vc = f64(q), f64(k)[0], f64(v)[0]
    out = []
    for b, p in enumerate(positions):
        if table is None:
            K, V = kc[b], vc[b]
        else:
            K = O.gather_paged(kc, table[b], p + 1, page)
            V = O.gather_paged(vc, table[b], p + 1, page)
        out.append(O.gqa_attention(qs[b], K, V, p + 1).reshape(-1))
    return np.stack(out)


def _case(paged, positions):
    # 64 query / 8 K/V heads, few sequences, long context: the key range is
    # split, so the partial sums really go through the library's fixed array
    shape = synth.LLAMA2_70B.with_(n_layers=1)
    B, nq, nkv, d, cap = len(positions), 64, 8, 128, 4112
    g = torch.Generator().manual_seed(91)
    q = torch.randn(B, nq, d, generator=g).to(torch.bfloat16).cuda()
    pos = torch.tensor(positions, dtype=torch.int32).cuda()
    table = None
    if paged:
        n_pages = [(p + 1 + 15) // 16 for p in positions]
        table, total = synth.page_table(n_pages, max(n_pages), 91)
        k = synth.cache_values((1, total, nkv, 16, d), 91, torch.bfloat16, stream=0).cuda()
        v = synth.cache_values((1, total, nkv, 16, d), 91, torch.bfloat16, stream=1).cuda()
        kv = binding.KVCache(shape, n_pages=total, page_size=16, page_table=table.cuda(), k=k, v=v)
        max_seq = max(n_pages) * 16
        table = table.numpy()
    else:
        k = synth.cache_values((1, B, nkv, cap, d), 91, torch.bfloat16, stream=0).cuda()
        v = synth.cache_values((1, B, nkv, cap, d), 91, torch.bfloat16, stream=1).cuda()
        kv = binding.KVCache(shape, batch=B, capacity=cap, k=k, v=v)
        max_seq = cap
    ref = _oracle_attention(q.cpu(), k.cpu(), v.cpu(), positions, table)
    return shape, q, pos, kv, max_seq, ref


@pytest.mark.parametrize("paged", [False, True])
def test_noalloc_attention_matches_workspace_entry_point(paged):
    need_gpu()
    positions = [4096, 3000, 17, 1]
    B, nq, d = len(positions), 64, 128
    shape, q, pos, kv, max_seq, oracle = _case(paged, positions)
    model = binding.Model(shape, to_dev({"layers": [synth.layer_weights(shape, 91, 0, std=0.01)]}),
                          max_batch=B, max_tokens=0, max_seq=max_seq, has_embed_head=False)
    ref = torch.empty(B, nq * d, dtype=torch.bfloat16, device="cuda")
    model.op_attention_decode(q, pos, 0, kv, ref)
    model.sync()
    cfg = binding.make_config(shape, B, 0, max_seq, has_embed_head=False)
    for _ in range(2):  # the fixed array keeps the previous call's contents
        out = torch.full((B, nq * d), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(cfg, q, pos, B, kv, out) == 0
        torch.cuda.synchronize()
        assert_close(out, ref.double().cpu().numpy(), BF16_TOL, "allocation-free decode attention")
        assert_close(out, oracle, BF16_TOL, "allocation-free decode attention vs oracle")
    assert_close(ref, oracle, BF16_TOL, "workspace decode attention vs oracle")


def test_noalloc_covers_the_cache_beyond_max_seq():
    # positions between cfg->max_seq and the cache capacity: the fixed array
    # is planned for every cache slot, so the result still matches the oracle
    need_gpu()
    positions = [4096, 3000, 17, 1]
    B, nq, d = len(positions), 64, 128
    shape, q, pos, kv, _, oracle = _case(False, positions)
    cfg = binding.make_config(shape, B, 0, 1024, has_embed_head=False)
    out = torch.full((B, nq * d), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(cfg, q, pos, B, kv, out) == 0
    torch.cuda.synchronize()
    assert_close(out, oracle, BF16_TOL, "allocation-free decode attention, positions past max_seq")


def test_noalloc_rejects_scratch_beyond_its_limit():
    need_gpu()
    # 128 query heads x 64 sequences x several key splits needs more than the
    # fixed array holds: refused with OUT_OF_RANGE before anything is enqueued
    shape = synth.LLAMA2_70B.with_(n_layers=1, n_q_heads=128)
    B, cap = 64, 4112
    cfg = binding.make_config(shape, B, 0, cap, has_embed_head=False)
    q = torch.zeros(B, 128, 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.full((B,), 4096, dtype=torch.int32, device="cuda")
    kv = binding.KVCache(shape, batch=B, capacity=cap)  # full-size buffers, never read here
    out = torch.zeros(B, 128 * 128, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(cfg, q, pos, B, kv, out) == 3
