"""FP8 E4M3 projection weights with one scale per output row (llama_config
weight_dtype LLAMA_W_E4M3) against the oracle's quantize_rows_e4m3: the
device quantiser bit for bit, then the GEMMs that stream the E4M3 bytes and
convert them to bf16 in shared memory, through a 7B layer's decode step (K
split over a cluster, RoPE/append and RMSNorm epilogues), a 7B layer's
prefill (several activation tiles, the last one ragged) and a two-layer model
(norms fused across layers, bf16 embedding and LM head). The oracle quantises
the same bf16 weights itself and computes with code * scale in fp64."""
import numpy as np
import pytest
import torch

from _common import BF16_TOL, assert_close, f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = pytest.mark.gpu

L7 = synth.LLAMA2_7B.with_(n_layers=1)


def _oracle_layer(lw):
    """fp64 layer weights as the model uses them: projections quantised by the
    oracle (from the same bf16 values) and dequantised."""
    out = {k: f64(v) for k, v in lw.items()}
    for n in binding.PROJECTIONS:
        codes, s = O.quantize_rows_e4m3(f64(lw[n]).astype(np.float32))
        out[n] = O.dequantize_rows(codes, s)
    return out


def test_quantize_rows_matches_the_oracle_bit_for_bit():
    need_gpu()
    g = torch.Generator().manual_seed(71)
    w = torch.randn(300, 4096, generator=g) * 0.02
    w[7] = 0.0
    w[11] *= 500.0
    w[13] = torch.linspace(-3.0, 3.0, 4096)
    w = w.to(torch.bfloat16)
    codes, s = binding.quantize_rows_e4m3(w.cuda())
    torch.cuda.synchronize()
    want_codes, want_s = O.quantize_rows_e4m3(f64(w).astype(np.float32))
    np.testing.assert_array_equal(s.cpu().double().numpy(), want_s)
    np.testing.assert_array_equal(codes.cpu().view(torch.float8_e4m3fn).double().numpy(), want_codes)
    with pytest.raises(binding.LlamaError, match="INVALID_ARG"):
        binding.quantize_rows_e4m3(w[:, :40].cuda())  # rows of 40 bytes: not a 16-byte pitch


def test_layer_7b_decode_bs32_ctx1024_e4m3_weights():
    need_gpu()
    shape, B, S, seed = L7, 32, 1024, 1101
    lw = synth.layer_weights(shape, seed, 0, std=0.02)
    nkv, d = shape.n_kv_heads, shape.head_dim
    cap = S + 16
    K = synth.cache_values((1, B, nkv, cap, d), seed, torch.bfloat16, stream=0)
    V = synth.cache_values((1, B, nkv, cap, d), seed, torch.bfloat16, stream=1)
    K[:, :, :, S:] = 0
    V[:, :, :, S:] = 0
    kv = binding.KVCache(shape, batch=B, capacity=cap, k=K.cuda(), v=V.cuda())
    lwq = binding.quantize_layer_e4m3(to_dev(lw))
    m = binding.Model(shape, {"layers": [lwq]}, max_batch=B, max_tokens=0, max_seq=cap,
                      has_embed_head=False)
    assert m.cfg.weight_dtype == binding.W_E4M3
    x = synth.hidden_input(B, shape.hidden, seed)
    pos = torch.full((B,), S, dtype=torch.int32)
    h = x.cuda()
    m.decode_hidden(h, pos.cuda(), kv)
    m.sync()
    ref = O.layer_decode(f64(x), _oracle_layer(lw), shape, f64(K)[0], f64(V)[0], pos.numpy())
    assert_close(h, ref, BF16_TOL, "7B layer decode over E4M3 weights")


def test_layer_7b_prefill_e4m3_weights_ragged_tiles():
    need_gpu()
    shape, B, T, seed = L7, 2, 100, 1102  # 200 rows: a full and a ragged 128-row tile
    lw = synth.layer_weights(shape, seed, 0, std=0.02)
    x = synth.hidden_input(B * T, shape.hidden, seed)
    kv = binding.KVCache(shape, batch=B, capacity=T)
    m = binding.Model(shape, {"layers": [binding.quantize_layer_e4m3(to_dev(lw))]}, max_batch=B,
                      max_tokens=B * T, max_seq=T, has_embed_head=False)
    h = x.cuda()
    m.prefill_hidden(h, B, T, kv)
    m.sync()
    K = np.zeros((B, shape.n_kv_heads, T, shape.head_dim))
    Vc = np.zeros_like(K)
    ref = O.layer_prefill(f64(x).reshape(B, T, -1), _oracle_layer(lw), shape, K, Vc)
    assert_close(h.view(B, T, -1), ref, BF16_TOL, "7B layer prefill over E4M3 weights")
    assert_close(kv.k[0, 1, :, T - 1], K[1, :, T - 1], BF16_TOL, "cached K, last row")


def test_two_layer_model_prefill_and_greedy_decode_e4m3_weights():
    need_gpu()
    shape = synth.Shape(2, 256, 4, 2, 128, 512, 512, dtype="bf16")
    B, T, cap, seed = 2, 24, 32, 1103
    w = synth.model_weights(shape, seed)
    toks = synth.token_ids(B, T + 3, shape.vocab, seed)
    wd = to_dev(w)
    wd["layers"] = [binding.quantize_layer_e4m3(lw) for lw in wd["layers"]]
    m = binding.Model(shape, wd, max_batch=B, max_tokens=B * T, max_seq=cap)
    kv = binding.KVCache(shape, batch=B, capacity=cap)
    wo = dict(w)
    wo["layers"] = [_oracle_layer(lw) for lw in w["layers"]]
    ref = O.Model(shape, wo, B, cap)
    lg = torch.empty(B, shape.vocab, device="cuda")
    ids = torch.empty(B, dtype=torch.int32, device="cuda")
    m.prefill(toks[:, :T].contiguous().cuda(), kv, lg, ids)
    m.sync()
    assert_close(lg, ref.prefill(toks[:, :T].numpy())[:, -1], BF16_TOL, "prefill logits")
    for t in range(T, T + 3):
        pos = torch.full((B,), t, dtype=torch.int32)
        m.decode_step(toks[:, t].contiguous().cuda(), pos.cuda(), kv, lg, ids)
        m.sync()
        want = ref.decode(toks[:, t].numpy(), pos.numpy())
        assert_close(lg, want, BF16_TOL, "decode logits step %d" % t)
        np.testing.assert_array_equal(ids.cpu().numpy(), O.greedy(f64(lg)))


def test_e4m3_weights_need_a_bf16_model():
    need_gpu()
    shape = synth.TINY.with_(n_layers=1)  # fp32 model
    w = to_dev(synth.model_weights(shape, 3))
    for lw in w["layers"]:
        for n in binding.PROJECTIONS:
            lw[n + "_scale"] = torch.ones(lw[n].shape[0], device="cuda")
    with pytest.raises(binding.LlamaError, match="UNSUPPORTED"):
        binding.Model(shape, w, max_batch=1, max_tokens=4, max_seq=8)
