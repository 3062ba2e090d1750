"""Full Llama2-7B architecture (random-init bf16 weights): prefill 512 random
ids per sequence at batch 8, then 256 greedy decode steps.

The CPU oracle follows two sequences through all 32 layers, teacher-forced
with the GPU's own choices (greedy paths of bf16 and fp64 arithmetic may part
ways once two logits are within rounding of each other): one fp64 prefill of
the prompt plus the first 256 chosen ids gives the prefill's last-row logits
and the logits of every decode step (decoding a token equals the prefill row
at its position, "Llama2架构与推理全解析" §2.4); steps 0-4, 64, 128 and 256
are compared. Step 256 is also compared with a fresh GPU prefill of the
768-token sequence, a property that holds at any size.
"""
import numpy as np
import pytest
import torch

from _common import BF16_TOL, assert_close, f64, need_gpu, to_dev
from llama2_decoder_forward_gb300 import binding, synth
from oracle import llama_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_full_7b_prefill_and_greedy_decode():
    need_gpu()
    shape = synth.LLAMA2_7B
    seed = 1003
    B, T, steps, cap = 8, 512, 256, 768
    V = shape.vocab
    w = synth.model_weights(shape, seed)
    prompt = synth.token_ids(B, T, V, seed)
    model = binding.Model(shape, to_dev(w), max_batch=B, max_tokens=B * T, max_seq=cap)
    kv = binding.KVCache(shape, batch=B, capacity=cap)
    logits = torch.empty(steps + 1, B, V, device="cuda")
    ids = torch.empty(steps + 1, B, dtype=torch.int32, device="cuda")
    model.prefill(prompt.cuda(), kv, logits[0], ids[0])
    for s in range(steps):
        pos = torch.full((B,), T + s, dtype=torch.int32, device="cuda")
        model.decode_step(ids[s], pos, kv, logits[s + 1], ids[s + 1])
    model.sync()
    lg = logits.cpu()
    gi = ids.cpu().numpy()
    assert np.all(np.isfinite(lg.numpy()))
    np.testing.assert_array_equal(gi, O.greedy(f64(lg)))  # each id is its row's argmax

    # far end: step 256 against a fresh prefill of prompt + the 256 fed ids
    ext = torch.cat([prompt[0], torch.from_numpy(gi[:steps, 0])]).to(torch.int32)
    kv1 = binding.KVCache(shape, batch=1, capacity=cap)
    lg1 = torch.empty(1, V, device="cuda")
    model.prefill(ext[None].contiguous().cuda(), kv1, lg1)
    model.sync()
    assert_close(lg[steps, 0], f64(lg1)[0], BF16_TOL, "decode step 256 vs prefill of 768 tokens")

    # oracle: sequences 0 and 5 through all 32 layers, teacher-forced
    chk = [0, 1, 2, 3, 4, 64, 128, 256]
    seqs = [0, 5]
    seq = np.stack([np.concatenate([prompt[b].numpy(), gi[:steps, b]]) for b in seqs])
    Tn = seq.shape[1]
    h = O.embed(O.as64(w["embed"]), seq)
    K = np.zeros((len(seqs), shape.n_kv_heads, Tn, shape.head_dim))
    Vc = np.zeros_like(K)
    for lw in w["layers"]:
        h = O.layer_prefill(h, {k: O.as64(v) for k, v in lw.items()}, shape, K, Vc)
    rows = [T - 1 + s for s in chk]
    ref = O.lm_head(h[:, rows], O.as64(w["final_norm"]), O.as64(w["lm_head"]), shape.rms_eps)
    got = np.stack([f64(lg[chk, b]) for b in seqs])
    assert_close(got, ref, BF16_TOL, "sequences 0 and 5: prefill and decode steps %s" % chk)
    # a GPU choice may differ from the oracle's only where the oracle's top two
    # logits are closer than the tolerance
    top2 = np.sort(ref, -1)[..., -2:]
    clear = top2[..., 1] - top2[..., 0] > BF16_TOL[0] + BF16_TOL[1] * np.abs(top2[..., 1])
    chosen = np.stack([gi[chk, b] for b in seqs])
    assert np.all(chosen[clear] == O.greedy(ref)[clear])
