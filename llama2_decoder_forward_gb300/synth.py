"""Seeded synthetic inputs for the Llama2 decoder forward.

This module is shared by the tests, the benchmark and the CPU oracle. It only
draws random numbers and rounds them to the storage type; it holds none of the
forward pass's arithmetic.

Recipe (the pages print no dataset or trained weights, so every input is drawn):
  * weights ~ N(0, std), std 0.02 (0.01 for the 70B-shaped layer);
  * RMSNorm gains gamma = 1 + N(0, 0.1);
  * embedding table and LM head ~ N(0, 0.02), independent (untied);
  * layer-only inputs: hidden x ~ N(0, 1), cached K/V ~ N(0, 1);
  * token ids uniform in [0, vocab); ragged context lengths uniform integers
    in [lo, hi]; page ids a random permutation of the pool.
Values are drawn in fp32 by torch's seeded generator and rounded to bf16
(round-to-nearest-even, torch's float->bfloat16 cast) for bf16 shapes.
Seeds: 1000 + config index for weights, +100 for hidden/cache inputs,
+200 for token ids and lengths, +300 for the page permutation; each layer
draws from its own stream so one layer can be regenerated alone.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Shape:
    """Hyper-parameters of a Llama2-style decoder (size table of
    "Llama2架构与推理全解析" §1.6)."""

    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    dtype: str = "bf16"  # storage type of weights, cache and GEMM inputs: "f32" | "bf16"

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Shape":
        return replace(self, **kw)


# The tiny fp32 model and the Llama2 sizes (7B / 13B / 70B rows of the size table).
TINY = Shape(2, 256, 4, 2, 64, 688, 1024, dtype="f32")
LLAMA2_7B = Shape(32, 4096, 32, 32, 128, 11008, 32000)
LLAMA2_13B = Shape(40, 5120, 40, 40, 128, 13824, 32000)
LLAMA2_70B = Shape(80, 8192, 64, 8, 128, 28672, 32000)

LAYER_NAMES = ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def _gen(seed, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, dtype, mean=0.0):
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def layer_weights(shape: Shape, seed: int, layer: int, std: float = 0.02, device="cpu",
                  n_kv_used: int | None = None) -> dict:
    """One decoder layer's weights in storage dtype, row-major, projections [out, in].

    wqkv stacks the Q, K and V projections along rows: q rows [0, n_q*d),
    k rows [n_q*d, (n_q+n_kv)*d), v rows after that.
    """
    H, d, I = shape.hidden, shape.head_dim, shape.intermediate
    dt = shape.torch_dtype
    g = _gen(seed * 1_000_003 + 7919 * (layer + 1), device)
    w = {}
    w["attn_norm"] = _normal((H,), 0.1, g, device, dt, mean=1.0)
    w["wqkv"] = _normal((shape.qkv_rows, H), std, g, device, dt)
    w["wo"] = _normal((H, shape.n_q_heads * d), std, g, device, dt)
    w["ffn_norm"] = _normal((H,), 0.1, g, device, dt, mean=1.0)
    w["w_gate"] = _normal((I, H), std, g, device, dt)
    w["w_up"] = _normal((I, H), std, g, device, dt)
    w["w_down"] = _normal((H, I), std, g, device, dt)
    return w


def gqa_variant(w: dict, shape: Shape, n_kv: int) -> dict:
    """The same layer with only the first n_kv K/V heads kept (GQA variant of the
    ragged paged workload: Wk/Wv keep their first n_kv*d rows)."""
    d, nq, nkv = shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    q = w["wqkv"][: nq * d]
    k = w["wqkv"][nq * d: nq * d + n_kv * d]
    v = w["wqkv"][(nq + nkv) * d: (nq + nkv) * d + n_kv * d]
    out = dict(w)
    out["wqkv"] = torch.cat([q, k, v], 0).contiguous()
    return out


def model_weights(shape: Shape, seed: int, std: float = 0.02, device="cpu") -> dict:
    """Embedding, final norm, LM head and every layer's weights."""
    dt = shape.torch_dtype
    g = _gen(seed * 1_000_003 + 1, device)
    out = {
        "embed": _normal((shape.vocab, shape.hidden), 0.02, g, device, dt),
        "final_norm": _normal((shape.hidden,), 0.1, g, device, dt, mean=1.0),
        "lm_head": _normal((shape.vocab, shape.hidden), 0.02, g, device, dt),
    }
    out["layers"] = [layer_weights(shape, seed, l, std, device) for l in range(shape.n_layers)]
    return out


def hidden_input(rows: int, hidden: int, seed: int, device="cpu") -> torch.Tensor:
    """Layer input x ~ N(0, 1), fp32 (the residual stream is kept in fp32)."""
    return _normal((rows, hidden), 1.0, _gen(seed + 100, device), device, torch.float32)


def cache_values(shape_tuple, seed: int, dtype, device="cpu", stream: int = 0) -> torch.Tensor:
    """Cached K or V entries ~ N(0, 1), already in cache storage dtype."""
    return _normal(shape_tuple, 1.0, _gen(seed + 100 + 17 * (stream + 1), device), device, dtype)


def token_ids(batch: int, length: int, vocab: int, seed: int) -> torch.Tensor:
    g = _gen(seed + 200)
    return torch.randint(0, vocab, (batch, length), generator=g, dtype=torch.int32)


def ragged_lengths(batch: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Context lengths uniform integers in [lo, hi] inclusive."""
    g = _gen(seed + 200)
    return torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int32)


def page_table(n_pages_per_seq, max_pages: int, seed: int):
    """Random-permutation page table.

    n_pages_per_seq: list of page counts; pages are drawn as one random
    permutation of range(sum(counts)) and dealt out in order. Unused slots
    of a row hold -1. Returns (table [B, max_pages] int32, n_pages_total).
    """
    total = int(sum(n_pages_per_seq))
    g = _gen(seed + 300)
    perm = torch.randperm(total, generator=g).to(torch.int32)
    table = torch.full((len(n_pages_per_seq), max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(n_pages_per_seq):
        table[b, :n] = perm[off: off + n]
        off += n
    return table, total
