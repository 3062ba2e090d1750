"""Plain CPU oracle of the Llama2 decoder forward (prefill and decode), fp64.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
cpu_baseline / reference legs of bench.py may import or call this module. The
CUDA library never reaches it and it shares no code, constant or table with
the CUDA library; the only module both sides use is the seeded input
generator (llama2_decoder_forward_gb300.synth), which holds none of the
method's arithmetic.

Everything is computed in float64 from the stored input values (bf16 inputs are
widened exactly); no intermediate value is rounded. Each step follows the
pages' definition in their order, with numpy's matmul as the only library
primitive:

  embed -> for each layer [ h += attn(rmsnorm(h)); h += ffn(rmsnorm(h)) ]
        -> logits = lm_head(rmsnorm(h))
("Llama2架构与推理全解析" §2.3, the pseudocode of the main computation.)

Readings taken where the pages are garbled or silent (listed again in the
design notes):
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma; the operator between
    mean(x^2) and eps was lost in extraction and is read as "+" (§1.2).
  * RoPE pairs adjacent dims (2j, 2j+1) as one complex number, the form
    f(q, m) = (W_q x_m) * e^{i m theta} of "Llama2架构全景解析" §1.1, with
    theta_j = base^(-2j/d), j = 0 .. d/2-1 (§1.4: "high dims fast, low dims slow"
    read as pair 0 fastest). Positions are 0-based.
  * Only Q and K are rotated; the cache stores the rotated K and the plain V.
  * Scores are scaled by 1/sqrt(head_dim); the causal mask lets a query at
    position m see keys 0..m, the new token included (§2.3, §2.4).
  * GQA: query head h reads K/V head floor(h / G), G = n_q / n_kv (§1.5).
  * No biases anywhere; embedding and LM head are separate matrices (§2.3).
  * Greedy choice: argmax, lowest index on ties (§2.5).
  * The KV cache holds K and V in the model's storage type: the pages keep the
    cache in half precision to halve its memory ("Llama2架构全景解析" §2.1),
    so a bf16 model's cache stores each value rounded to bf16 (nearest, ties
    to even) and an fp32 model's cache rounds to fp32; an FP8 cache (FP8 is
    named as a latency option in "Llama2架构全景解析" §3.2) stores
    E4M3(value / scale) * scale, nearest with ties to even, saturating at
    +-448. Attention reads the stored values. This is the only rounding in
    the oracle (cache_dtype="f64" turns it off).

Parity status: every function here is pinned by tests/test_oracle_pins.py
(closed forms, invariants, library routines, brute force). The end-to-end
logits on random weights have no printed value to match (end-to-end parity
unpinned as a whole): they rest on the pinned parts plus the
decode-equals-prefill, extend-equals-prefill and paged-equals-contiguous
checks.
"""
from __future__ import annotations

import numpy as np

f64 = np.float64


def as64(t) -> np.ndarray:
    """Widen a torch tensor or array (fp32 / bf16) to float64 exactly."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=f64)


# --------------------------------------------------------------------------
# Layer operations
# --------------------------------------------------------------------------

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value (8 significant bits), ties to even: with
    x = m * 2^e, m in [0.5, 1), keep rint(m * 256) / 256 * 2^e."""
    m, e = np.frexp(np.asarray(x, dtype=f64))
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


E4M3_MAX = 448.0  # largest finite FP8 E4M3 value (1.75 * 2^8)


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest FP8 E4M3 value, ties to even, saturating at +-448: 3 fraction
    bits, exponent bias 7, smallest normal 2^-6, subnormal spacing 2^-9. With
    |x| = m * 2^e, m in [0.5, 1), the spacing is 2^(max(e - 1, -6) - 3)."""
    x = np.asarray(x, dtype=f64)
    a = np.abs(x)
    _, e = np.frexp(a)
    step = np.maximum(e - 1, -6) - 3
    q = np.ldexp(np.rint(np.ldexp(a, -step)), step)
    return np.sign(x) * np.minimum(q, E4M3_MAX)


def cache_store(values: np.ndarray, cache_dtype: str, scale: float = 1.0) -> np.ndarray:
    """Values as a KV cache of the given storage type holds them. "e4m3"
    stores e4m3(v / scale) and reads it back times scale (the FP8 cache of
    "Llama2架构全景解析" §3.2, reading R28)."""
    if cache_dtype == "bf16":
        return round_to_bf16(values)
    if cache_dtype == "f32":
        return np.asarray(values, dtype=np.float32).astype(f64)
    if cache_dtype == "e4m3":
        return round_to_e4m3(np.asarray(values, dtype=f64) / scale) * scale
    return np.asarray(values, dtype=f64)


def quantize_rows_e4m3(w: np.ndarray):
    """FP8 E4M3 weights with one scale per output row (row m of a [out, in]
    matrix; FP8 as the latency option of "Llama2架构全景解析" §3.2, reading
    R29): s_m = max_k |w[m, k]| / 448 (1 for an all-zero row) and
    code[m, k] = e4m3(w[m, k] / s_m), so the largest entry of every row maps
    to +-448. The scale and the quotient are fp32 operations (the
    quantisation kernel's precision; they decide the integer code), the
    rounding to E4M3 is nearest with ties to even. Returns (codes as E4M3
    values in float64, scales as float64 holding fp32 values); the weight the
    model then uses is codes * scales[:, None]."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w32), axis=1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (w32 / s[:, None]).astype(np.float32)
    return round_to_e4m3(q.astype(f64)), s.astype(f64)


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The weight an E4M3 matrix stands for: code * row scale, exactly."""
    return np.asarray(codes, dtype=f64) * np.asarray(scales, dtype=f64)[:, None]


def _kv_store(cdt, k, v):
    """K and V as stored: cdt is a storage type, or ("e4m3", k_scale, v_scale)."""
    if isinstance(cdt, tuple):
        name, ks, vs = cdt
        return cache_store(k, name, ks), cache_store(v, name, vs)
    return cache_store(k, cdt), cache_store(v, cdt)

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis, each token on its own
    ("Llama2架构与推理全解析" §1.2): y = x / sqrt(mean(x^2) + eps) * gamma."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gamma


def linear(u: np.ndarray, w: np.ndarray) -> np.ndarray:
    """u @ W^T with W stored [out, in]; equal to the pages' x W with W [in, out]
    (§1.3's SwiGLU(x) = (silu(x W_gate) * x W_up) W_down notation)."""
    return u @ w.T


def rope_frequencies(head_dim: int, theta: float) -> np.ndarray:
    """theta_j = base^(-2j/d) for pair j = 0 .. d/2-1 (§1.4)."""
    j = np.arange(head_dim // 2, dtype=f64)
    return np.power(f64(theta), -2.0 * j / head_dim)


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate each adjacent pair (x[2j], x[2j+1]) of every head by angle
    m * theta_j, m the token's position ("Llama2架构与推理全解析" §1.4;
    "Llama2架构全景解析" §1.1). x: [rows, heads, d]; positions: [rows]."""
    d = x.shape[-1]
    phi = np.asarray(positions, dtype=f64)[:, None] * rope_frequencies(d, theta)[None, :]
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    a = x[..., 0::2]
    b = x[..., 1::2]
    out = np.empty_like(x, dtype=f64)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) (§1.3)."""
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(u, w_gate, w_up, w_down) -> np.ndarray:
    """SwiGLU(u) = (silu(u W_gate) * (u W_up)) W_down (§1.3)."""
    return linear(silu(linear(u, w_gate)) * linear(u, w_up), w_down)


def softmax(s: np.ndarray) -> np.ndarray:
    """Softmax along the last axis with the row maximum subtracted before exp
    (the logit-max subtraction of "LLM架构全景解析" §3.2)."""
    z = s - np.max(s, axis=-1, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=-1, keepdims=True)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Scaled dot-product attention of one query over the given keys
    (§2.3): p = softmax(K q / sqrt(d)); o = p V. q [d]; K, V [n, d]."""
    d = q.shape[-1]
    p = softmax((K @ q) / np.sqrt(f64(d)))
    return p @ V


def gqa_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_keys: int) -> np.ndarray:
    """All query heads of one token over keys 0..n_keys-1 of its sequence (§1.5).
    q [n_q, d]; K, V [n_kv, S, d]. Head h uses K/V head h // G."""
    n_q = q.shape[0]
    n_kv = K.shape[0]
    G = n_q // n_kv
    out = np.empty_like(q, dtype=f64)
    for h in range(n_q):
        g = h // G
        out[h] = attend(q[h], K[g, :n_keys], V[g, :n_keys])
    return out


# --------------------------------------------------------------------------
# One decoder layer
# --------------------------------------------------------------------------

def _split_qkv(qkv, n_q, n_kv, d):
    rows = qkv.shape[0]
    q = qkv[:, : n_q * d].reshape(rows, n_q, d)
    k = qkv[:, n_q * d: (n_q + n_kv) * d].reshape(rows, n_kv, d)
    v = qkv[:, (n_q + n_kv) * d:].reshape(rows, n_kv, d)
    return q, k, v


def layer_decode(x, lw, shape, K, V, positions, cache_dtype=None):
    """Decode step of one layer (§2.3 main computation, §2.4 KV cache).

    x: [B, H] hidden input. lw: dict of float64 weights. K, V: per-sequence
    caches [B, n_kv, S_cap, d] (float64 arrays, updated in place: the new
    token's rotated K and its V are stored at slot positions[b], as the
    cache's storage type holds them; cache_dtype defaults to the model's).
    Returns the layer output [B, H].
    """
    cdt = shape.dtype if cache_dtype is None else cache_dtype
    n_q, n_kv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    pos = np.asarray(positions, dtype=np.int64)
    u = rmsnorm(x, lw["attn_norm"], shape.rms_eps)
    q, k, v = _split_qkv(linear(u, lw["wqkv"]), n_q, n_kv, d)
    q = rope(q, pos, shape.rope_theta)
    k = rope(k, pos, shape.rope_theta)
    B = x.shape[0]
    o = np.empty((B, n_q, d), dtype=f64)
    for b in range(B):
        m = int(pos[b])
        K[b, :, m], V[b, :, m] = _kv_store(cdt, k[b], v[b])
        o[b] = gqa_attention(q[b], K[b], V[b], m + 1)
    h = x + linear(o.reshape(B, n_q * d), lw["wo"])
    u2 = rmsnorm(h, lw["ffn_norm"], shape.rms_eps)
    return h + swiglu_ffn(u2, lw["w_gate"], lw["w_up"], lw["w_down"])


def layer_prefill(x, lw, shape, K, V, rows=None, cache_dtype=None):
    """Prefill of one layer for a fresh prompt (§2.1): x [B, T, H], token t at
    position t. Writes rotated K and V of every prompt token into K, V
    ([B, n_kv, S_cap, d], in place) and returns the output rows.

    rows: optional list of token indices whose outputs are wanted (all by
    default); K/V of every token are still computed, since later rows read them.
    The cache stores K/V in cache_dtype (default: the model's storage type).
    """
    cdt = shape.dtype if cache_dtype is None else cache_dtype
    n_q, n_kv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    B, T, H = x.shape
    rows = list(range(T)) if rows is None else list(rows)
    pos_all = np.arange(T)
    out = np.empty((B, len(rows), H), dtype=f64)
    q_rows = np.asarray(rows)
    wq = lw["wqkv"][: n_q * d]
    wkv = lw["wqkv"][n_q * d:]
    for b in range(B):
        u = rmsnorm(x[b], lw["attn_norm"], shape.rms_eps)
        kv = linear(u, wkv)
        k = kv[:, : n_kv * d].reshape(T, n_kv, d)
        v = kv[:, n_kv * d:].reshape(T, n_kv, d)
        k = rope(k, pos_all, shape.rope_theta)
        K[b, :, :T], V[b, :, :T] = _kv_store(cdt, np.transpose(k, (1, 0, 2)),
                                             np.transpose(v, (1, 0, 2)))
        q = linear(u[q_rows], wq).reshape(len(rows), n_q, d)
        q = rope(q, q_rows, shape.rope_theta)
        o = np.empty((len(rows), n_q, d), dtype=f64)
        for i, t in enumerate(rows):
            o[i] = gqa_attention(q[i], K[b], V[b], t + 1)
        h = x[b, q_rows] + linear(o.reshape(len(rows), n_q * d), lw["wo"])
        u2 = rmsnorm(h, lw["ffn_norm"], shape.rms_eps)
        out[b] = h + swiglu_ffn(u2, lw["w_gate"], lw["w_up"], lw["w_down"])
    return out


def layer_extend(x, lw, shape, K, V, seq_of_row, positions, cache_dtype=None):
    """One layer over a batch of new tokens of several sequences at once: the
    continuous-batching step ("Llama2架构全景解析" §3.1 and "基于LLAMA2与PyTorch的高效推理框架实践指南"
    §三.2 name continuous batching; §2.1's
    prefill and §2.4's decode are its two special cases). Row r is the token of
    sequence seq_of_row[r] at position positions[r]; any mix of whole prompts,
    prompt pieces after earlier pieces, and single decode tokens.

    Every row's rotated K and its V go into K, V ([B_cap, n_kv, S_cap, d], in
    place, in the cache's storage type) first; then row r attends over keys
    0 .. positions[r] of its sequence (the causal mask of §2.3: earlier rows
    of the same piece and everything cached before it). Returns [rows, H].
    """
    cdt = shape.dtype if cache_dtype is None else cache_dtype
    n_q, n_kv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    seq = np.asarray(seq_of_row, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    R = x.shape[0]
    u = rmsnorm(x, lw["attn_norm"], shape.rms_eps)
    q, k, v = _split_qkv(linear(u, lw["wqkv"]), n_q, n_kv, d)
    q = rope(q, pos, shape.rope_theta)
    k = rope(k, pos, shape.rope_theta)
    for r in range(R):
        K[seq[r], :, pos[r]], V[seq[r], :, pos[r]] = _kv_store(cdt, k[r], v[r])
    o = np.empty((R, n_q, d), dtype=f64)
    for r in range(R):
        o[r] = gqa_attention(q[r], K[seq[r]], V[seq[r]], int(pos[r]) + 1)
    h = x + linear(o.reshape(R, n_q * d), lw["wo"])
    u2 = rmsnorm(h, lw["ffn_norm"], shape.rms_eps)
    return h + swiglu_ffn(u2, lw["w_gate"], lw["w_up"], lw["w_down"])


# --------------------------------------------------------------------------
# Whole model
# --------------------------------------------------------------------------

def embed(table: np.ndarray, tokens) -> np.ndarray:
    """Row lookup in the [vocab, hidden] embedding table (§2.3)."""
    return table[np.asarray(tokens, dtype=np.int64)]


def lm_head(h, final_norm, w_lm, eps):
    """logits = lm_head(rmsnorm(h)) with its own gain (§2.3 pseudocode)."""
    return linear(rmsnorm(h, final_norm, eps), w_lm)


def greedy(logits: np.ndarray) -> np.ndarray:
    """Greedy choice: index of the largest logit, lowest index on ties (§2.5)."""
    return np.argmax(logits, axis=-1).astype(np.int32)


def sample_detail(logits, history, temperature: float, top_k: int, top_p: float,
                  repetition_penalty: float, u: float) -> dict:
    """Sampling of one next token from one row of logits ("Llama2架构与推理全解析"
    §2.5 from logits to sampling, §3.3 sampling parameters; "Llama2架构全景解析"
    §2.2 step 3: probs = softmax(logits / T), then a draw).

    Steps, in this order (the pages name the parts; their order and the
    penalty's form are the readings listed in the design notes):
      1. repetition penalty r: each distinct token id of `history` has its
         logit divided by r when positive, multiplied by r otherwise (§2.5
         asks for a lower probability for ids already produced);
      2. temperature T: s = logit / T; T == 0 is the greedy limit (argmax,
         lowest index on ties);
      3. top-k: keep the k largest s (ties broken by the lower index);
      4. softmax over the kept tokens;
      5. top-p: in the same order keep the smallest prefix whose cumulative
         probability reaches p (§2.5, nucleus sampling);
      6. renormalise and draw with the uniform u in [0, 1): the first token,
         in ascending vocabulary order, whose cumulative probability exceeds
         u (the last kept token if rounding leaves none).
    top_k <= 0 or >= V and top_p >= 1 switch steps 3 and 5 off.

    Returns {"token", "kept" (ids, ascending), "q" (their probabilities),
    "cdf_lo", "cdf_hi" (each kept token's interval of u), "z" (penalised
    logits), "s_sorted" (kept s, descending), "cum_sorted" (step-5
    cumulative probabilities in that order)}.
    """
    z = np.array(logits, dtype=f64)
    V = z.shape[0]
    if repetition_penalty != 1.0 and history is not None:
        seen = np.unique(np.asarray([t for t in np.asarray(history).ravel() if 0 <= t < V],
                                    dtype=np.int64))
        zs = z[seen]
        z[seen] = np.where(zs > 0, zs / repetition_penalty, zs * repetition_penalty)
    if temperature == 0:
        t = int(np.argmax(z))
        return {"token": t, "kept": np.array([t]), "q": np.array([1.0]),
                "cdf_lo": np.array([0.0]), "cdf_hi": np.array([1.0]), "z": z,
                "s_sorted": np.array([z[t]]), "cum_sorted": np.array([1.0])}
    s = z / temperature
    order = np.lexsort((np.arange(V), -s))  # s descending, lower index first on ties
    if 0 < top_k < V:
        order = order[:top_k]
    e = np.exp(s[order] - s[order[0]])
    cum = np.cumsum(e / e.sum())
    if top_p < 1.0:
        n = int(np.argmax(cum >= top_p)) + 1 if np.any(cum >= top_p) else len(order)
        order, e = order[:n], e[:n]
    q_sorted = e / e.sum()
    asc = np.argsort(order)
    kept, q = order[asc], q_sorted[asc]
    hi = np.cumsum(q)
    lo = hi - q
    pick = np.nonzero(hi > u)[0]
    token = int(kept[pick[0]]) if len(pick) else int(kept[-1])
    return {"token": token, "kept": kept, "q": q, "cdf_lo": lo, "cdf_hi": hi, "z": z,
            "s_sorted": s[order], "cum_sorted": cum}


def sample(logits, histories, temperature, top_k, top_p, repetition_penalty, uniforms):
    """sample_detail for each row of logits [B, V]; returns the token ids."""
    return np.array([sample_detail(logits[b], None if histories is None else histories[b],
                                   temperature, top_k, top_p, repetition_penalty,
                                   float(uniforms[b]))["token"]
                     for b in range(len(logits))], dtype=np.int32)


class Model:
    """fp64 copy of a model's weights plus per-sequence caches."""

    def __init__(self, shape, weights: dict, batch: int, capacity: int, cache_dtype=None):
        self.shape = shape
        self.cache_dtype = cache_dtype
        self.embed_t = as64(weights["embed"]) if weights.get("embed") is not None else None
        self.final_norm = as64(weights["final_norm"]) if weights.get("final_norm") is not None else None
        self.lm = as64(weights["lm_head"]) if weights.get("lm_head") is not None else None
        self.layers = [{k: as64(v) for k, v in lw.items()} for lw in weights["layers"]]
        n_kv, d = shape.n_kv_heads, shape.head_dim
        self.K = [np.zeros((batch, n_kv, capacity, d)) for _ in self.layers]
        self.V = [np.zeros((batch, n_kv, capacity, d)) for _ in self.layers]

    def prefill(self, tokens):
        """All prompt rows through every layer; returns logits of every row
        [B, T, V] (the API keeps only the last row; the oracle keeps all)."""
        h = embed(self.embed_t, tokens)
        for l, lw in enumerate(self.layers):
            h = layer_prefill(h, lw, self.shape, self.K[l], self.V[l], cache_dtype=self.cache_dtype)
        return lm_head(h, self.final_norm, self.lm, self.shape.rms_eps)

    def extend(self, tokens, seq_of_row, positions):
        """New tokens of several sequences (layer_extend); logits of every row."""
        h = embed(self.embed_t, tokens)
        for l, lw in enumerate(self.layers):
            h = layer_extend(h, lw, self.shape, self.K[l], self.V[l], seq_of_row, positions,
                             cache_dtype=self.cache_dtype)
        return lm_head(h, self.final_norm, self.lm, self.shape.rms_eps)

    def decode(self, tokens, positions):
        """One token per sequence at its position; returns logits [B, V]."""
        h = embed(self.embed_t, tokens)
        for l, lw in enumerate(self.layers):
            h = layer_decode(h, lw, self.shape, self.K[l], self.V[l], positions,
                             cache_dtype=self.cache_dtype)
        return lm_head(h, self.final_norm, self.lm, self.shape.rms_eps)


def generate_greedy(model: Model, prompt, n_steps: int):
    """Prefill, then n_steps greedy decode steps, each feeding the previous
    choice (§3.4 generation loop). Returns (ids [B, n_steps+1], logits
    [B, n_steps+1, V]) where entry 0 comes from the prefill's last row."""
    prompt = np.asarray(prompt)
    B, T = prompt.shape
    lg = model.prefill(prompt)[:, -1]
    ids = [greedy(lg)]
    logits = [lg]
    for s in range(n_steps):
        pos = np.full(B, T + s)
        lg = model.decode(ids[-1], pos)
        ids.append(greedy(lg))
        logits.append(lg)
    return np.stack(ids, 1), np.stack(logits, 1)


# --------------------------------------------------------------------------
# Paged cache
# --------------------------------------------------------------------------

def gather_paged(pool: np.ndarray, table_row, n_tokens: int, page_size: int) -> np.ndarray:
    """Logical cache of one sequence from a paged pool
    ("Llama2架构全景解析" §2.3, PagedAttention): token m lives in page
    table_row[m // P] at offset m % P. pool: [n_pages, n_kv, P, d].
    Returns [n_kv, n_tokens, d]."""
    n_kv, d = pool.shape[1], pool.shape[3]
    out = np.empty((n_kv, n_tokens, d), dtype=f64)
    for m in range(n_tokens):
        out[:, m] = pool[int(table_row[m // page_size]), :, m % page_size]
    return out


def layer_decode_paged(x, lw, shape, Kpool, Vpool, table, positions, page_size, cache_dtype=None):
    """Decode step of one layer over a paged cache: gather each sequence's
    pages into a logical contiguous cache, run layer_decode, and write the
    new token's K/V back into its page slot."""
    B = x.shape[0]
    pos = np.asarray(positions, dtype=np.int64)
    cap = int(pos.max()) + 1
    n_kv, d = shape.n_kv_heads, shape.head_dim
    K = np.zeros((B, n_kv, cap, d))
    V = np.zeros((B, n_kv, cap, d))
    for b in range(B):
        n = int(pos[b])
        K[b, :, :n] = gather_paged(Kpool, table[b], n, page_size)
        V[b, :, :n] = gather_paged(Vpool, table[b], n, page_size)
    out = layer_decode(x, lw, shape, K, V, pos, cache_dtype=cache_dtype)
    for b in range(B):
        m = int(pos[b])
        page = int(table[b][m // page_size])
        Kpool[page, :, m % page_size] = K[b, :, m]
        Vpool[page, :, m % page_size] = V[b, :, m]
    return out


# --------------------------------------------------------------------------
# Size facts
# --------------------------------------------------------------------------

def param_count(shape) -> int:
    """Parameters of a model: embedding + LM head + per layer (Wqkv, Wo,
    gate/up/down, two gains) + final gain."""
    H, I, d = shape.hidden, shape.intermediate, shape.head_dim
    per_layer = shape.qkv_rows * H + H * shape.n_q_heads * d + 3 * H * I + 2 * H
    return 2 * shape.vocab * H + shape.n_layers * per_layer + H


def kv_cache_bytes(shape, seq_len: int, bytes_per_elem: int) -> int:
    """KV cache size = 2 x layers x KV heads x head dim x length x element
    bytes ("Llama2架构与推理全解析" §2.4)."""
    return 2 * shape.n_layers * shape.n_kv_heads * shape.head_dim * seq_len * bytes_per_elem
