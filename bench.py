"""Benchmark: Llama2-7B decode step (32 layers, batch 32, 1024 cached positions).

One step = one llama_decode_step: embedding, 32 x (RMSNorm, Q/K/V projection,
RoPE + KV append, GQA flash-decode attention over 1025 keys, output
projection + residual, RMSNorm, gate/up + SiLU*up, down + residual), final
RMSNorm, LM head and greedy argmax, for 32 sequences. Weights are random
N(0, 0.02) bf16 of the 7B architecture, the cache holds N(0, 1) bf16 values at
positions 0..1023 of every layer, token ids are uniform; all synthetic.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload model|layer|prefill|extend]
  python bench.py --impl reference ...   (the CPU oracle on a bounded sample)

Prints one JSON line (rank 0). Under torchrun each rank runs its own replica of
the workload on its GPU (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Llama2-7B decode tokens/s (bs32, ctx1024); decode-step HBM GB/s vs peak"


def workload_name(workload):
    """The decode workload both arms (GPU and CPU oracle) report in config."""
    if workload == "model":
        return ("llama2-7b decode step: 32 layers + embedding + LM head + greedy, "
                "batch 32, 1024 cached positions, contiguous KV")
    return "one llama2-7b decoder layer, decode step, batch 32, 1024 cached positions"
B, CTX, CAP = 32, 1024, 1040


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _traffic(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or
    None when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = {"attn_decode": "k_attention.cu", "gemm": "k_gemm.cu"}[kernel]
    with open(os.path.join(ROOT, "llama2_decoder_forward_gb300", "csrc", src), "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == B_WORKLOAD:
            return float(parts[3]) if parts[2] == h else None
    return None


B_WORKLOAD = "model"


class Clocks:
    """nvidia-smi sampler for the timed region: started before it (and waited
    for until its first sample arrives), sampling every 20 ms; the summary
    keeps the samples taken between mark_start() and mark_end()."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None
        self.lines = []
        self.t0 = self.t1 = None

    def _read(self):
        for line in self.p.stdout:
            self.lines.append((time.perf_counter(), line))

    def __enter__(self):
        import threading
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "20"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
            t = time.perf_counter()
            while not self.lines and time.perf_counter() - t < 5:
                time.sleep(0.01)
        except Exception:
            self.p = None
        self.mark_start()
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *a):
        if self.t1 is None:
            self.mark_end()
        if self.p:
            time.sleep(0.05)
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        window = [l for t, l in self.lines if self.t0 <= t <= self.t1 + 0.025]
        for line in window:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "interval_ms": 20}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_result(ms_per_step, tokens_per_step, device=None):
    """Combine the replicas of a multi-GPU run: the slowest rank's step time
    (max over ranks) and the whole job's tokens per second (every rank decodes
    its own batch; no data crosses ranks). Single process: unchanged."""
    import torch
    import torch.distributed as dist
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    if ws > 1:
        t = torch.tensor([float(ms_per_step)], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_per_step = float(t.item())
    return ms_per_step, tokens_per_step * ws / (ms_per_step * 1e-3)


# ----------------------------------------------------------------------------- GPU arm
def build_model(workload, device, kv_e4m3=False, w_e4m3=False):
    import torch
    from llama2_decoder_forward_gb300 import binding, synth

    shape = synth.LLAMA2_7B if workload == "model" else synth.LLAMA2_7B.with_(n_layers=1)
    seed = 1003
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def rn(*s, std=0.02, mean=0.0):
        t = torch.randn(*s, generator=g, device=device, dtype=torch.float32)
        t.mul_(std).add_(mean)
        return t.to(torch.bfloat16)

    H, I, V = shape.hidden, shape.intermediate, shape.vocab
    layers = []
    for _ in range(shape.n_layers):
        layers.append({"attn_norm": rn(H, std=0.1, mean=1.0), "wqkv": rn(shape.qkv_rows, H),
                       "wo": rn(H, H), "ffn_norm": rn(H, std=0.1, mean=1.0), "w_gate": rn(I, H),
                       "w_up": rn(I, H), "w_down": rn(H, I)})
    if w_e4m3:  # E4M3 projections with row scales, quantised on the device
        layers = [binding.quantize_layer_e4m3(lw) for lw in layers]
        torch.cuda.synchronize()
    w = {"layers": layers}
    if workload == "model":
        w.update(embed=rn(V, H), final_norm=rn(H, std=0.1, mean=1.0), lm_head=rn(V, H))
    if kv_e4m3:  # one byte per value: N(0, 1) / scale rounded to E4M3
        kv = binding.KVCache(shape, batch=B, capacity=CAP, e4m3=(1.0 / 64, 1.0 / 64))
        for t in (kv.k, kv.v):
            f = torch.randn(t.numel() // (CAP * shape.head_dim), CTX, shape.head_dim,
                            generator=g, device=device) * 64
            t.view(-1, CAP, shape.head_dim)[:, :CTX] = f.clamp_(-448, 448).to(
                torch.float8_e4m3fn).view(torch.uint8)
            t.view(-1, CAP, shape.head_dim)[:, CTX:].zero_()
            del f
    else:
        kv = binding.KVCache(shape, batch=B, capacity=CAP)
        for t in (kv.k, kv.v):
            t.view(-1, CAP, shape.head_dim)[:, :CTX].normal_(generator=g)
            t.view(-1, CAP, shape.head_dim)[:, CTX:].zero_()
    model = binding.Model(shape, w, max_batch=B, max_tokens=B, max_seq=CAP,
                          has_embed_head=(workload == "model"))
    return shape, model, kv, w


def _time_ms(fn, stream, steps, warmup=3):
    """Average device time of fn() over `steps` calls, CUDA events on `stream`
    after `warmup` untimed calls."""
    import torch
    torch.cuda.synchronize()  # inputs drawn on the default stream are complete
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def prefill_70b_layer_numbers(m, x, kv, stream, tflops, steps=3):
    """Prefill of 4096 rows through one 70B-shaped layer: tokens/s, and the
    GEMMs' and the attention's algorithmic TFLOP/s against the bf16 peak
    (the attention counts the unmasked half, 4 n_q d T(T+1)/2)."""
    from llama2_decoder_forward_gb300 import synth
    s70 = synth.LLAMA2_70B
    T = x.shape[0]
    fn = lambda: m.prefill_hidden(x, 1, T, kv)
    ms = _time_ms(fn, stream, steps)
    m.profile(["gemm", "attn_prefill"])
    for _ in range(2):
        fn()
    gm, _ = m.profile_read("gemm")
    am, _ = m.profile_read("attn_prefill")
    m.profile([])
    m.sync()
    gm, am = gm / 2, am / 2
    H, I = s70.hidden, s70.intermediate
    gflop = 2.0 * T * (s70.qkv_rows * H + H * s70.n_q_heads * s70.head_dim + 3 * H * I)
    aflop = 4.0 * s70.n_q_heads * s70.head_dim * (T * (T + 1) / 2)
    g_tf = gflop / (gm * 1e-3) / 1e12
    a_tf = aflop / (am * 1e-3) / 1e12
    return {"tokens_per_s": T / (ms * 1e-3), "ms": ms,
            "gemm": {"tflops": g_tf, "frac": g_tf / tflops, "ms": gm},
            "attention": {"tflops": a_tf, "frac": a_tf / tflops, "ms": am}}


def extra_workloads(dev, stream, w7, hbm, tflops):
    """The other workloads of the scope table, each timed after the headline
    decode step (not part of its timed region): the 8 x 512 prefill of the full
    7B model, one 70B-shaped layer (decode at batch 32 over 4096 positions,
    and a 4096-token prefill), and ragged paged decode on 7B layer shapes (MHA
    and GQA; the attention alone per context-length bin too)."""
    import torch
    from llama2_decoder_forward_gb300 import binding, synth

    out = {}
    g = torch.Generator(device=dev)
    g.manual_seed(2024)

    def rn(*s, std=0.02, mean=0.0):
        t = torch.randn(*s, generator=g, device=dev, dtype=torch.float32)
        return t.mul_(std).add_(mean).to(torch.bfloat16)

    def layer(shape, std):
        H, I = shape.hidden, shape.intermediate
        return {"attn_norm": rn(H, std=0.1, mean=1.0), "wqkv": rn(shape.qkv_rows, H, std=std),
                "wo": rn(H, shape.n_q_heads * shape.head_dim, std=std),
                "ffn_norm": rn(H, std=0.1, mean=1.0), "w_gate": rn(I, H, std=std),
                "w_up": rn(I, H, std=std), "w_down": rn(H, I, std=std)}

    def layer_params(shape):
        H, I = shape.hidden, shape.intermediate
        return shape.qkv_rows * H + H * shape.n_q_heads * shape.head_dim + 3 * H * I

    def prof(model, fn, kinds, steps):
        model.profile(kinds)
        for _ in range(steps):
            fn()
        r = {k: model.profile_read(k) for k in kinds}
        model.profile([])
        model.sync()
        return {k: (ms / steps, n / steps) for k, (ms, n) in r.items()}

    # ---- the FP8 options of the same decode step (not the headline configuration):
    # an E4M3 KV cache, then E4M3 projection weights with row scales
    def decode_variant(weights, kv, name):
        m = binding.Model(synth.LLAMA2_7B, weights, max_batch=B, max_tokens=B, max_seq=CAP,
                          stream=stream)
        tok = torch.randint(0, synth.LLAMA2_7B.vocab, (B,), generator=g, device=dev,
                            dtype=torch.int32)
        pos = torch.full((B,), CTX, dtype=torch.int32, device=dev)
        lg = torch.empty(B, synth.LLAMA2_7B.vocab, device=dev)
        ids = torch.empty(B, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        m.capture_decode(tok, pos, kv, lg, ids, advance=False)
        ms = _time_ms(m.graph_launch, stream, 20)
        m.profile(["attn_decode", "gemm"])
        for _ in range(5):
            m.decode_step(tok, pos, kv, lg, ids)
        am, an = m.profile_read("attn_decode")
        gm, _ = m.profile_read("gemm")
        m.profile([])
        m.sync()
        return {"workload": name, "tokens_per_s": B / (ms * 1e-3), "ms": ms,
                "attn_decode_ms": am / max(an, 1), "gemm_ms_per_step": gm / 5}

    s7 = synth.LLAMA2_7B
    kv8 = binding.KVCache(s7, batch=B, capacity=CAP, e4m3=(1.0 / 64, 1.0 / 64))
    for t in (kv8.k, kv8.v):
        view = t.view(-1, CAP, s7.head_dim)
        for i in range(0, view.shape[0], 4096):
            f = torch.randn(min(4096, view.shape[0] - i), CTX, s7.head_dim, generator=g,
                            device=dev) * 64
            view[i:i + 4096, :CTX] = f.clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        view[:, CTX:].zero_()
    r = decode_variant(w7, kv8, "7B decode step as the headline, KV cache E4M3 (byte per value)")
    kvb = B * s7.n_kv_heads * (CTX + 1) * s7.head_dim * 2  # K and V bytes of one layer
    r["attn_decode_gbs"] = kvb / (r["attn_decode_ms"] * 1e-3) / 1e9
    r["attn_decode_frac"] = r["attn_decode_gbs"] / hbm
    out["decode_kv_e4m3"] = r
    del kv8
    torch.cuda.empty_cache()
    w8 = dict(w7)
    w8["layers"] = [binding.quantize_layer_e4m3(lw) for lw in w7["layers"]]
    kvb16 = binding.KVCache(s7, batch=B, capacity=CAP)
    for t in (kvb16.k, kvb16.v):
        t.view(-1, CAP, s7.head_dim)[:, :CTX].normal_(generator=g)
        t.view(-1, CAP, s7.head_dim)[:, CTX:].zero_()
    out["decode_w_e4m3"] = decode_variant(
        w8, kvb16, "7B decode step as the headline, projection weights E4M3 with row scales")
    del w8, kvb16
    torch.cuda.empty_cache()

    # ---- full 7B prefill, 8 sequences x 512 tokens (the same weights)
    shape = synth.LLAMA2_7B
    Bp, Tp = 8, 512
    m = binding.Model(shape, w7, max_batch=Bp, max_tokens=Bp * Tp, max_seq=768, stream=stream)
    kvp = binding.KVCache(shape, batch=Bp, capacity=768)
    toks = torch.randint(0, shape.vocab, (Bp, Tp), generator=g, device=dev, dtype=torch.int32)
    lg = torch.empty(Bp, shape.vocab, device=dev)
    ids = torch.empty(Bp, dtype=torch.int32, device=dev)
    fn = lambda: m.prefill(toks, kvp, lg, ids)
    ms = _time_ms(fn, stream, 5)
    k = prof(m, fn, ["gemm", "attn_prefill"], 3)
    rows = Bp * Tp
    gflop = 2.0 * rows * layer_params(shape) * shape.n_layers + 2.0 * Bp * shape.vocab * shape.hidden
    aflop = 4.0 * shape.n_q_heads * shape.head_dim * (Tp * (Tp + 1) / 2) * Bp * shape.n_layers
    g_tf = gflop / (k["gemm"][0] * 1e-3) / 1e12
    a_tf = aflop / (k["attn_prefill"][0] * 1e-3) / 1e12
    out["prefill_7b"] = {
        "workload": "llama2-7b prefill, 8 sequences x 512 random ids, 32 layers + LM head on last rows",
        "tokens_per_s": rows / (ms * 1e-3), "ms": ms,
        "gemm": {"tflops": g_tf, "frac": g_tf / tflops, "ms": k["gemm"][0], "launches": k["gemm"][1]},
        "attention": {"tflops": a_tf, "frac": a_tf / tflops, "ms": k["attn_prefill"][0]}}
    del m, kvp
    torch.cuda.empty_cache()

    # ---- one 70B-shaped layer: decode at batch 32 over 4096 positions, and a 4096-token prefill
    s70 = synth.LLAMA2_70B.with_(n_layers=1)
    w70 = {"layers": [layer(s70, 0.01)]}
    S70, cap70 = 4096, 4112
    m = binding.Model(s70, w70, max_batch=B, max_tokens=S70, max_seq=cap70, has_embed_head=False,
                      stream=stream)
    kv = binding.KVCache(s70, batch=B, capacity=cap70)
    kv.k.normal_(generator=g)
    kv.v.normal_(generator=g)
    h0 = torch.randn(B, s70.hidden, generator=g, device=dev)
    h = h0.clone()
    pos = torch.full((B,), S70, dtype=torch.int32, device=dev)
    fn = lambda: m.decode_hidden(h, pos, kv)
    ms = _time_ms(fn, stream, 20)
    k = prof(m, fn, ["attn_decode", "gemm"], 5)
    kvb = B * s70.n_kv_heads * (S70 + 1) * s70.head_dim * 2 * 2
    wb = layer_params(s70) * 2
    out["layer_70b_decode"] = {
        "workload": "one llama2-70b layer (64 q / 8 kv heads), decode at batch 32 over 4096 cached positions",
        "ms": ms, "gbs": (wb + kvb) / (ms * 1e-3) / 1e9, "frac": (wb + kvb) / (ms * 1e-3) / 1e9 / hbm,
        "algorithmic_bytes": wb + kvb,
        "attention": {"gbs": kvb / (k["attn_decode"][0] * 1e-3) / 1e9,
                      "frac": kvb / (k["attn_decode"][0] * 1e-3) / 1e9 / hbm},
        "gemm": {"gbs": wb / (k["gemm"][0] * 1e-3) / 1e9,
                 "frac": wb / (k["gemm"][0] * 1e-3) / 1e9 / hbm}}
    kv1 = binding.KVCache(s70, batch=1, capacity=cap70)
    x = torch.randn(S70, s70.hidden, generator=g, device=dev)
    out["layer_70b_prefill_4096"] = {
        "workload": "one llama2-70b layer, causal prefill of 4096 tokens at batch 1",
        **prefill_70b_layer_numbers(m, x, kv1, stream, tflops)}
    del m, kv, kv1, w70, x
    torch.cuda.empty_cache()

    # ---- ragged paged decode on 7B layer shapes, MHA and GQA (32 q / 8 kv)
    lens = synth.ragged_lengths(64, 128, 4096, 1005)
    n_pages = [(int(L) + 1 + 15) // 16 for L in lens]
    table, total = synth.page_table(n_pages, max(n_pages), 1005)
    table = table.to(dev)
    posr = lens.to(dev)
    base = layer(synth.LLAMA2_7B.with_(n_layers=1), 0.02)
    rag = {}
    for name, nkv in (("mha", 32), ("gqa", 8)):
        s5 = synth.LLAMA2_7B.with_(n_layers=1)
        lw = base if nkv == 32 else synth.gqa_variant(base, s5, nkv)
        s5 = s5.with_(n_kv_heads=nkv)
        m = binding.Model(s5, {"layers": [lw]}, max_batch=64, max_tokens=0, max_seq=max(n_pages) * 16,
                          has_embed_head=False, stream=stream)
        kvr = binding.KVCache(s5, n_pages=total, page_size=16, page_table=table)
        kvr.k.normal_(generator=g)
        kvr.v.normal_(generator=g)
        h0 = torch.randn(64, s5.hidden, generator=g, device=dev)
        h = h0.clone()
        fn = lambda: m.decode_hidden(h, posr, kvr)
        ms = _time_ms(fn, stream, 20)
        kvb = int(sum(int(L) + 1 for L in lens)) * nkv * s5.head_dim * 2 * 2
        wb = layer_params(s5) * 2
        q = torch.randn(64, s5.n_q_heads, s5.head_dim, generator=g, device=dev).to(torch.bfloat16)
        o = torch.empty(64, s5.n_q_heads * s5.head_dim, device=dev, dtype=torch.bfloat16)
        am = _time_ms(lambda: m.op_attention_decode(q, posr, 0, kvr, o), stream, 20)
        bins = []
        for lo, hi in ((128, 1024), (1025, 2048), (2049, 3072), (3073, 4096)):
            idx = [i for i, L in enumerate(lens.tolist()) if lo <= L <= hi]
            if not idx:
                continue
            it = torch.tensor(idx, device=dev)
            kb = binding.KVCache(s5, n_pages=total, page_size=16,
                                 page_table=table[it].contiguous(), k=kvr.k, v=kvr.v)
            qb, pb = q[it].contiguous(), posr[it].contiguous()
            ob = o[: len(idx)]
            bm = _time_ms(lambda: m.op_attention_decode(qb, pb, 0, kb, ob), stream, 20)
            bb = int(sum(int(lens[i]) + 1 for i in idx)) * nkv * s5.head_dim * 4
            bins.append({"lengths": [lo, hi], "sequences": len(idx), "ms": bm,
                         "gbs": bb / (bm * 1e-3) / 1e9, "frac": bb / (bm * 1e-3) / 1e9 / hbm})
        rag[name] = {"ms": ms, "gbs": (wb + kvb) / (ms * 1e-3) / 1e9,
                     "frac": (wb + kvb) / (ms * 1e-3) / 1e9 / hbm,
                     "attention": {"ms": am, "gbs": kvb / (am * 1e-3) / 1e9,
                                   "frac": kvb / (am * 1e-3) / 1e9 / hbm},
                     "attention_by_length": bins}
        del m, kvr
        torch.cuda.empty_cache()
    out["ragged_paged_7b_layer"] = {
        "workload": "one llama2-7b layer, 64 sequences with cached lengths uniform in [128, 4096], "
                    "pages of 16 tokens in a random permutation, decode one token each",
        **rag}
    return out


def run_gpu(args):
    import torch
    from llama2_decoder_forward_gb300 import binding
    import __graft_entry__

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    __graft_entry__.build()
    shape, model, kv, w7 = build_model(args.workload, dev, kv_e4m3=args.kv == "e4m3",
                                       w_e4m3=args.weights == "e4m3")
    torch.cuda.synchronize()  # inputs are drawn on the default stream; the model runs on its own
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    tokens = torch.randint(0, shape.vocab, (B,), generator=g, device=dev, dtype=torch.int32)
    positions = torch.full((B,), CTX, dtype=torch.int32, device=dev)
    logits = torch.empty(B, shape.vocab, device=dev)
    ids = torch.empty(B, dtype=torch.int32, device=dev)
    hidden0 = torch.randn(B, shape.hidden, generator=g, device=dev)
    hidden = hidden0.clone()

    stream = torch.cuda.Stream(device=dev)
    model.set_stream(stream)
    use_graph = args.workload == "model" and not args.no_graph

    def step():
        if args.workload == "model":
            if use_graph:
                model.graph_launch()
            else:
                model.decode_step(tokens, positions, kv, logits, ids)
        else:
            with torch.cuda.stream(stream):
                hidden.copy_(hidden0)
            model.decode_hidden(hidden, positions, kv)

    torch.cuda.synchronize()
    if use_graph:  # the whole decode step as one CUDA graph (positions stay at 1024)
        model.capture_decode(tokens, positions, kv, logits, ids, advance=False)

    for _ in range(args.warmup):
        step()
    model.sync()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    n0 = model.launch_count()
    with Clocks(local) as clk:
        barrier()
        clk.mark_start()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
        clk.mark_end()
    launches = model.launch_count() - n0
    ms = e0.elapsed_time(e1) / args.steps
    model.sync()
    # per-kernel device time: a second pass over the same steps (direct
    # launches) with the library's event hooks around every launch of the two
    # big kernel classes
    dominant = "attn_decode"
    model.profile([dominant, "gemm"])
    for _ in range(args.steps):
        if args.workload == "model":
            model.decode_step(tokens, positions, kv, logits, ids)
        else:
            step()
    attn_ms, attn_n = model.profile_read(dominant)
    gemm_ms, gemm_n = model.profile_read("gemm")
    model.profile([])
    model.sync()
    sample_ms = None
    if args.workload == "model":
        # the sampler on this step's logits (not part of the greedy step timed
        # above): T 0.7, top-k 50, top-p 0.9, repetition penalty 1.1 over a
        # 1024-token history per sequence
        hist = torch.randint(0, shape.vocab, (B, CTX), generator=g, device=dev, dtype=torch.int32)
        hlen = torch.full((B,), CTX, dtype=torch.int32, device=dev)
        uni = torch.rand(B, generator=g, device=dev)
        sids = torch.empty(B, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        kw = dict(temperature=0.7, top_k=50, top_p=0.9, repetition_penalty=1.1, history=hist,
                  history_len=hlen)
        for _ in range(3):
            model.sample(logits, uni, sids, **kw)
        model.profile(["sample"])
        for _ in range(20):
            model.sample(logits, uni, sids, **kw)
        s_ms, s_n = model.profile_read("sample")
        model.profile([])
        model.sync()
        sample_ms = s_ms / max(s_n, 1)
    ms, value = replica_result(ms, B, dev)

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = None
    if args.workload == "model":
        th = tokens.cpu().pin_memory()
        ph = positions.cpu().pin_memory()
        lh = torch.empty(B, shape.vocab).pin_memory()
        ih = torch.empty(B, dtype=torch.int32).pin_memory()
        model.decode_step_host(th, ph, kv, lh, ih)
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            model.decode_step_host(th, ph, kv, lh, ih)
        el = time.perf_counter() - t0
        e2e = {"value": B * ws * args.steps / el, "unit": "tokens/s",
               "h2d_bytes_per_step": 2 * B * 4, "d2h_bytes_per_step": B * shape.vocab * 4 + B * 4}

    if rank != 0:
        return
    hbm, tflops, peak_kind = _peaks()
    L = shape.n_layers
    kv_elem = 1 if args.kv == "e4m3" else 2
    kv_bytes = B * shape.n_kv_heads * (CTX + 1) * shape.head_dim * 2 * kv_elem  # K and V per layer
    attn_avg = attn_ms / max(attn_n, 1)
    achieved = kv_bytes / (attn_avg * 1e-3) / 1e9
    w_rows = shape.qkv_rows + shape.hidden + 3 * shape.intermediate  # wqkv, wo, gate, up, down
    w_elems = (shape.qkv_rows + shape.hidden) * shape.hidden + 3 * shape.hidden * shape.intermediate
    # bf16 weights, or E4M3 bytes plus one fp32 scale per row
    wbytes = w_elems * 2 if args.weights == "bf16" else w_elems + 4 * w_rows
    lm_bytes = shape.vocab * shape.hidden * 2 if args.workload == "model" else 0
    step_bytes = L * (wbytes + kv_bytes) + lm_bytes
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" + ("" if args.kv == "bf16" else " (KV cache e4m3)") +
                 ("" if args.weights == "bf16" else " (projection weights e4m3)"),
        "data": "synthetic (random-init 7B weights N(0,0.02), cache N(0,1), uniform token ids)",
        "config": {"workload": workload_name(args.workload),
                   "batch": B, "context": CTX, "kv_cache": args.kv, "weights": args.weights, "l2": "inputs larger than L2 (%.1f GB per step)" % (step_bytes / 1e9),
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "launch": "cuda graph of the step" if use_graph else "direct launches"},
        "step_hbm_gbs": step_bytes / (ms * 1e-3) / 1e9,
        "step_hbm_frac": step_bytes / (ms * 1e-3) / 1e9 / hbm,
        "roofline": {"kernel": "attn_decode (flash-decode over the KV cache)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": peak_kind,
                     "traffic": _traffic("attn_decode") if args.kv == "bf16" else None,
                     "algorithmic_bytes_per_launch": kv_bytes, "avg_launch_ms": attn_avg,
                     "launches": attn_n},
        "kernels": {"attn_decode_ms_per_step": attn_ms / args.steps,
                    "gemm_ms_per_step": gemm_ms / args.steps,
                    "gemm_gbs": (L * wbytes + lm_bytes) / (gemm_ms / args.steps * 1e-3) / 1e9
                    if gemm_ms > 0 else None,
                    "sample_ms": sample_ms},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if (args.workload == "model" and args.kv == "bf16" and args.weights == "bf16"
            and not args.no_extra):
        line["workloads"] = extra_workloads(dev, stream, w7, hbm, tflops)
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    print(json.dumps(line), flush=True)


def run_prefill(args):
    """Prefill of 8 sequences x 512 random ids on the full 7B model (the
    prefill half of the full-model workload): prefill tokens/s and the tensor
    throughput of the GEMMs (the dense contraction that bounds prefill)."""
    import torch
    import __graft_entry__
    from llama2_decoder_forward_gb300 import binding, synth

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    __graft_entry__.build()
    Bp, Tp, cap = 8, 512, 768
    # fewer layers: the same kernels and launch shapes in a few GB (profiling)
    shape = synth.LLAMA2_7B.with_(n_layers=args.layers)
    g = torch.Generator(device=dev)
    g.manual_seed(1004)

    def rn(*s, std=0.02, mean=0.0):
        t = torch.randn(*s, generator=g, device=dev, dtype=torch.float32)
        return t.mul_(std).add_(mean).to(torch.bfloat16)

    H, I, V = shape.hidden, shape.intermediate, shape.vocab
    w = {"layers": [{"attn_norm": rn(H, std=0.1, mean=1.0), "wqkv": rn(shape.qkv_rows, H), "wo": rn(H, H),
                     "ffn_norm": rn(H, std=0.1, mean=1.0), "w_gate": rn(I, H), "w_up": rn(I, H),
                     "w_down": rn(H, I)} for _ in range(shape.n_layers)],
         "embed": rn(V, H), "final_norm": rn(H, std=0.1, mean=1.0), "lm_head": rn(V, H)}
    model = binding.Model(shape, w, max_batch=Bp, max_tokens=Bp * Tp, max_seq=cap)
    kv = binding.KVCache(shape, batch=Bp, capacity=cap)
    tokens = torch.randint(0, V, (Bp, Tp), generator=g, device=dev, dtype=torch.int32)
    logits = torch.empty(Bp, V, device=dev)
    ids = torch.empty(Bp, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        model.prefill(tokens, kv, logits, ids)
    model.sync()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(0) as clk:
        e0.record()
        for _ in range(args.steps):
            model.prefill(tokens, kv, logits, ids)
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    model.profile(["gemm", "attn_prefill"])
    for _ in range(args.steps):
        model.prefill(tokens, kv, logits, ids)
    gemm_ms, gemm_n = model.profile_read("gemm")
    att_ms, att_n = model.profile_read("attn_prefill")
    model.profile([])
    model.sync()
    rows = Bp * Tp
    layer_params = shape.qkv_rows * H + H * H + 3 * H * I
    gemm_flops = 2.0 * rows * layer_params * shape.n_layers + 2.0 * Bp * V * H
    att_flops = 4.0 * shape.n_q_heads * shape.head_dim * (Tp * (Tp + 1) / 2) * Bp * shape.n_layers
    hbm, tflops, peak_kind = _peaks()
    g_tf = gemm_flops / (gemm_ms / args.steps * 1e-3) / 1e12
    line = {"metric": "Llama2-7B prefill tokens/s (bs8, 512 tokens)", "value": rows / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init 7B weights, uniform ids)",
            "config": {"workload": "llama2-7b prefill, 8 sequences x 512 tokens, %d layers + LM head on last rows"
                                   % shape.n_layers},
            "roofline": {"kernel": "gemm_tm_kernel (prefill projections) + gemm_tc_kernel (LM head)",
                         "bound": "tensor",
                         "achieved": g_tf, "peak": tflops, "unit": "TFLOP/s", "frac": g_tf / tflops,
                         "peak_source": peak_kind, "traffic": None,
                         "algorithmic_flops_per_step": gemm_flops, "launches_per_step": gemm_n / args.steps},
            "kernels": {"gemm_ms_per_step": gemm_ms / args.steps, "attn_prefill_ms_per_step": att_ms / args.steps,
                        "attn_prefill_tflops": att_flops / (att_ms / args.steps * 1e-3) / 1e12 if att_ms else None},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_prefill70(args):
    """One 70B-shaped layer, causal prefill of 4096 tokens at batch 1 (the
    prefill half of the 70B-layer workload), for profiling the prefill GEMMs
    and attention at that size."""
    import torch
    import __graft_entry__
    from llama2_decoder_forward_gb300 import binding, synth

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    __graft_entry__.build()
    s70 = synth.LLAMA2_70B.with_(n_layers=1)
    g = torch.Generator(device=dev)
    g.manual_seed(1002)

    def rn(*s, std=0.01, mean=0.0):
        t = torch.randn(*s, generator=g, device=dev, dtype=torch.float32)
        return t.mul_(std).add_(mean).to(torch.bfloat16)

    H, I, T = s70.hidden, s70.intermediate, 4096
    w = {"layers": [{"attn_norm": rn(H, std=0.1, mean=1.0), "wqkv": rn(s70.qkv_rows, H),
                     "wo": rn(H, H), "ffn_norm": rn(H, std=0.1, mean=1.0), "w_gate": rn(I, H),
                     "w_up": rn(I, H), "w_down": rn(H, I)}]}
    stream = torch.cuda.Stream(device=dev)
    m = binding.Model(s70, w, max_batch=1, max_tokens=T, max_seq=T + 16, has_embed_head=False,
                      stream=stream)
    kv = binding.KVCache(s70, batch=1, capacity=T + 16)
    x = torch.randn(T, H, generator=g, device=dev)
    hbm, tflops, peak_kind = _peaks()
    with Clocks(0) as clk:
        r = prefill_70b_layer_numbers(m, x, kv, stream, tflops, steps=args.steps)
    line = {"metric": "Llama2-70B layer prefill tokens/s (4096 tokens)", "value": r["tokens_per_s"],
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": 3, "ms_per_step": r["ms"],
            "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": "one llama2-70b layer, causal prefill of 4096 tokens"},
            "kernels": r, "peak_tflops": tflops, "peak_source": peak_kind, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_extend(args):
    """One continuous-batching step on the full 7B model: 28 sequences decode
    one token at position 1024 while 4 others feed a 256-token prompt piece
    at positions 512..767, all in one llama_extend call (1052 rows)."""
    import torch
    import __graft_entry__
    from llama2_decoder_forward_gb300 import binding, synth

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    __graft_entry__.build()
    n_dec, n_pre, piece, ctx, pstart, cap = 28, 4, 256, 1024, 512, 1040
    B = n_dec + n_pre
    shape = synth.LLAMA2_7B
    g = torch.Generator(device=dev)
    g.manual_seed(1005)

    def rn(*s, std=0.02, mean=0.0):
        t = torch.randn(*s, generator=g, device=dev, dtype=torch.float32)
        return t.mul_(std).add_(mean).to(torch.bfloat16)

    H, I, V = shape.hidden, shape.intermediate, shape.vocab
    w = {"layers": [{"attn_norm": rn(H, std=0.1, mean=1.0), "wqkv": rn(shape.qkv_rows, H), "wo": rn(H, H),
                     "ffn_norm": rn(H, std=0.1, mean=1.0), "w_gate": rn(I, H), "w_up": rn(I, H),
                     "w_down": rn(H, I)} for _ in range(shape.n_layers)],
         "embed": rn(V, H), "final_norm": rn(H, std=0.1, mean=1.0), "lm_head": rn(V, H)}
    counts = [1] * n_dec + [piece] * n_pre
    starts = [ctx] * n_dec + [pstart] * n_pre
    rows = sum(counts)
    model = binding.Model(shape, w, max_batch=B, max_tokens=rows, max_seq=cap)
    kv = binding.KVCache(shape, batch=B, capacity=cap)
    kv.k.normal_(generator=g)
    kv.v.normal_(generator=g)
    tokens = torch.randint(0, V, (rows,), generator=g, device=dev, dtype=torch.int32)
    cu = torch.tensor([0] + [sum(counts[:i + 1]) for i in range(B)], dtype=torch.int32, device=dev)
    st = torch.tensor(starts, dtype=torch.int32, device=dev)
    logits = torch.empty(B, V, device=dev)
    ids = torch.empty(B, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    def step():
        model.extend(tokens, cu, st, kv, logits, ids, max_rows=piece)

    for _ in range(args.warmup):
        step()
    model.sync()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(0) as clk:
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    model.profile(["gemm", "attn_prefill", "attn_decode"])
    for _ in range(args.steps):
        step()
    gemm_ms, gemm_n = model.profile_read("gemm")
    att_ms, att_n = model.profile_read("attn_prefill")
    dec_ms, dec_n = model.profile_read("attn_decode")
    model.profile([])
    model.sync()
    layer_params = shape.qkv_rows * H + H * H + 3 * H * I
    gemm_flops = 2.0 * rows * layer_params * shape.n_layers + 2.0 * B * V * H
    keys = n_pre * sum(pstart + i + 1 for i in range(piece))  # rows of the prompt pieces
    att_bytes = n_dec * (ctx + 1) * shape.n_kv_heads * shape.head_dim * 4 * shape.n_layers
    hbm, tflops, peak_kind = _peaks()
    g_tf = gemm_flops / (gemm_ms / args.steps * 1e-3) / 1e12
    line = {"metric": "Llama2-7B continuous-batching step tokens/s (28 decode + 4 x 256-token prompt pieces)",
            "value": rows / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init 7B weights, uniform ids, N(0,1) cache)",
            "config": {"workload": "llama2-7b extend step: 28 sequences decode at position 1024, 4 feed "
                                   "256-token prompt pieces at positions 512..767; one call, 1052 rows"},
            "roofline": {"kernel": "gemm_tm_kernel (Q/K/V, gate/up) + gemm_tc_kernel (O, down, LM head)",
                         "bound": "tensor",
                         "achieved": g_tf, "peak": tflops, "unit": "TFLOP/s", "frac": g_tf / tflops,
                         "peak_source": peak_kind, "traffic": None,
                         "algorithmic_flops_per_step": gemm_flops, "launches_per_step": gemm_n / args.steps},
            "kernels": {"gemm_ms_per_step": gemm_ms / args.steps,
                        "piece_attn_ms_per_step": att_ms / args.steps,
                        "piece_attn_tflops": 4.0 * shape.n_q_heads * shape.head_dim * keys * shape.n_layers
                        / (att_ms / args.steps * 1e-3) / 1e12 if att_ms else None,
                        "decode_attn_ms_per_step": dec_ms / args.steps,
                        "decode_attn_gbs": att_bytes / (dec_ms / args.steps * 1e-3) / 1e9 if dec_ms else None},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- CPU oracle arm
class OracleStep:
    """The oracle's whole decode step on `n_seq` of the 32 sequences. Model
    workload: the embedding, all 32 decoder layers (each a full fp64
    layer_decode over a 1024-position cache), the final RMSNorm, the LM head
    and the greedy choice; layer workload: one layer_decode on a hidden
    input. One layer's fp64 weights and one layer's cache serve every layer
    call (32 distinct fp64 layers would need 52 GB of host memory; the
    arithmetic of each call is the same). Inputs are drawn once; only the
    oracle's arithmetic is timed."""

    def __init__(self, n_seq, workload="model"):
        import numpy as np
        import torch
        from llama2_decoder_forward_gb300 import synth
        from oracle import llama_oracle as O

        self.O = O
        self.n_seq = n_seq
        self.model = workload == "model"
        self.shape = shape = synth.LLAMA2_7B if self.model else synth.LLAMA2_7B.with_(n_layers=1)
        one = shape.with_(n_layers=1)
        self.lw = {k: O.as64(v) for k, v in synth.layer_weights(one, 1003, 0).items()}
        self.K = O.as64(synth.cache_values((n_seq, shape.n_kv_heads, CTX + 1, shape.head_dim), 1003,
                                           torch.bfloat16, stream=0))
        self.V = O.as64(synth.cache_values((n_seq, shape.n_kv_heads, CTX + 1, shape.head_dim), 1003,
                                           torch.bfloat16, stream=1))
        self.pos = np.full(n_seq, CTX)
        if self.model:
            g = torch.Generator().manual_seed(5)
            rn = lambda *s: O.as64((torch.randn(*s, generator=g) * 0.02).to(torch.bfloat16))
            self.embed = rn(shape.vocab, shape.hidden)
            self.lm = rn(shape.vocab, shape.hidden)
            self.fn = self.lw["ffn_norm"]
            self.tokens = synth.token_ids(1, n_seq, shape.vocab, 1003).numpy()[0]
            self.desc = ("the fp64 oracle's whole decode step (embedding, 32 layer decodes over "
                         "1024 cached positions, final norm, LM head, greedy) for %d of the 32 "
                         "sequences" % n_seq)
        else:
            self.x = O.as64(synth.hidden_input(n_seq, shape.hidden, 1003))
            self.desc = ("the fp64 oracle's decode step of one 7B layer over 1024 cached "
                         "positions for %d of the 32 sequences" % n_seq)

    def step_seconds(self):
        O = self.O
        t0 = time.perf_counter()
        h = O.embed(self.embed, self.tokens) if self.model else self.x
        for _ in range(self.shape.n_layers):
            h = O.layer_decode(h, self.lw, self.shape, self.K, self.V, self.pos)
        if self.model:
            O.greedy(O.lm_head(h, self.fn, self.lm, self.shape.rms_eps))
        return time.perf_counter() - t0


def _cores():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name") or line.startswith("CPU part"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _single_thread_seconds(n_seq, workload):
    """One oracle step on one core (BLAS limited to one thread, in a fresh
    process so the limit takes effect before numpy loads)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = "import bench; print(bench.OracleStep(%d, %r).step_seconds())" % (n_seq, workload)
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=300)
        return float(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None


def cpu_baseline(workload):
    """Timed oracle on the host cores beside the GPU number: the whole step
    for all 32 sequences (best of two), plus a one-core step on one sequence."""
    o = OracleStep(B, workload)
    sec = min(o.step_seconds() for _ in range(2))
    st = _single_thread_seconds(1, workload)
    return {"value": B / sec, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
            "cpu_model": _cpu_model(), "step_s": sec,
            "single_thread": {"value": 1.0 / st if st else None, "unit": "tokens/s",
                              "step_s": st, "sample": "the same step for 1 sequence on 1 core"},
            "sample": o.desc + " (best of 2)"}


REF_SEQS = 8  # sequences per reference-arm step: a bounded sample of the batch of 32


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    o = OracleStep(REF_SEQS, args.workload)
    for _ in range(args.warmup):
        o.step_seconds()
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(args.steps):
        total += o.step_seconds()
    ms = total / args.steps * 1e3
    v = REF_SEQS / (ms * 1e-3)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(args.workload), "batch": B, "context": CTX,
                       "kv_cache": "bf16", "weights": "bf16", "parallelism": "CPU oracle, rank 0",
                       "sample": "%d of the %d sequences per step" % (REF_SEQS, B)},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                             "cpu_model": _cpu_model(), "sample": o.desc},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="model",
                    choices=["model", "layer", "prefill", "prefill70", "extend"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=32,
                    help="prefill workload: decoder layers (fewer for a small profiling case)")
    ap.add_argument("--no-graph", action="store_true", help="launch the step's kernels directly")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads timed after the headline step")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "e4m3"],
                    help="KV-cache storage (e4m3: the FP8 cache; not the headline configuration)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "e4m3"],
                    help="projection weights (e4m3: FP8 with row scales; not the headline "
                         "configuration)")
    args = ap.parse_args()
    global B_WORKLOAD
    B_WORKLOAD = args.workload
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "prefill":
        run_prefill(args)
    elif args.workload == "extend":
        run_extend(args)
    elif args.workload == "prefill70":
        run_prefill70(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
