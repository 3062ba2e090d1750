"""Python binding of the C ABI in include/llama_gb300.h.

Argument marshalling only: every step of the forward pass runs in the CUDA
library. PyTorch tensors supply device memory and the stream; their data
pointers go through ctypes. If the shared library is missing the binding
raises at once; there is no other code path.
"""
from __future__ import annotations

import ctypes
import os

from .build import CHECKED_LIB
from .build import LIB as _MAIN_LIB

# LLAMA_GB300_BOUNDS_CHECK=1 selects the bounds-check build of the same sources
LIB = CHECKED_LIB if os.environ.get("LLAMA_GB300_BOUNDS_CHECK") == "1" else _MAIN_LIB

c_int32 = ctypes.c_int32
c_void_p = ctypes.c_void_p

F32, BF16 = 0, 1
EPI_STORE_F32, EPI_RESID_F32, EPI_STORE_T, EPI_SWIGLU = 0, 1, 2, 3
EPI_SPLIT_X = 16  # OR-ed flag: x (and bf16 outputs) in the hi/lo pair layout
KERNELS = ("rmsnorm", "gemm", "rope_append", "attn_decode", "attn_prefill", "embed", "argmax",
           "sample")
FLAG_TOKEN_RANGE, FLAG_POS_RANGE, FLAG_PAGE_RANGE, FLAG_WAIT_TIMEOUT, FLAG_INDEX = 1, 2, 4, 8, 16
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "OUT_OF_RANGE", 4: "CUDA",
          5: "DEVICE_CHECK", 6: "WORKSPACE"}


class LlamaConfig(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("hidden", c_int32), ("n_q_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("intermediate", c_int32),
                ("vocab", c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("dtype", c_int32), ("max_batch", c_int32), ("max_tokens", c_int32),
                ("max_seq", c_int32), ("has_embed_head", c_int32), ("weight_dtype", c_int32)]


LAYER_MATS = ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")
PROJECTIONS = ("wqkv", "wo", "w_gate", "w_up", "w_down")
W_MODEL, W_E4M3 = 0, 1


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in LAYER_MATS] + [(n + "_scale", c_void_p) for n in PROJECTIONS]


class Weights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("final_norm", c_void_p), ("lm_head", c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


class Sampling(ctypes.Structure):
    """llama_sampling: temperature (0 = greedy), top_k (<= 0 off), top_p (1 = off),
    repetition_penalty (1 = off)."""
    _fields_ = [("temperature", ctypes.c_float), ("top_k", c_int32), ("top_p", ctypes.c_float),
                ("repetition_penalty", ctypes.c_float)]


KV_MODEL, KV_E4M3 = 0, 1


class KV(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("page_size", c_int32), ("capacity", c_int32),
                ("batch_capacity", c_int32), ("n_pages", c_int32), ("page_table", c_void_p),
                ("max_pages_per_seq", c_int32), ("kv_dtype", c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


_SIGS = {
    "llama_workspace_bytes": (c_int32, [ctypes.POINTER(LlamaConfig), ctypes.POINTER(ctypes.c_size_t)]),
    "llama_init": (c_int32, [ctypes.POINTER(LlamaConfig), ctypes.POINTER(Weights), c_void_p,
                             ctypes.c_size_t, c_void_p, ctypes.POINTER(c_void_p)]),
    "llama_set_stream": (c_int32, [c_void_p, c_void_p]),
    "llama_prefill": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, ctypes.POINTER(KV), c_void_p,
                                c_void_p]),
    "llama_decode_step": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, ctypes.POINTER(KV),
                                    c_void_p, c_void_p]),
    "llama_decode_step_host": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, ctypes.POINTER(KV),
                                         c_void_p, c_void_p]),
    "llama_prefill_hidden": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, ctypes.POINTER(KV)]),
    "llama_decode_hidden": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, ctypes.POINTER(KV)]),
    "llama_extend": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_int32,
                               ctypes.POINTER(KV), c_void_p, c_void_p]),
    "llama_extend_hidden": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32,
                                      c_int32, ctypes.POINTER(KV)]),
    "llama_graph_capture_decode": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, ctypes.POINTER(KV),
                                             c_void_p, c_void_p, c_int32]),
    "llama_graph_launch": (c_int32, [c_void_p]),
    "llama_sync_status": (c_int32, [c_void_p]),
    "llama_last_device_flags": (ctypes.c_uint32, [c_void_p]),
    "llama_check_wait_timeout": (c_int32, [c_void_p, c_int32]),
    "llama_quantize_rows_e4m3": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_void_p,
                                           c_void_p]),
    "llama_bounds_checked": (c_int32, []),
    "llama_strerror": (ctypes.c_char_p, [c_int32]),
    "llama_free": (c_int32, [c_void_p]),
    "llama_profile_enable": (c_int32, [c_void_p, ctypes.c_uint32]),
    "llama_profile_read": (c_int32, [c_void_p, c_int32, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_int64)]),
    "llama_launch_count": (ctypes.c_int64, [c_void_p]),
    "llama_op_rmsnorm": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p]),
    "llama_op_linear": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_int32,
                                  c_int32, c_void_p]),
    "llama_op_rope_append": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_int32,
                                       ctypes.POINTER(KV), c_void_p, c_void_p, c_void_p]),
    "llama_op_attention_decode": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                            ctypes.POINTER(KV), c_void_p]),
    "llama_attention_decode_noalloc": (c_int32, [ctypes.POINTER(LlamaConfig), c_void_p, c_void_p, c_int32,
                                                 c_int32, ctypes.POINTER(KV), c_void_p, c_void_p]),
    "llama_op_attention_prefill": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                             c_void_p]),
    "llama_op_embed": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p]),
    "llama_op_argmax": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_void_p]),
    "llama_sample": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, ctypes.POINTER(Sampling), c_void_p,
                               c_void_p, c_int32, c_void_p, c_void_p]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("%s is not built (run llama2_decoder_forward_gb300.build."
                               "build_library() or __graft_entry__.build())" % os.path.basename(LIB))
        l = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def exported_symbols():
    return list(_SIGS)


class LlamaError(RuntimeError):
    def __init__(self, rc, what, flags=0):
        self.rc = rc
        self.flags = flags
        msg = "%s failed: %s (%s)" % (what, STATUS.get(rc, rc), lib().llama_strerror(rc).decode())
        if flags:
            msg += " device flags 0x%x" % flags
        super().__init__(msg)


def _p(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def make_config(shape, max_batch, max_tokens, max_seq, has_embed_head=True,
                weight_dtype=W_MODEL) -> LlamaConfig:
    return LlamaConfig(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads,
                       shape.head_dim, shape.intermediate, shape.vocab if has_embed_head else 0,
                       shape.rms_eps, shape.rope_theta, F32 if shape.dtype == "f32" else BF16,
                       max_batch, max_tokens, max_seq, 1 if has_embed_head else 0, weight_dtype)


def quantize_rows_e4m3(w, stream=None):
    """E4M3 codes (uint8 [rows, cols]) and per-row fp32 scales of a bf16 device
    matrix, by the library's quantiser (llama_quantize_rows_e4m3)."""
    import torch
    w = w.contiguous()
    rows, cols = w.shape
    codes = torch.empty(rows, cols, dtype=torch.uint8, device=w.device)
    scales = torch.empty(rows, dtype=torch.float32, device=w.device)
    rc = lib().llama_quantize_rows_e4m3(_p(w), rows, cols, _p(codes), _p(scales),
                                        _stream_handle(stream))
    if rc:
        raise LlamaError(rc, "llama_quantize_rows_e4m3")
    return codes, scales


def quantize_layer_e4m3(lw, stream=None):
    """A layer's weight dict with its five projections as E4M3 codes plus
    "<name>_scale" row scales (norm gains unchanged)."""
    out = dict(lw)
    for n in PROJECTIONS:
        out[n], out[n + "_scale"] = quantize_rows_e4m3(lw[n], stream)
    return out


def workspace_bytes(cfg: LlamaConfig) -> int:
    n = ctypes.c_size_t(0)
    rc = lib().llama_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n))
    if rc:
        raise LlamaError(rc, "llama_workspace_bytes")
    return n.value


class KVCache:
    """Caller-owned KV cache in the library's layout (torch device memory).

    contiguous: k, v [n_layers, batch, n_kv, capacity, d]
    paged     : k, v [n_layers, n_pages, n_kv, page_size, d] + page_table [B, max_pages] int32
    e4m3=(k_scale, v_scale): one FP8 E4M3 byte per value (uint8 tensors), read
    back as e4m3 * scale.
    """

    def __init__(self, shape, *, batch=None, capacity=None, n_pages=None, page_size=0,
                 page_table=None, dtype=None, device="cuda", k=None, v=None, e4m3=None):
        import torch
        self.kv_dtype = KV_E4M3 if e4m3 else KV_MODEL
        self.k_scale, self.v_scale = e4m3 if e4m3 else (1.0, 1.0)
        dt = torch.uint8 if e4m3 else (dtype or shape.torch_dtype)
        L, nkv, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
        self.page_size = page_size
        self.page_table = page_table
        if page_size == 0:
            full = (L, batch, nkv, capacity, d)
            self.batch, self.capacity, self.n_pages, self.max_pages = batch, capacity, 0, 0
        else:
            full = (L, n_pages, nkv, page_size, d)
            self.batch, self.capacity, self.n_pages = 0, 0, n_pages
            self.max_pages = page_table.shape[1]
        self.k = k if k is not None else torch.zeros(full, dtype=dt, device=device)
        self.v = v if v is not None else torch.zeros(full, dtype=dt, device=device)
        assert tuple(self.k.shape) == full and tuple(self.v.shape) == full

    def struct(self) -> KV:
        return KV(self.k.data_ptr(), self.v.data_ptr(), self.page_size, self.capacity, self.batch,
                  self.n_pages, None if self.page_table is None else self.page_table.data_ptr(),
                  self.max_pages, self.kv_dtype, self.k_scale, self.v_scale)


class Model:
    """A library context over device-resident weights.

    weights: dict as produced by synth.model_weights / layer_weights, already
    on the GPU ({"embed", "final_norm", "lm_head", "layers": [...]}); a
    layer-only model passes {"layers": [...]} and has_embed_head=False.
    Layers made by quantize_layer_e4m3 (E4M3 projections with row scales)
    select weight_dtype LLAMA_W_E4M3.
    """

    def __init__(self, shape, weights, *, max_batch, max_tokens, max_seq, has_embed_head=True,
                 stream=None):
        import torch
        self.shape = shape
        self.weights = weights  # keep the tensors alive
        layers = weights["layers"]
        if len(layers) != shape.n_layers:
            raise ValueError("shape has %d layers, weights have %d" % (shape.n_layers, len(layers)))
        # E4M3 projections (quantize_layer_e4m3) carry "<name>_scale" entries
        w8 = "wqkv_scale" in layers[0]
        self.cfg = make_config(shape, max_batch, max_tokens, max_seq, has_embed_head,
                               W_E4M3 if w8 else W_MODEL)
        nbytes = workspace_bytes(self.cfg)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        arr = (LayerWeights * len(layers))()
        for i, lw in enumerate(layers):
            scales = [lw[n + "_scale"].data_ptr() if w8 else None for n in PROJECTIONS]
            arr[i] = LayerWeights(*([lw[n].data_ptr() for n in LAYER_MATS] + scales))
        self._layers_arr = arr
        w = Weights(_p(weights.get("embed")), _p(weights.get("final_norm")), _p(weights.get("lm_head")),
                    ctypes.cast(arr, ctypes.POINTER(LayerWeights)))
        ctx = c_void_p()
        rc = lib().llama_init(ctypes.byref(self.cfg), ctypes.byref(w), _p(self.workspace), nbytes,
                              _stream_handle(stream), ctypes.byref(ctx))
        if rc:
            raise LlamaError(rc, "llama_init")
        self.ctx = ctx

    def __del__(self):
        ctx = getattr(self, "ctx", None)
        if ctx is not None and _lib is not None:
            _lib.llama_free(ctx)
            self.ctx = None

    def _chk(self, rc, what):
        if rc:
            raise LlamaError(rc, what)

    def set_stream(self, stream):
        self._chk(lib().llama_set_stream(self.ctx, _stream_handle(stream)), "llama_set_stream")

    # ---- forward pass
    def prefill(self, tokens, kv: KVCache, logits, next_ids=None):
        B, T = tokens.shape
        self._chk(lib().llama_prefill(self.ctx, _p(tokens), B, T, ctypes.byref(kv.struct()),
                                      _p(logits), _p(next_ids)), "llama_prefill")

    def extend(self, tokens, cu_rows, start_pos, kv: KVCache, logits, next_ids=None,
               max_rows=None):
        """Continuous-batching step (llama_extend): tokens [n_rows] packed by
        cu_rows [B+1] (device int32), sequence b's first row at start_pos[b]."""
        B = start_pos.shape[0]
        if max_rows is None:
            max_rows = int((cu_rows[1:] - cu_rows[:-1]).max())
        self._chk(lib().llama_extend(self.ctx, _p(tokens), tokens.shape[0], _p(cu_rows),
                                     _p(start_pos), B, max_rows, ctypes.byref(kv.struct()),
                                     _p(logits), _p(next_ids)), "llama_extend")

    def extend_hidden(self, hidden, cu_rows, start_pos, kv: KVCache, max_rows=None):
        B = start_pos.shape[0]
        if max_rows is None:
            max_rows = int((cu_rows[1:] - cu_rows[:-1]).max())
        self._chk(lib().llama_extend_hidden(self.ctx, _p(hidden), hidden.shape[0], _p(cu_rows),
                                            _p(start_pos), B, max_rows,
                                            ctypes.byref(kv.struct())), "llama_extend_hidden")

    def decode_step(self, tokens, positions, kv: KVCache, logits, next_ids=None):
        self._chk(lib().llama_decode_step(self.ctx, _p(tokens), _p(positions), tokens.shape[0],
                                          ctypes.byref(kv.struct()), _p(logits), _p(next_ids)),
                  "llama_decode_step")

    def decode_step_host(self, tokens, positions, kv: KVCache, logits=None, next_ids=None):
        rc = lib().llama_decode_step_host(self.ctx, _p(tokens), _p(positions), tokens.shape[0],
                                          ctypes.byref(kv.struct()), _p(logits), _p(next_ids))
        if rc:
            raise LlamaError(rc, "llama_decode_step_host", lib().llama_last_device_flags(self.ctx))

    def capture_decode(self, tokens, positions, kv: KVCache, logits, next_ids=None, advance=False):
        """Capture one decode step into a CUDA graph (the context's stream must be a
        non-default stream, see set_stream). Keep the buffers alive while replaying."""
        self._graph_args = (tokens, positions, kv, logits, next_ids)
        self._graph_kv = kv.struct()
        self._chk(lib().llama_graph_capture_decode(self.ctx, _p(tokens), _p(positions), tokens.shape[0],
                                                   ctypes.byref(self._graph_kv), _p(logits),
                                                   _p(next_ids), 1 if advance else 0),
                  "llama_graph_capture_decode")

    def graph_launch(self):
        self._chk(lib().llama_graph_launch(self.ctx), "llama_graph_launch")

    def prefill_hidden(self, hidden, B, T, kv: KVCache):
        self._chk(lib().llama_prefill_hidden(self.ctx, _p(hidden), B, T, ctypes.byref(kv.struct())),
                  "llama_prefill_hidden")

    def decode_hidden(self, hidden, positions, kv: KVCache):
        self._chk(lib().llama_decode_hidden(self.ctx, _p(hidden), _p(positions), hidden.shape[0],
                                            ctypes.byref(kv.struct())), "llama_decode_hidden")

    def sync(self):
        """Synchronise; raise LlamaError carrying the device flags on a kernel-side check."""
        rc = lib().llama_sync_status(self.ctx)
        if rc:
            raise LlamaError(rc, "llama_sync_status", lib().llama_last_device_flags(self.ctx))

    def sync_status(self):
        rc = lib().llama_sync_status(self.ctx)
        return rc, lib().llama_last_device_flags(self.ctx)

    def check_wait_timeout(self, limit_us):
        """Enqueue the bounded-wait check (a wait that runs out after limit_us)."""
        self._chk(lib().llama_check_wait_timeout(self.ctx, int(limit_us)), "llama_check_wait_timeout")

    # ---- profiling
    def profile(self, kinds):
        mask = 0
        for k in kinds:
            mask |= 1 << KERNELS.index(k)
        self._chk(lib().llama_profile_enable(self.ctx, mask), "llama_profile_enable")

    def profile_read(self, kind):
        ms = ctypes.c_double()
        n = ctypes.c_int64()
        self._chk(lib().llama_profile_read(self.ctx, KERNELS.index(kind), ctypes.byref(ms),
                                           ctypes.byref(n)), "llama_profile_read")
        return ms.value, n.value

    def launch_count(self):
        return lib().llama_launch_count(self.ctx)

    # ---- single operations
    def op_rmsnorm(self, x, gamma, out, rows=None, stride=1, offset=0):
        rows = rows if rows is not None else x.shape[0]
        self._chk(lib().llama_op_rmsnorm(self.ctx, _p(x), rows, stride, offset, _p(gamma), _p(out)),
                  "llama_op_rmsnorm")

    def op_linear(self, x, w, out, epilogue, w_up=None, n_rows=None):
        """n_rows: logical activation rows (defaults to x.shape[0]; give it for the
        hi/lo pair layout, whose tensor has 2 * round16(n_rows) rows)."""
        M, K = w.shape
        n = x.shape[0] if n_rows is None else n_rows
        self._chk(lib().llama_op_linear(self.ctx, _p(x), n, _p(w), _p(w_up), M, K, epilogue,
                                        _p(out)), "llama_op_linear")

    def op_rope_append(self, qkv, rows_per_seq, positions, layer, kv: KVCache, q_out, k_out=None,
                       v_out=None):
        self._chk(lib().llama_op_rope_append(self.ctx, _p(qkv), qkv.shape[0], rows_per_seq,
                                             _p(positions), layer, ctypes.byref(kv.struct()),
                                             _p(q_out), _p(k_out), _p(v_out)), "llama_op_rope_append")

    def op_attention_decode(self, q, positions, layer, kv: KVCache, out):
        self._chk(lib().llama_op_attention_decode(self.ctx, _p(q), _p(positions), q.shape[0], layer,
                                                  ctypes.byref(kv.struct()), _p(out)),
                  "llama_op_attention_decode")

    def op_attention_prefill(self, q, k, v, B, T, out):
        self._chk(lib().llama_op_attention_prefill(self.ctx, _p(q), _p(k), _p(v), B, T, _p(out)),
                  "llama_op_attention_prefill")

    def op_embed(self, tokens, out):
        self._chk(lib().llama_op_embed(self.ctx, _p(tokens), tokens.numel(), _p(out)), "llama_op_embed")

    def op_argmax(self, logits, ids):
        B, V = logits.shape
        self._chk(lib().llama_op_argmax(self.ctx, _p(logits), B, V, _p(ids)), "llama_op_argmax")

    def sample(self, logits, uniforms, next_ids, *, temperature=1.0, top_k=0, top_p=1.0,
               repetition_penalty=1.0, history=None, history_len=None):
        """Draw next_ids[b] from logits[b] (see llama_sample). history: [B, S] int32
        device ids and history_len: [B] int32 counts, or None."""
        sp = Sampling(temperature, top_k, top_p, repetition_penalty)
        stride = history.shape[1] if history is not None else 0
        self._chk(lib().llama_sample(self.ctx, _p(logits), logits.shape[0], logits.shape[1],
                                     ctypes.byref(sp),
                                     _p(history), _p(history_len), stride, _p(uniforms),
                                     _p(next_ids)), "llama_sample")
