"""Device-side plumbing around libg4: upload host weights with PyTorch, hold the borrowed
tensors alive, and marshal calls.  No decoder arithmetic happens here."""
import ctypes

import numpy as np
import torch

from . import g4 as _g4


def _dev(a, device):
    """Host numpy array (any integer dtype) -> CUDA tensor of the same bytes."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(device, non_blocking=False)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def stream_handle(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Decoder:
    """One libg4 handle.  `weights` is a host weight dict in the canonical format (synth).
    kv_format "bf16" or "int8" (cache rows); kv_page_size 0 (static rows) or a power of two
    (paged cache of kv_pages pages, 0 = as many as static rows would take).  Vocabulary
    tables given as int4 dicts (packed, scales) select the int4 table format."""

    def __init__(self, cfg, weights, max_batch, max_context, device=0, kv_format="bf16", kv_page_size=0,
                 kv_pages=0):
        t4 = [isinstance(weights[k], dict) for k in ("embed", "ple_table")]
        if t4[0] != t4[1]:
            raise ValueError("the token embedding and the per-layer table share one table format")
        self.cfg = cfg
        self.device = torch.device("cuda", device)
        self.max_batch, self.max_context = max_batch, max_context
        self.fmt = weights["fmt"]
        self.table_format = "w4a16" if t4[0] else "bf16"
        self.c = _g4.make_config(cfg, self.fmt, max_batch, max_context, kv_format, kv_page_size, kv_pages,
                                 self.table_format)
        keep, tmp = [], []

        def borrow(a):
            t = _dev(a, self.device)
            keep.append(t)
            return _ptr(t)

        def linear(x):
            lin = _g4.g4_linear()
            if "w" in x:
                t = _dev(x["w"], self.device)
                tmp.append(t)
                lin.w = t.data_ptr()
            else:
                t = _dev(x["packed"], self.device)
                s = _dev(x["scales"], self.device)
                tmp.extend([t, s])
                lin.w, lin.scales = t.data_ptr(), s.data_ptr()
            return lin

        L = cfg["num_layers"]
        layers = (_g4.g4_layer_weights * L)()
        for l, lw in enumerate(weights["layers"]):
            for n in _g4.LINEAR_NAMES:
                setattr(layers[l], n, linear(lw[n]))
            for n in _g4.NORM_NAMES:
                setattr(layers[l], n, borrow(lw[n]))
            layers[l].layer_scale = float(lw["layer_scale"])
        w = _g4.g4_weights()
        if self.table_format == "w4a16":
            w.embed = borrow(weights["embed"]["packed"])
            w.embed_scales = borrow(weights["embed"]["scales"])
            w.ple_table = borrow(weights["ple_table"]["packed"])
            w.ple_table_scales = borrow(weights["ple_table"]["scales"])
        else:
            w.embed = borrow(weights["embed"])
            w.ple_table = borrow(weights["ple_table"])
        w.ple_model_proj = linear(weights["ple_model_proj"])
        w.ple_proj_norm = borrow(weights["ple_proj_norm"])
        w.final_norm = borrow(weights["final_norm"])
        w.layers = layers
        torch.cuda.synchronize(self.device)
        self.h = _g4.g4_create(self.c, w, device)
        del tmp                         # linears were copied into the library's layout
        self._keep = keep               # embed, per-layer table and gains are borrowed
        self._trace = None
        torch.cuda.empty_cache()

    # -- calls -------------------------------------------------------------------------------
    def prefill(self, slots, prompts, start_pos=None, stream=None, want_logits=False):
        """prompts: list of host int arrays.  Returns (next ids [n] int32, logits [n, V] or None),
        both device tensors (valid after the stream synchronises)."""
        n = len(prompts)
        lens = [len(p) for p in prompts]
        offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        toks = torch.from_numpy(np.concatenate([np.asarray(p, np.int32) for p in prompts])).to(self.device)
        nxt = torch.empty(n, dtype=torch.int32, device=self.device)
        logits = torch.empty(n, self.cfg["vocab"], dtype=torch.float32, device=self.device) if want_logits else None
        start = [0] * n if start_pos is None else list(start_pos)
        _g4.g4_prefill(self.h, stream_handle(stream), list(slots), offsets.tolist(), start, _ptr(toks),
                       _ptr(nxt), _ptr(logits))
        self._last_prefill_tokens = toks   # keep alive until the stream runs
        return nxt, logits

    def decode_step(self, d_slots, d_tokens, d_positions, d_next, d_logits=None, stream=None):
        n = d_tokens.numel()
        _g4.g4_decode_step(self.h, stream_handle(stream), n, _ptr(d_slots), _ptr(d_tokens), _ptr(d_positions),
                           _ptr(d_next), _ptr(d_logits))

    def profile_step(self, d_slots, d_tokens, d_positions, d_next, d_logits=None, repeats=1, stream=None):
        return _g4.g4_profile_step(self.h, stream_handle(stream), d_tokens.numel(), _ptr(d_slots), _ptr(d_tokens),
                                   _ptr(d_positions), _ptr(d_next), _ptr(d_logits), repeats)

    def reserve(self, slot, n_positions, stream=None):
        """Paged cache: pages for positions [0, n_positions) of `slot` (no-op when static)."""
        _g4.g4_kv_reserve(self.h, stream_handle(stream), int(slot), int(n_positions))

    def release(self, slot, stream=None):
        """Paged cache: return the slot's pages to the pool."""
        _g4.g4_kv_release(self.h, stream_handle(stream), int(slot))

    def pages_free(self):
        return _g4.g4_kv_pages_free(self.h)

    def device_error(self, stream=None):
        return _g4.g4_get_device_error(self.h, stream_handle(stream))

    def set_trace(self, enable):
        c = self.cfg
        stride = max(c["hidden"], c["num_q_heads"] * max(c["head_dim_full"], c["head_dim_sliding"]))
        if enable:
            self._trace = torch.zeros(c["num_layers"], 2, self.max_batch, stride, dtype=torch.float32,
                                      device=self.device)
            _g4.g4_set_trace(self.h, _ptr(self._trace), self._trace.numel())
        else:
            _g4.g4_set_trace(self.h, None, 0)
            self._trace = None
        return self._trace

    def step_mode(self, n_seq=1):
        """1: persistent single-launch step; 0: one launch per phase."""
        return _g4.lib.g4_step_mode(self.h, n_seq)

    def set_step_mode(self, mode):
        """0 (default): one launch per phase; 1: persistent single-launch step for n_seq <= 2."""
        _g4.g4_set_step_mode(self.h, int(mode))

    def device_bytes(self):
        return _g4.lib.g4_device_bytes(self.h)

    def close(self):
        if getattr(self, "h", None) is not None:
            _g4.g4_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LinearOp:
    """Standalone projection kernel (the decode step's GEMV) on one weight matrix."""

    def __init__(self, fmt, lin, device=0):
        self.device = torch.device("cuda", device)
        n_out, n_in = lin["shape"]
        self.n_out, self.n_in = n_out, n_in
        if fmt == "bf16":
            w = _dev(lin["w"], self.device)
            s = None
        else:
            w = _dev(lin["packed"], self.device)
            s = _dev(lin["scales"], self.device)
        h = ctypes.c_void_p()
        st = _g4.lib.g4_linear_create(device, _g4.G4_W4A16 if fmt == "w4a16" else _g4.G4_BF16, n_out, n_in,
                                      _ptr(w), _ptr(s), ctypes.byref(h))
        _g4.check(st, "g4_linear_create")
        self.h = h

    def __call__(self, x, stream=None):
        y = torch.empty(x.shape[0], self.n_out, dtype=torch.float32, device=self.device)
        _g4.check(_g4.lib.g4_linear_forward(self.h, stream_handle(stream), x.shape[0], _ptr(x), _ptr(y)),
                  "g4_linear_forward")
        return y

    def close(self):
        if getattr(self, "h", None) is not None:
            _g4.lib.g4_linear_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def argmax_rows(logits, stream=None):
    ids = torch.empty(logits.shape[0], dtype=torch.int32, device=logits.device)
    _g4.check(_g4.lib.g4_argmax_rows(logits.device.index, stream_handle(stream), logits.shape[0],
                                     logits.shape[1], _ptr(logits), _ptr(ids)), "g4_argmax_rows")
    return ids


def argmax_rows_static(logits, stream=None):
    """Allocation-free row argmax (fixed scratch inside the library; see include/g4.h)."""
    ids = torch.empty(logits.shape[0], dtype=torch.int32, device=logits.device)
    _g4.check(_g4.lib.g4_argmax_rows_static(logits.device.index, stream_handle(stream), logits.shape[0],
                                            logits.shape[1], _ptr(logits), _ptr(ids)), "g4_argmax_rows_static")
    return ids
