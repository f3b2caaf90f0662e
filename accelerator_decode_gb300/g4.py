"""ctypes binding of libg4 (include/g4.h): the same entry points, argument marshalling only.

Every step of the decode runs in libg4's CUDA kernels; PyTorch only provides device memory
and streams.  There is no fallback: if libg4.so is missing or fails to load, importing the
binding raises.
"""
import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_int64, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libg4.so")

G4_OK = 0
G4_ERR_INVALID_ARG = -1
G4_ERR_UNSUPPORTED = -2
G4_ERR_OOM = -3
G4_ERR_CUDA = -4
G4_ERR_CONTEXT_OVERFLOW = -5
G4_ERR_TIMEOUT = -6
G4_ERR_DEVICE_CHECK = -7
G4_BF16 = 0
G4_W4A16 = 1
G4_KV_BF16 = 0
G4_KV_INT8 = 1
G4_DEV_BAD_TOKEN = 1
G4_DEV_BAD_POSITION = 2
G4_DEV_TIMEOUT = 4
G4_DEV_BAD_SLOT = 8

_INT_FIELDS = ("num_layers", "num_kv_shared_layers", "hidden", "num_q_heads", "num_kv_heads",
               "head_dim_sliding", "head_dim_full", "sliding_window", "full_every", "mlp",
               "mlp_shared", "ple_dim", "vocab", "max_batch", "max_context", "weight_format",
               "group_size")
_FLOAT_FIELDS = ("rms_eps", "rope_theta_sliding", "rope_theta_full", "attn_scale_sliding",
                 "attn_scale_full")
_TAIL_FIELDS = ("kv_format", "kv_page_size", "kv_pages", "table_format")
LINEAR_NAMES = ("q", "k", "v", "o", "gate", "up", "down", "ple_gate", "ple_proj")
NORM_NAMES = ("in_norm", "post_attn_norm", "pre_ffw_norm", "post_ffw_norm", "post_ple_norm",
              "q_norm", "k_norm")


class g4_config(ctypes.Structure):
    _fields_ = ([(n, c_int32) for n in _INT_FIELDS] + [(n, c_float) for n in _FLOAT_FIELDS]
                + [(n, c_int32) for n in _TAIL_FIELDS])


class g4_linear(ctypes.Structure):
    _fields_ = [("w", c_void_p), ("scales", c_void_p)]


class g4_layer_weights(ctypes.Structure):
    _fields_ = ([(n, g4_linear) for n in LINEAR_NAMES] + [(n, c_void_p) for n in NORM_NAMES]
                + [("layer_scale", c_float)])


class g4_weights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("ple_table", c_void_p), ("ple_model_proj", g4_linear),
                ("ple_proj_norm", c_void_p), ("final_norm", c_void_p),
                ("layers", POINTER(g4_layer_weights)), ("embed_scales", c_void_p),
                ("ple_table_scales", c_void_p)]


class g4_phase_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", c_int32), ("ms_total", ctypes.c_double),
                ("bytes_total", ctypes.c_double)]


class G4Error(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = f"{where}: {status_string(status)} ({status})"
        cuda = last_cuda_error()
        if cuda:
            msg += f"; {cuda}"
        super().__init__(msg)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libg4.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                          "or python -m accelerator_decode_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    sigs = {
        "g4_create": (c_int, [POINTER(g4_config), POINTER(g4_weights), c_int, POINTER(P)]),
        "g4_prefill": (c_int, [P, P, c_int32, POINTER(c_int32), POINTER(c_int32), POINTER(c_int32),
                               P, P, P]),
        "g4_decode_step": (c_int, [P, P, c_int32, P, P, P, P, P]),
        "g4_get_device_error": (c_int, [P, P, POINTER(c_int32)]),
        "g4_set_trace": (c_int, [P, P, c_int64]),
        "g4_device_bytes": (c_int64, [P]),
        "g4_step_mode": (c_int32, [P, c_int32]),
        "g4_set_step_mode": (c_int, [P, c_int32]),
        "g4_profile_step": (c_int, [P, P, c_int32, P, P, P, P, P, c_int32, POINTER(g4_phase_stat), c_int32,
                                    POINTER(c_int32)]),
        "g4_free": (None, [P]),
        "g4_kv_reserve": (c_int, [P, P, c_int32, c_int32]),
        "g4_timeout_probe": (c_int, [P, P, c_int64]),
        "g4_kv_release": (c_int, [P, P, c_int32]),
        "g4_kv_pages_free": (c_int32, [P]),
        "g4_status_string": (ctypes.c_char_p, [c_int]),
        "g4_last_cuda_error": (ctypes.c_char_p, []),
        "g4_linear_create": (c_int, [c_int, c_int32, c_int32, c_int32, P, P, POINTER(P)]),
        "g4_linear_forward": (c_int, [P, P, c_int32, P, P]),
        "g4_linear_free": (None, [P]),
        "g4_argmax_rows": (c_int, [c_int, P, c_int32, c_int32, P, P]),
        "g4_argmax_rows_static": (c_int, [c_int, P, c_int32, c_int32, P, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(s):
    return lib.g4_status_string(s).decode()


def last_cuda_error():
    return lib.g4_last_cuda_error().decode()


def check(status, where):
    if status != G4_OK:
        raise G4Error(status, where)


def make_config(cfg, weight_format, max_batch, max_context, kv_format="bf16", kv_page_size=0, kv_pages=0,
                table_format="bf16"):
    c = g4_config()
    c.kv_format = G4_KV_INT8 if kv_format == "int8" else G4_KV_BF16
    c.kv_page_size = int(kv_page_size)
    c.kv_pages = int(kv_pages)
    c.table_format = G4_W4A16 if table_format == "w4a16" else G4_BF16
    for n in _INT_FIELDS:
        if n == "weight_format":
            c.weight_format = G4_W4A16 if weight_format == "w4a16" else G4_BF16
        elif n == "max_batch":
            c.max_batch = max_batch
        elif n == "max_context":
            c.max_context = max_context
        else:
            setattr(c, n, int(cfg[n]))
    for n in _FLOAT_FIELDS:
        setattr(c, n, float(cfg[n]))
    return c


# Thin wrappers with the C names -------------------------------------------------------------
def g4_create(cfg_struct, weights_struct, device):
    h = c_void_p()
    check(lib.g4_create(ctypes.byref(cfg_struct), ctypes.byref(weights_struct), device, ctypes.byref(h)),
          "g4_create")
    return h


def g4_prefill(h, stream, slots, offsets, start_pos, d_tokens, d_next_ids, d_logits):
    n = len(slots)
    arr = lambda v: (c_int32 * len(v))(*[int(x) for x in v])
    check(lib.g4_prefill(h, stream, n, arr(slots), arr(offsets), arr(start_pos), d_tokens,
                         d_next_ids, d_logits), "g4_prefill")


def g4_decode_step(h, stream, n_seq, d_slots, d_tokens, d_positions, d_next_ids, d_logits):
    check(lib.g4_decode_step(h, stream, n_seq, d_slots, d_tokens, d_positions, d_next_ids, d_logits),
          "g4_decode_step")


def g4_get_device_error(h, stream):
    w = c_int32(0)
    s = lib.g4_get_device_error(h, stream, ctypes.byref(w))
    return s, w.value


def g4_set_step_mode(h, mode):
    check(lib.g4_set_step_mode(h, mode), "g4_set_step_mode")


def g4_set_trace(h, d_trace, capacity):
    check(lib.g4_set_trace(h, d_trace, capacity), "g4_set_trace")


def g4_profile_step(h, stream, n_seq, d_slots, d_tokens, d_positions, d_next_ids, d_logits, repeats):
    """Per-phase timing: list of dicts(name, launches, ms_total, bytes_total)."""
    arr = (g4_phase_stat * 64)()
    n = c_int32(0)
    check(lib.g4_profile_step(h, stream, n_seq, d_slots, d_tokens, d_positions, d_next_ids, d_logits, repeats,
                              arr, 64, ctypes.byref(n)), "g4_profile_step")
    return [dict(name=arr[i].name.decode(), launches=arr[i].launches, ms_total=arr[i].ms_total,
                 bytes_total=arr[i].bytes_total) for i in range(n.value)]


def g4_kv_reserve(h, stream, slot, n_positions):
    check(lib.g4_kv_reserve(h, stream, slot, n_positions), "g4_kv_reserve")


def g4_kv_release(h, stream, slot):
    check(lib.g4_kv_release(h, stream, slot), "g4_kv_release")


def g4_kv_pages_free(h):
    return lib.g4_kv_pages_free(h)


def g4_free(h):
    lib.g4_free(h)
