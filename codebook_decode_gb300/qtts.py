"""ctypes binding of the C ABI in include/qtts.h, one Python function per C
entry point with the same name. Argument marshalling only: every step of the
frame runs in libqtts.so's CUDA kernels. Raises if the library is missing.

Arrays may be torch tensors (device or host) or numpy arrays (host); the
binding passes their data pointers.
"""
import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqtts.so")

QTTS_OK = 0
QTTS_E_INVALID = -1
QTTS_E_CUDA = -2
QTTS_E_OOM = -3
QTTS_E_MISSING = -4
QTTS_E_UNUSED = -5
QTTS_E_SHAPE = -6
QTTS_E_BATCH = -7
QTTS_E_STATE = -8
QTTS_E_POOL = -9
QTTS_E_DEVICE = -10
QTTS_E_TIMEOUT = -11
(QTTS_DEV_OK, QTTS_DEV_BAD_SESSION, QTTS_DEV_BAD_PAGE, QTTS_DEV_BAD_SAMPLING, QTTS_DEV_BAD_CODE,
 QTTS_DEV_TIMEOUT) = range(6)
QTTS_OPT_STEPWISE = 1
QTTS_OPT_TRACE = 3
QTTS_OPT_RING_SLOTS = 4
QTTS_OPT_TC_MIN_ROWS = 5
QTTS_OPT_KSPLIT_MIN_ROWS = 6
QTTS_OPT_WAIT_LIMIT_US = 7
QTTS_OPT_CHUNK_TALKER_MIN_B = 8


class QttsError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"qtts error {code}: {msg}")
        self.code = code


class Config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab0",
        "cp_hidden", "cp_layers", "cp_n_q_heads", "cp_n_kv_heads", "cp_head_dim", "cp_ffn", "cp_vocab",
        "n_codebooks", "eos_id", "n_codes", "proj_bias")] + [
        ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("cp_rope_theta", C.c_float),
        ("page_size", C.c_int32), ("max_batch", C.c_int32), ("max_context", C.c_int32),
        ("kv_pool_pages", C.c_int32)]


class Tensor(C.Structure):
    _fields_ = [("name", C.c_char_p), ("dtype", C.c_int32), ("ndim", C.c_int32), ("shape", C.c_int64 * 2),
                ("data", C.c_void_p)]


class Session(C.Structure):
    _fields_ = [("kv_len", C.c_int32), ("eos_allowed", C.c_int32), ("temperature", C.c_float),
                ("top_k", C.c_int32), ("rep_penalty", C.c_float), ("cp_temperature", C.c_float),
                ("cp_top_k", C.c_int32), ("reserved", C.c_int32)]


class Rng(C.Structure):
    _fields_ = [("key0", C.c_uint32), ("key1", C.c_uint32), ("frame_ctr", C.c_uint32), ("reserved", C.c_uint32)]


_lib = None
_P = C.c_void_p

# (name, restype, argtypes) of every exported function
SIGNATURES = [
    ("qtts_abi_version", C.c_int, []),
    ("qtts_last_error", C.c_char_p, [_P]),
    ("qtts_create", C.c_int, [C.POINTER(Config), C.c_int, C.POINTER(_P)]),
    ("qtts_destroy", None, [_P]),
    ("qtts_load_weights", C.c_int, [_P, C.POINTER(Tensor), C.c_int]),
    ("qtts_quantize_int8", C.c_int, [_P]),
    ("qtts_set_int8", C.c_int, [_P, C.c_int]),
    ("qtts_export_int8", C.c_int, [_P, C.c_char_p, _P, _P]),
    ("qtts_kv_alloc_pages", C.c_int, [_P, C.c_int, _P]),
    ("qtts_kv_free_pages", C.c_int, [_P, C.c_int, _P]),
    ("qtts_kv_pool_free_count", C.c_int, [_P]),
    ("qtts_kv_write", C.c_int, [_P, C.c_int, C.c_int, _P, _P, _P]),
    ("qtts_kv_read", C.c_int, [_P, C.c_int, C.c_int, _P, _P, _P]),
    ("qtts_kv_write_noalloc", C.c_int, [_P, C.c_int, C.c_int, _P, _P, _P, _P]),
    ("qtts_frame_step", C.c_int, [_P, C.c_int, _P, _P, C.c_int] + [_P] * 8),
    ("qtts_frame_step_host", C.c_int, [_P, C.c_int, _P, _P, C.c_int] + [_P] * 8),
    ("qtts_frame_talker", C.c_int, [_P, C.c_int, _P, _P, C.c_int] + [_P] * 8),
    ("qtts_frame_cp", C.c_int, [_P, C.c_int, _P, _P, C.c_int] + [_P] * 8),
    ("qtts_frame_steps", C.c_int, [_P, C.c_int, C.c_int, _P, _P, C.c_int] + [_P] * 9),
    ("qtts_talker_prefill", C.c_int, [_P, C.c_int, _P, _P, C.c_int, _P, C.c_int, _P]),
    ("qtts_frame_status", C.c_int, [_P, C.POINTER(C.c_int)]),
    ("qtts_feedback_embed", C.c_int, [_P, C.c_int, _P, _P, _P, _P]),
    ("qtts_sample", C.c_int, [_P, C.c_int, C.c_int, _P, C.c_int, _P, _P, _P, _P, _P]),
    ("qtts_set_option", C.c_int, [_P, C.c_int, C.c_int]),
    ("qtts_frame_weight_bytes", C.c_int, [_P, C.POINTER(C.c_int64)]),
    ("qtts_frame_trace", C.c_int, [_P, _P, C.c_int]),
]


def load_library(path=LIB_PATH):
    """Load libqtts.so (built by codebook_decode_gb300.build). Raises if missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: run __graft_entry__.build() first")
        L = C.CDLL(path)
        for name, res, args in SIGNATURES:
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def ptr(a):
    """Data pointer of a torch tensor / numpy array / None."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    return a.ctypes.data


def _check(model, rc):
    if rc != QTTS_OK:
        msg = load_library().qtts_last_error(model)
        raise QttsError(rc, msg.decode() if msg else "")
    return rc


def _stream(s):
    if s is None:
        return None
    return s.cuda_stream if hasattr(s, "cuda_stream") else s


def qtts_abi_version():
    return load_library().qtts_abi_version()


def qtts_create(cfg, device=0):
    m = C.c_void_p()
    _check(None, load_library().qtts_create(C.byref(cfg), device, C.byref(m)))
    return m


def qtts_destroy(m):
    load_library().qtts_destroy(m)


def qtts_load_weights(m, named):
    """named: dict name -> array of bf16 bits (host numpy or torch)."""
    items = list(named.items())
    arr = (Tensor * len(items))()
    keep = []
    for i, (n, a) in enumerate(items):
        b = n.encode()
        keep.append(b)
        shape = tuple(a.shape)
        arr[i].name = b
        arr[i].dtype = 0
        arr[i].ndim = len(shape)
        arr[i].shape[0] = shape[0]
        arr[i].shape[1] = shape[1] if len(shape) > 1 else 0
        arr[i].data = ptr(a)
    return _check(m, load_library().qtts_load_weights(m, arr, len(items)))


def qtts_quantize_int8(m):
    return _check(m, load_library().qtts_quantize_int8(m))


def qtts_set_int8(m, enable):
    return _check(m, load_library().qtts_set_int8(m, int(enable)))


def qtts_export_int8(m, name, q_host, s_host):
    return _check(m, load_library().qtts_export_int8(m, name.encode(), ptr(q_host), ptr(s_host)))


def qtts_kv_alloc_pages(m, ids_host):
    return _check(m, load_library().qtts_kv_alloc_pages(m, len(ids_host), ptr(ids_host)))


def qtts_kv_free_pages(m, ids_host):
    return _check(m, load_library().qtts_kv_free_pages(m, len(ids_host), ptr(ids_host)))


def qtts_kv_pool_free_count(m):
    return load_library().qtts_kv_pool_free_count(m)


def qtts_kv_write(m, layer, n_tok, pages_host, k, v):
    return _check(m, load_library().qtts_kv_write(m, layer, n_tok, ptr(pages_host), ptr(k), ptr(v)))


def qtts_kv_read(m, layer, n_tok, pages_host, k_host, v_host):
    return _check(m, load_library().qtts_kv_read(m, layer, n_tok, ptr(pages_host), ptr(k_host), ptr(v_host)))


def qtts_kv_write_noalloc(m, layer, n_tok, pages_host, k, v, stream=None):
    """qtts_kv_write through the library's static staging array: no device
    allocation, queued on `stream`."""
    return _check(m, load_library().qtts_kv_write_noalloc(m, layer, n_tok, ptr(pages_host), ptr(k), ptr(v),
                                                          _stream(stream)))


def qtts_frame_step(m, B, sessions, block_tables, bt_stride, in_embeds, rng, seen, forced_codes, codes_out,
                    eos_out, logits_out=None, stream=None):
    return _check(m, load_library().qtts_frame_step(
        m, B, ptr(sessions), ptr(block_tables), bt_stride, ptr(in_embeds), ptr(rng), ptr(seen), ptr(forced_codes),
        ptr(codes_out), ptr(eos_out), ptr(logits_out), _stream(stream)))


def qtts_frame_step_host(m, B, sessions, block_tables, bt_stride, in_embeds, rng, seen, forced_codes, codes_out,
                         eos_out, logits_out=None, stream=None):
    return _check(m, load_library().qtts_frame_step_host(
        m, B, ptr(sessions), ptr(block_tables), bt_stride, ptr(in_embeds), ptr(rng), ptr(seen), ptr(forced_codes),
        ptr(codes_out), ptr(eos_out), ptr(logits_out), _stream(stream)))


def qtts_frame_talker(m, B, sessions, block_tables, bt_stride, in_embeds, rng, seen, forced_codes, codes_out,
                      eos_out, logits_out=None, stream=None):
    return _check(m, load_library().qtts_frame_talker(
        m, B, ptr(sessions), ptr(block_tables), bt_stride, ptr(in_embeds), ptr(rng), ptr(seen), ptr(forced_codes),
        ptr(codes_out), ptr(eos_out), ptr(logits_out), _stream(stream)))


def qtts_frame_cp(m, B, sessions, block_tables, bt_stride, in_embeds, rng, seen, forced_codes, codes_out, eos_out,
                  logits_out=None, stream=None):
    return _check(m, load_library().qtts_frame_cp(
        m, B, ptr(sessions), ptr(block_tables), bt_stride, ptr(in_embeds), ptr(rng), ptr(seen), ptr(forced_codes),
        ptr(codes_out), ptr(eos_out), ptr(logits_out), _stream(stream)))


def qtts_frame_steps(m, n_frames, B, sessions, block_tables, bt_stride, in_embeds, text_embeds, rng, seen,
                     forced_codes, codes_out, eos_out, logits_out=None, stream=None):
    return _check(m, load_library().qtts_frame_steps(
        m, n_frames, B, ptr(sessions), ptr(block_tables), bt_stride, ptr(in_embeds), ptr(text_embeds), ptr(rng),
        ptr(seen), ptr(forced_codes), ptr(codes_out), ptr(eos_out), ptr(logits_out), _stream(stream)))


def qtts_talker_prefill(m, B, sessions, block_tables, bt_stride, embeds, n_tok, stream=None):
    return _check(m, load_library().qtts_talker_prefill(
        m, B, ptr(sessions), ptr(block_tables), bt_stride, ptr(embeds), n_tok, _stream(stream)))


def qtts_frame_status(m, raise_on_error=True):
    """Returns (rc, device error word); the word is cleared by the call."""
    e = C.c_int(0)
    rc = load_library().qtts_frame_status(m, C.byref(e))
    if raise_on_error:
        _check(m, rc)
    return rc, e.value


def qtts_feedback_embed(m, B, codes, text, next_out, stream=None):
    return _check(m, load_library().qtts_feedback_embed(m, B, ptr(codes), ptr(text), ptr(next_out),
                                                        _stream(stream)))


def qtts_sample(m, B, codebook, logits, V, sessions, rng, seen, codes_out, stream=None):
    return _check(m, load_library().qtts_sample(m, B, codebook, ptr(logits), V, ptr(sessions), ptr(rng), ptr(seen),
                                                ptr(codes_out), _stream(stream)))


def qtts_set_option(m, option, value):
    return _check(m, load_library().qtts_set_option(m, option, value))


def qtts_frame_weight_bytes(m):
    v = C.c_int64(0)
    _check(m, load_library().qtts_frame_weight_bytes(m, C.byref(v)))
    return v.value


def qtts_frame_trace(m, host_u64):
    """Fill a uint64 numpy array with the last traced frame's stage stamps."""
    n = load_library().qtts_frame_trace(m, ptr(host_u64), len(host_u64))
    if n < 0:
        _check(m, n)
    return n
