"""ctypes binding of ``include/lat.h`` -- argument marshalling only.

Every step of the path runs in ``liblat.so``'s CUDA kernels; this module only
builds the C structs, passes device pointers (``tensor.data_ptr()``) and turns
status codes into exceptions.  There is no fallback: if the library is missing
or no sm_103 GPU is present, calls raise.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblat.so")

LAT_PI0_ACTION_EXPERT, LAT_PI0_PREFIX, LAT_DIT = 0, 1, 2
STATUS = ["LAT_OK", "LAT_ERR_ARG", "LAT_ERR_SHAPE", "LAT_ERR_ALIGN", "LAT_ERR_CUDA", "LAT_ERR_OOM",
          "LAT_ERR_TIMEOUT", "LAT_ERR_STATE", "LAT_ERR_UNSUPPORTED", "LAT_ERR_RANGE"]


class LatError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS[code] if 0 <= code < len(STATUS) else code}: {msg}")
        self.code = code


class ModelDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("kind", "D", "Hq", "Hkv", "dh", "F", "L", "S", "T_prefix", "T_q", "act_dim",
                 "n_hist", "t_dim", "patch_dim", "max_batch", "n_streams")] + \
               [("rope_base", ctypes.c_float), ("eps", ctypes.c_float), ("prefix_lm", ctypes.c_int),
                ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int), ("text_len", ctypes.c_int),
                ("page_tokens", ctypes.c_int)]


_P = ctypes.c_void_p


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("g_attn", "wq", "wk", "wv", "wo", "g_ffn", "wg", "wu", "wd", "w1", "w2",
                                  "g_cross", "b_cross", "cq", "ck", "cv", "co")]


class Weights(ctypes.Structure):
    _fields_ = [("blocks", ctypes.POINTER(BlockWeights))] + \
               [(n, _P) for n in ("w_in", "b_in", "w1", "b1", "w2", "b2", "w_state", "b_state", "g_final",
                                  "w_out", "b_out", "w_patch", "b_patch", "wt1", "bt1", "wt2", "bt2",
                                  "wmod", "bmod")]


class ChunkDesc(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_int), ("chunk", ctypes.c_int), ("step", ctypes.c_int)]


_lib = None


def lib():
    """Load liblat.so (build it first with ``build.build()``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run latency_transformer_block_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        st = ctypes.c_int
        L.lat_create.argtypes = [ctypes.POINTER(ModelDesc), ctypes.POINTER(Weights), ctypes.POINTER(_P)]
        L.lat_create.restype = st
        L.lat_set_schedule.argtypes = [_P, ctypes.POINTER(ctypes.c_float), ctypes.c_int]
        L.lat_set_schedule.restype = st
        L.lat_prefill_kv.argtypes = [_P, _P, ctypes.c_int, _P, _P]
        L.lat_prefill_kv.restype = st
        L.lat_block_forward.argtypes = [_P, ctypes.c_int, _P, ctypes.POINTER(ChunkDesc), ctypes.c_int, _P, _P]
        L.lat_block_forward.restype = st
        L.lat_denoise_chunk.argtypes = [_P, _P, _P, _P, _P]
        L.lat_denoise_chunk.restype = st
        L.lat_debug_indices.argtypes = [_P, ctypes.POINTER(ChunkDesc), ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        L.lat_debug_indices.restype = st
        L.lat_debug_gemm.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
        L.lat_debug_gemm.restype = st
        L.lat_debug_attention.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int, _P]
        L.lat_debug_attention.restype = st
        L.lat_chunk_attention_noalloc.argtypes = [_P, _P, _P, _P] + [ctypes.c_int] * 5 + [_P]
        L.lat_chunk_attention_noalloc.restype = st
        L.lat_debug_dense_gemm.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, _P, _P]
        L.lat_debug_dense_gemm.restype = st
        L.lat_debug_clear.argtypes = [_P, _P]
        L.lat_debug_clear.restype = st
        L.lat_debug_step.argtypes = [_P, _P, ctypes.c_int, _P]
        L.lat_debug_step.restype = st
        L.lat_debug_trace.argtypes = [_P, _P, ctypes.c_longlong]
        L.lat_debug_trace.restype = st
        L.lat_dit_interval.argtypes = [_P, _P, _P, ctypes.POINTER(ChunkDesc), ctypes.c_int, _P]
        L.lat_dit_interval.restype = st
        L.lat_dit_pipeline_push.argtypes = [_P, _P, ctypes.c_int, _P, _P, ctypes.POINTER(ctypes.c_int), _P]
        L.lat_dit_pipeline_push.restype = st
        L.lat_dit_pipeline_reset.argtypes = [_P, ctypes.c_int]
        L.lat_dit_pipeline_reset.restype = st
        L.lat_dit_set_text.argtypes = [_P, ctypes.c_int, _P, _P]
        L.lat_dit_set_text.restype = st
        L.lat_dit_bind_pages.argtypes = [_P, _P]
        L.lat_dit_bind_pages.restype = st
        L.lat_clear_error.argtypes = [_P]
        L.lat_clear_error.restype = st
        L.lat_debug_timeout.argtypes = [_P, _P]
        L.lat_debug_timeout.restype = st
        L.lat_debug_wait_skew.argtypes = [_P, ctypes.c_int, ctypes.c_int]
        L.lat_debug_wait_skew.restype = st
        L.lat_debug_act_terms.argtypes = [_P, ctypes.c_int]
        L.lat_debug_act_terms.restype = st
        L.lat_sync.argtypes = [_P]
        L.lat_sync.restype = st
        L.lat_status_str.argtypes = [ctypes.c_int]
        L.lat_status_str.restype = ctypes.c_char_p
        L.lat_last_error.argtypes = []
        L.lat_last_error.restype = ctypes.c_char_p
        L.lat_destroy.argtypes = [_P]
        L.lat_destroy.restype = None
        _lib = L
    return _lib


def check(code):
    if code != 0:
        raise LatError(code, lib().lat_last_error().decode(errors="replace"))


def ptr(t):
    """Device pointer of a torch tensor (or None)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def stream_ptr(stream):
    return None if stream is None else ctypes.c_void_p(stream.cuda_stream)


def chunk_attention_noalloc(q, k, v, out, T_q, T_kv, Hq, Hkv, dh, stream=None):
    """Context-free chunk attention whose scratch is the library's static array."""
    check(lib().lat_chunk_attention_noalloc(ptr(q), ptr(k), ptr(v), ptr(out), T_q, T_kv, Hq, Hkv, dh,
                                            stream_ptr(stream)))


class Context:
    """Owns one lat_ctx; keeps the ctypes structs alive while it exists."""

    def __init__(self, desc: ModelDesc, weights: Weights):
        self._desc = desc
        self._weights = weights
        h = _P()
        check(lib().lat_create(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(h)))
        self.handle = h

    def set_schedule(self, t):
        arr = (ctypes.c_float * len(t))(*t)
        check(lib().lat_set_schedule(self.handle, arr, len(t)))

    def prefill_kv(self, patch_emb, B, kv, stream=None):
        check(lib().lat_prefill_kv(self.handle, ptr(patch_emb), B, ptr(kv), stream_ptr(stream)))

    def block_forward(self, layer, x, kv, chunks=None, stream=None):
        if chunks is None:
            check(lib().lat_block_forward(self.handle, layer, ptr(x), None, 1, ptr(kv), stream_ptr(stream)))
        else:
            arr = (ChunkDesc * len(chunks))(*[ChunkDesc(*c) for c in chunks])
            check(lib().lat_block_forward(self.handle, layer, ptr(x), arr, len(chunks), ptr(kv),
                                          stream_ptr(stream)))

    def dit_interval(self, kv, lat, chunks, stream=None):
        arr = (ChunkDesc * len(chunks))(*[ChunkDesc(*c) for c in chunks])
        check(lib().lat_dit_interval(self.handle, ptr(kv), ptr(lat), arr, len(chunks), stream_ptr(stream)))

    def dit_pipeline_push(self, kv, stream_id, noise=None, done=None, stream=None):
        """Admit `noise` (or drain when None); returns the index of the chunk completed (or -1)."""
        out = ctypes.c_int(-1)
        check(lib().lat_dit_pipeline_push(self.handle, ptr(kv), stream_id, ptr(noise), ptr(done),
                                          ctypes.byref(out), stream_ptr(stream)))
        return out.value

    def dit_pipeline_reset(self, stream_id):
        check(lib().lat_dit_pipeline_reset(self.handle, stream_id))

    def dit_set_text(self, stream_id, text, stream=None):
        check(lib().lat_dit_set_text(self.handle, stream_id, ptr(text), stream_ptr(stream)))

    def dit_bind_pages(self, table):
        check(lib().lat_dit_bind_pages(self.handle, ptr(table)))

    def denoise_chunk(self, kv, state, x, stream=None):
        check(lib().lat_denoise_chunk(self.handle, ptr(kv), ptr(state), ptr(x), stream_ptr(stream)))

    def debug_indices(self, chunks=None, n=None):
        if chunks is None:
            arr, n = None, int(n)
        else:
            n = len(chunks)
            arr = (ChunkDesc * n)(*[ChunkDesc(*c) for c in chunks])
        slots = (ctypes.c_int * n)()
        pos = (ctypes.c_int * n)()
        check(lib().lat_debug_indices(self.handle, arr, n, slots, pos))
        return list(slots), list(pos)

    def debug_gemm(self, which, layer, reps, stream=None):
        check(lib().lat_debug_gemm(self.handle, which, layer, reps, stream_ptr(stream)))

    def debug_attention(self, q, k, v, out, T_q, T_kv, stream=None):
        check(lib().lat_debug_attention(self.handle, ptr(q), ptr(k), ptr(v), ptr(out), T_q, T_kv,
                                        stream_ptr(stream)))

    def debug_dense_gemm(self, which, layer, act, M, terms, out, stream=None):
        check(lib().lat_debug_dense_gemm(self.handle, which, layer, ptr(act), M, terms, ptr(out),
                                         stream_ptr(stream)))

    def debug_clear(self, stream=None):
        check(lib().lat_debug_clear(self.handle, stream_ptr(stream)))

    def debug_step(self, kv, reps, stream=None):
        check(lib().lat_debug_step(self.handle, ptr(kv), reps, stream_ptr(stream)))

    def debug_trace(self, buf=None):
        """Record phase timestamps of the step kernel into `buf` (int64 device tensor), or stop (None)."""
        check(lib().lat_debug_trace(self.handle, ptr(buf) if buf is not None else None,
                                    buf.numel() if buf is not None else 0))

    def sync(self):
        check(lib().lat_sync(self.handle))

    def clear_error(self):
        check(lib().lat_clear_error(self.handle))

    def debug_timeout(self, stream=None):
        check(lib().lat_debug_timeout(self.handle, stream_ptr(stream)))

    def debug_act_terms(self, terms):
        """Dense path: multiply 1 or 2 fp16 planes of the activation (precision study)."""
        check(lib().lat_debug_act_terms(self.handle, terms))

    def debug_wait_skew(self, which, extra):
        """Make one bounded wait of the step kernel's first block expect `extra` arrivals too many."""
        check(lib().lat_debug_wait_skew(self.handle, which, extra))

    def close(self):
        if getattr(self, "handle", None):
            lib().lat_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
