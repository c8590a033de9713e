"""ctypes binding of the C ABI in include/gqa_attn.h (argument marshalling only).

Every function here has the name of the C entry point it calls and forwards raw device
pointers; all arithmetic of the block runs in the library's CUDA kernels.  Torch tensors
are accepted for convenience and passed as ``tensor.data_ptr()``.  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH

GQA_OK = 0
STATUS_NAMES = {0: "GQA_OK", 1: "GQA_ERR_INVALID_ARG", 2: "GQA_ERR_SHAPE", 3: "GQA_ERR_ALIGN",
                4: "GQA_ERR_CUDA", 5: "GQA_ERR_TIMEOUT", 6: "GQA_ERR_OOM", 7: "GQA_ERR_DEVICE"}

# Every symbol include/gqa_attn.h declares.
EXPORTED = ("attn_create", "attn_create_shard", "attn_prefill", "attn_decode", "attn_set_norm", "attn_prefill_residual",
            "attn_decode_residual", "attn_sync_status", "attn_debug_buffers",
            "attn_profile_begin", "attn_profile_end", "attn_debug_inject_timeout",
            "attn_debug_pair_schedule", "attn_debug_exp2", "attn_decode_attention_noalloc",
            "attn_decode_attention_noalloc_status", "attn_decode_attention_noalloc_debug_inject_timeout",
            "attn_destroy", "attn_strerror", "attn_last_cuda_error")

# Kernel kinds of attn_profile_end (GQA_KERNEL_* in include/gqa_attn.h).
KERNEL_KINDS = ("qkv_gemm", "qkv_splitk", "flash_prefill", "decode_attn", "out_gemm", "out_splitk",
                "rms_norm")

_lib = None


class GQAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().attn_strerror(status).decode()
        extra = ""
        if status == 4:
            extra = f" (cudaError {lib().attn_last_cuda_error()})"
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {msg}{extra}")


def lib() -> ctypes.CDLL:
    """Load libgqa_attn.so from the package directory (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first (__graft_entry__.build() or "
                           "python -m transformer_gqa_attention_gb300._build)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.attn_create.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(vp)]
    L.attn_create.restype = i32
    L.attn_create_shard.argtypes = [vp, vp, vp, vp, i32, vp, ctypes.POINTER(vp)]
    L.attn_create_shard.restype = i32
    L.attn_prefill.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, i32, i32, vp, vp]
    L.attn_prefill.restype = i32
    L.attn_decode.argtypes = [vp, vp, i32, i32, vp, vp, vp, i32, vp, vp]
    L.attn_decode.restype = i32
    L.attn_set_norm.argtypes = [vp, vp, ctypes.c_float, vp]
    L.attn_set_norm.restype = i32
    L.attn_prefill_residual.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, i32, i32, vp, vp]
    L.attn_prefill_residual.restype = i32
    L.attn_decode_residual.argtypes = [vp, vp, i32, i32, vp, vp, vp, i32, vp, vp]
    L.attn_decode_residual.restype = i32
    L.attn_sync_status.argtypes = [vp, vp]
    L.attn_sync_status.restype = i32
    L.attn_debug_buffers.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp)]
    L.attn_debug_buffers.restype = i32
    L.attn_profile_begin.argtypes = [vp]
    L.attn_profile_begin.restype = i32
    L.attn_profile_end.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i32), vp]
    L.attn_profile_end.restype = i32
    L.attn_debug_inject_timeout.argtypes = [vp, i32]
    L.attn_debug_inject_timeout.restype = i32
    ip = ctypes.POINTER(i32)
    L.attn_debug_pair_schedule.argtypes = [i32, i32, i32, ip, ip, ip, ip, i32, ip]
    L.attn_debug_pair_schedule.restype = i32
    L.attn_debug_exp2.argtypes = [vp, vp, vp, i32, vp]
    L.attn_debug_exp2.restype = i32
    L.attn_decode_attention_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
    L.attn_decode_attention_noalloc.restype = i32
    L.attn_decode_attention_noalloc_status.argtypes = [vp]
    L.attn_decode_attention_noalloc_status.restype = i32
    L.attn_decode_attention_noalloc_debug_inject_timeout.argtypes = []
    L.attn_decode_attention_noalloc_debug_inject_timeout.restype = i32
    L.attn_destroy.argtypes = [vp]
    L.attn_destroy.restype = None
    L.attn_strerror.argtypes = [i32]
    L.attn_strerror.restype = ctypes.c_char_p
    L.attn_last_cuda_error.argtypes = []
    L.attn_last_cuda_error.restype = i32
    _lib = L
    return L


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != GQA_OK:
        raise GQAError(fn, st)


def attn_create(wq, wk, wv, wo, stream=None) -> int:
    ctx = ctypes.c_void_p()
    _check("attn_create", lib().attn_create(_ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _stream(stream),
                                            ctypes.byref(ctx)))
    return ctx.value


def attn_create_shard(wq_shard, wk_shard, wv_shard, wo_shard, n_kv_local, stream=None) -> int:
    """Context for one tensor-parallel shard (n_kv_local kv groups; see tp.shard_weights)."""
    ctx = ctypes.c_void_p()
    _check("attn_create_shard", lib().attn_create_shard(_ptr(wq_shard), _ptr(wk_shard), _ptr(wv_shard),
                                                        _ptr(wo_shard), int(n_kv_local), _stream(stream),
                                                        ctypes.byref(ctx)))
    return ctx.value


def attn_prefill(ctx, x, B, T, R, causal, cache_k, cache_v, S_max, start_pos, delta, stream=None):
    _check("attn_prefill", lib().attn_prefill(ctx, _ptr(x), int(B), int(T), _ptr(R), int(bool(causal)),
                                              _ptr(cache_k), _ptr(cache_v), int(S_max), int(start_pos),
                                              _ptr(delta), _stream(stream)))


def attn_decode(ctx, x, B, start_pos, R_row, cache_k, cache_v, S_max, delta, stream=None):
    _check("attn_decode", lib().attn_decode(ctx, _ptr(x), int(B), int(start_pos), _ptr(R_row),
                                            _ptr(cache_k), _ptr(cache_v), int(S_max), _ptr(delta),
                                            _stream(stream)))


def attn_set_norm(ctx, norm_w, eps=1e-5, stream=None):
    _check("attn_set_norm", lib().attn_set_norm(ctx, _ptr(norm_w), float(eps), _stream(stream)))


def attn_prefill_residual(ctx, x, B, T, R, causal, cache_k, cache_v, S_max, start_pos, h_out, stream=None):
    _check("attn_prefill_residual",
           lib().attn_prefill_residual(ctx, _ptr(x), int(B), int(T), _ptr(R), int(bool(causal)), _ptr(cache_k),
                                       _ptr(cache_v), int(S_max), int(start_pos), _ptr(h_out), _stream(stream)))


def attn_decode_residual(ctx, x, B, start_pos, R_row, cache_k, cache_v, S_max, h_out, stream=None):
    _check("attn_decode_residual",
           lib().attn_decode_residual(ctx, _ptr(x), int(B), int(start_pos), _ptr(R_row), _ptr(cache_k),
                                      _ptr(cache_v), int(S_max), _ptr(h_out), _stream(stream)))


def attn_sync_status(ctx, stream=None):
    _check("attn_sync_status", lib().attn_sync_status(ctx, _stream(stream)))


def attn_debug_buffers(ctx):
    q, h = ctypes.c_void_p(), ctypes.c_void_p()
    _check("attn_debug_buffers", lib().attn_debug_buffers(ctx, ctypes.byref(q), ctypes.byref(h)))
    return q.value, h.value


def attn_profile_begin(ctx):
    _check("attn_profile_begin", lib().attn_profile_begin(ctx))


def attn_profile_end(ctx, stream=None):
    """-> {kind: (total_ms, launches)} for the launches since attn_profile_begin."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    _check("attn_profile_end", lib().attn_profile_end(ctx, ms, cnt, _stream(stream)))
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def attn_debug_pair_schedule(m_tiles, n_tiles, n_pairs):
    """The many-token projection GEMM's work schedule (host computation, no GPU needed):
    (full_rounds, tail_w, grid_ctas, items) with items a list of (pair, m tile, first column,
    width) in launch order."""
    i32 = ctypes.c_int
    full, tail, grid, n = i32(), i32(), i32(), i32()
    L = lib()
    st = L.attn_debug_pair_schedule(m_tiles, n_tiles, n_pairs, ctypes.byref(full), ctypes.byref(tail),
                                    ctypes.byref(grid), None, 0, ctypes.byref(n))
    if st not in (0, 2):  # GQA_ERR_SHAPE: the count is in n
        _check("attn_debug_pair_schedule", st)
    buf = (i32 * (4 * max(n.value, 1)))()
    _check("attn_debug_pair_schedule",
           L.attn_debug_pair_schedule(m_tiles, n_tiles, n_pairs, ctypes.byref(full), ctypes.byref(tail),
                                      ctypes.byref(grid), buf, n.value, ctypes.byref(n)))
    items = [tuple(buf[4 * i:4 * i + 4]) for i in range(n.value)]
    return full.value, tail.value, grid.value, items


def attn_debug_exp2(a, out_fma, out_mufu, stream=None):
    """Evaluate the softmax's two exponentials (FMA-pipe cubic, ex2.approx) on a fp32 device
    tensor into two fp32 device tensors of the same size."""
    _check("attn_debug_exp2", lib().attn_debug_exp2(_ptr(a), _ptr(out_fma), _ptr(out_mufu), int(a.numel()),
                                                    _stream(stream)))


def attn_debug_inject_timeout(ctx, kind):
    """Arm the one-shot failure-path test hook for the next launch of a kernel kind (a
    name from KERNEL_KINDS or its index)."""
    k = KERNEL_KINDS.index(kind) if isinstance(kind, str) else int(kind)
    _check("attn_debug_inject_timeout", lib().attn_debug_inject_timeout(ctx, k))


def attn_decode_attention_noalloc(q_r, cache_k, cache_v, B, kv_len, S_max, h, stream=None):
    """Decode attention into `h` without any device allocation by the library (see the
    header for the scratch-array limits and the first-call set-up)."""
    _check("attn_decode_attention_noalloc",
           lib().attn_decode_attention_noalloc(_ptr(q_r), _ptr(cache_k), _ptr(cache_v), int(B),
                                               int(kv_len), int(S_max), _ptr(h), _stream(stream)))


def attn_decode_attention_noalloc_status(stream=None):
    """Synchronise the stream and raise GQAError(GQA_ERR_TIMEOUT) if a bounded wait of an
    allocation-free call ran out since the last check (clears the status word)."""
    _check("attn_decode_attention_noalloc_status", lib().attn_decode_attention_noalloc_status(_stream(stream)))


def attn_decode_attention_noalloc_debug_inject_timeout():
    """Arm the one-shot failure-path hook for the next allocation-free decode call."""
    _check("attn_decode_attention_noalloc_debug_inject_timeout",
           lib().attn_decode_attention_noalloc_debug_inject_timeout())


def attn_destroy(ctx):
    if ctx:
        lib().attn_destroy(ctx)


def attn_strerror(status: int) -> str:
    return lib().attn_strerror(int(status)).decode()


def raw_status(fn_name: str, *args) -> int:
    """Call an entry point with raw ctypes-compatible arguments and return its status code
    (used by boundary tests that pass invalid arguments on purpose)."""
    return getattr(lib(), fn_name)(*args)
