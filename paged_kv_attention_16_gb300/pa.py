"""Thin ctypes binding over libpa.so (include/pa.h).

Argument marshalling only: every step of the attention runs in the CUDA
library.  Functions keep the C names and argument order; tensors are passed
as torch tensors (their device pointers are handed to the library) or raw
integer addresses.  There is no fallback: if libpa.so is missing or fails to
load, every call raises.
"""
import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")

PA_F32, PA_BF16 = 0, 1
PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)
PA_ERR_SCRATCH_LIMIT = 5
PA_STATIC_SCRATCH_BYTES = 64 * 1024 * 1024
PA_DEV_BAD_BLOCK = 0x1
PA_DEV_BAD_QLEN = 0x2
PA_DEV_BAD_SEQLEN = 0x4
PA_DEV_BAD_QSL = 0x8
PA_DEV_OVERFLOW = 0x10
PA_DEV_TIMEOUT = 0x20
PA_DEV_INTERNAL = 0x40
PA_KV_NHD, PA_KV_HND = 0, 1  # pa_kv_layout

# Every entry point declared in include/pa.h.
EXPORTS = ("pa_forward", "pa_forward_workspace_bytes", "pa_mla_decode", "pa_cache_write",
           "pa_mla_decode_workspace_bytes", "pa_reserve", "pa_get_device_status",
           "pa_status_string", "pa_num_sms", "pa_debug_gather", "pa_profile_enable",
           "pa_profile_read", "pa_kernel_name", "pa_forward_static_scratch", "pa_forward_ex",
           "pa_mla_prefill", "pa_mla_prefill_workspace_bytes", "pa_debug_wait_timeout")
PA_K_COUNT = 10


class ForwardOptions(ctypes.Structure):
    """pa_forward_options: sinks = device pointer to [num_heads] fp32 sink
    logits, or None."""
    _fields_ = [("sinks", ctypes.c_void_p), ("kv_layout", ctypes.c_int),
                ("sliding_window", ctypes.c_int), ("alibi_slopes", ctypes.c_void_p),
                ("alibi_sqrt", ctypes.c_int), ("max_query_len", ctypes.c_int)]


def layout_code(kv_layout):
    """pa_kv_layout of "nhd" ([num_blocks, block_size, Hk, D]) or "hnd"
    ([num_blocks, Hk, block_size, D]); ints pass through."""
    if isinstance(kv_layout, int):
        return kv_layout
    return {"nhd": PA_KV_NHD, "hnd": PA_KV_HND}[kv_layout]


class PaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def lib():
    """The loaded libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libpa.so not found at {_LIB_PATH}; build it with "
                               "paged_kv_attention_16_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32p, c_int, c_float = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.pa_forward.argtypes = [vp, vp, vp, i32p, i32p, i32p, c_int, c_int, c_int, c_int,
                                 c_float, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_int]
        L.pa_forward.restype = c_int
        L.pa_forward_workspace_bytes.argtypes = [c_int] * 8
        L.pa_forward_workspace_bytes.restype = ctypes.c_size_t
        L.pa_mla_decode.argtypes = [vp, vp, i32p, i32p, c_int, c_int, c_int, c_int, c_float, vp,
                                    vp, c_int, c_int, c_int, c_int, c_int]
        L.pa_mla_decode.restype = c_int
        L.pa_mla_decode_workspace_bytes.argtypes = [c_int] * 5
        L.pa_mla_decode_workspace_bytes.restype = ctypes.c_size_t
        L.pa_reserve.argtypes = [ctypes.c_size_t]
        L.pa_reserve.restype = c_int
        L.pa_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.pa_get_device_status.restype = c_int
        L.pa_status_string.argtypes = [c_int]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_num_sms.argtypes = []
        L.pa_num_sms.restype = c_int
        L.pa_cache_write.argtypes = [vp, vp, vp, vp, i32p, i32p, i32p, c_int, c_int, c_int, vp,
                                     c_int, c_int, c_int, c_int, c_int, c_int]
        L.pa_cache_write.restype = c_int
        L.pa_debug_gather.argtypes = [vp, i32p, i32p, c_int, c_int, c_int, c_int, c_int, c_int,
                                      c_int, vp, vp]
        L.pa_debug_gather.restype = c_int
        L.pa_profile_enable.argtypes = [c_int]
        L.pa_profile_enable.restype = c_int
        L.pa_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_int)]
        L.pa_profile_read.restype = c_int
        L.pa_forward_static_scratch.argtypes = L.pa_forward.argtypes + [vp]
        L.pa_forward_static_scratch.restype = c_int
        L.pa_forward_ex.argtypes = L.pa_forward.argtypes + [ctypes.POINTER(ForwardOptions)]
        L.pa_forward_ex.restype = c_int
        L.pa_mla_prefill.argtypes = [vp, vp, vp, i32p, i32p, i32p, c_int, c_int, c_int, c_int,
                                     c_int, c_int, c_float, vp, vp, c_int, c_int, c_int, c_int,
                                     c_int, ctypes.c_longlong, c_int]
        L.pa_mla_prefill.restype = c_int
        L.pa_mla_prefill_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int,
                                                     ctypes.c_longlong, c_int]
        L.pa_mla_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.pa_debug_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp]
        L.pa_debug_wait_timeout.restype = c_int
        L.pa_kernel_name.argtypes = [c_int]
        L.pa_kernel_name.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(status):
    return lib().pa_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, device=None):
    """The cudaStream_t to launch on: `stream`, else the current stream of
    `device` (the raw query costs a fraction of torch.cuda.current_stream(),
    which builds a Python object per call)."""
    if stream is None:
        if _raw_stream is not None and device is not None and device >= 0:
            return _raw_stream(device)
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


_options_cache = {}


def _forward_options(sinks, layout, sliding_window, alibi_slopes, alibi_sqrt, max_query_len):
    """A pa_forward_options struct, reused for a repeated set of options."""
    key = (_ptr(sinks), layout, int(sliding_window), _ptr(alibi_slopes), int(bool(alibi_sqrt)),
           int(max_query_len))
    opts = _options_cache.get(key)
    if opts is None:
        if len(_options_cache) > 256:
            _options_cache.clear()
        opts = _options_cache[key] = ForwardOptions(*key)
    return opts


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(status, where):
    if status != PA_OK:
        raise PaError(status, where)


def pa_forward(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, num_heads,
               num_kv_heads, head_dim, block_size, scale, out, stream=None, *, max_seq_len,
               kv_split_tokens=0, num_blocks=None, sinks=None, kv_layout="nhd",
               sliding_window=0, alibi_slopes=None, alibi_sqrt=False, max_query_len=0,
               check=True):
    """Unified paged attention (see include/pa.h).  Shapes are read from the
    tensors; max_seq_len is the host-known bound on seq_lens.  The options --
    sinks and alibi_slopes (fp32 device tensors of num_heads values), an HND
    kv_layout, a sliding window, sqrt ALiBi -- go through pa_forward_ex."""
    layout = layout_code(kv_layout)
    args = (
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(query_start_loc), int(num_heads), int(num_kv_heads), int(head_dim),
        int(block_size), float(scale), _ptr(out), _stream_ptr(stream, q.get_device()),
        _dtype_code(q), int(seq_lens.shape[0]), int(q.shape[0]), int(block_table.shape[1]),
        int(num_blocks if num_blocks is not None else k_cache.shape[0]), int(max_seq_len),
        int(kv_split_tokens))
    if (sinks is None and layout == PA_KV_NHD and not sliding_window
            and alibi_slopes is None and not max_query_len):
        st, where = lib().pa_forward(*args), "pa_forward"
    else:
        for name, t in (("sinks", sinks), ("alibi_slopes", alibi_slopes)):
            if isinstance(t, torch.Tensor) and (t.dtype != torch.float32
                                                or t.numel() != num_heads):
                raise TypeError(f"{name} must be a float32 tensor of num_heads elements")
        opts = _forward_options(sinks, layout, sliding_window, alibi_slopes, alibi_sqrt,
                                max_query_len)
        st, where = lib().pa_forward_ex(*args, ctypes.byref(opts)), "pa_forward_ex"
    if check:
        _check(st, where)
    return st


def pa_forward_static_scratch(q, k_cache, v_cache, block_table, seq_lens, query_start_loc,
                              num_heads, num_kv_heads, head_dim, block_size, scale, out,
                              stream=None, *, max_seq_len, kv_split_tokens=0, num_blocks=None,
                              device_status=None, check=True):
    """pa_forward with no device allocation (scratch in the library's fixed
    static region); device_status: optional int32 device tensor of one
    element that receives the PA_DEV_* bits."""
    st = lib().pa_forward_static_scratch(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(query_start_loc), int(num_heads), int(num_kv_heads), int(head_dim),
        int(block_size), float(scale), _ptr(out), _stream_ptr(stream), _dtype_code(q),
        int(seq_lens.shape[0]), int(q.shape[0]), int(block_table.shape[1]),
        int(num_blocks if num_blocks is not None else k_cache.shape[0]), int(max_seq_len),
        int(kv_split_tokens), _ptr(device_status))
    if check:
        _check(st, "pa_forward_static_scratch")
    return st


def pa_forward_workspace_bytes(dtype, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                               max_seq_len, kv_split_tokens=0):
    return lib().pa_forward_workspace_bytes(int(dtype), int(num_seqs), int(num_tokens),
                                            int(num_heads), int(num_kv_heads), int(head_dim),
                                            int(max_seq_len), int(kv_split_tokens))


def pa_mla_decode(q, kv_cache, block_table, seq_lens, num_heads, kv_lora_rank, rope_dim,
                  block_size, scale, out, stream=None, *, max_seq_len, kv_split_tokens=0,
                  check=True):
    st = lib().pa_mla_decode(
        _ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), int(num_heads),
        int(kv_lora_rank), int(rope_dim), int(block_size), float(scale), _ptr(out),
        _stream_ptr(stream), int(seq_lens.shape[0]), int(block_table.shape[1]),
        int(kv_cache.shape[0]), int(max_seq_len), int(kv_split_tokens))
    if check:
        _check(st, "pa_mla_decode")
    return st


def pa_mla_decode_workspace_bytes(num_seqs, num_heads, kv_lora_rank, max_seq_len,
                                  kv_split_tokens=0):
    return lib().pa_mla_decode_workspace_bytes(int(num_seqs), int(num_heads),
                                               int(kv_lora_rank), int(max_seq_len),
                                               int(kv_split_tokens))


def pa_reserve(nbytes):
    _check(lib().pa_reserve(int(nbytes)), "pa_reserve")


def pa_get_device_status(stream=None):
    v = ctypes.c_uint32(0)
    _check(lib().pa_get_device_status(_stream_ptr(stream), ctypes.byref(v)),
           "pa_get_device_status")
    return int(v.value)


def pa_profile_enable(on=True):
    _check(lib().pa_profile_enable(1 if on else 0), "pa_profile_enable")


def pa_profile_read():
    """{kernel name: (total ms, launches)} of the launches timed since the
    last read (synchronises)."""
    ms = (ctypes.c_double * PA_K_COUNT)()
    n = (ctypes.c_int * PA_K_COUNT)()
    _check(lib().pa_profile_read(ms, n), "pa_profile_read")
    out = {}
    for i in range(PA_K_COUNT):
        if n[i]:
            out[pa_kernel_name(i)] = (float(ms[i]), int(n[i]))
    return out


def pa_kernel_name(kernel_id):
    return lib().pa_kernel_name(int(kernel_id)).decode()


def pa_num_sms():
    return int(lib().pa_num_sms())


def pa_cache_write(k_new, v_new, k_cache, v_cache, block_table, seq_lens, query_start_loc,
                   block_size, stream=None, kv_layout="nhd", check=True):
    """pa_cache_write on torch tensors: k_new/v_new [T, Hk, D], caches
    [num_blocks, block_size, Hk, D] ("nhd") or [num_blocks, Hk, block_size, D]
    ("hnd"), written in place."""
    dt = PA_BF16 if k_new.dtype == torch.bfloat16 else PA_F32
    st = lib().pa_cache_write(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(query_start_loc), int(k_new.shape[1]), int(k_new.shape[2]),
        int(block_size), _stream_ptr(stream), dt, int(seq_lens.shape[0]), int(k_new.shape[0]),
        int(block_table.shape[1]), int(k_cache.shape[0]), layout_code(kv_layout))
    if check:
        _check(st, "pa_cache_write")
    return st


def pa_debug_gather(k_cache, block_table, seq_lens, block_size, max_seq_len, dense_out,
                    stream=None):
    row_elems = int(k_cache[0, 0].numel())
    st = lib().pa_debug_gather(_ptr(k_cache), _ptr(block_table), _ptr(seq_lens),
                               int(seq_lens.shape[0]), int(block_table.shape[1]),
                               int(k_cache.shape[0]), int(block_size), row_elems,
                               int(k_cache.element_size()), int(max_seq_len), _ptr(dense_out),
                               _stream_ptr(stream))
    _check(st, "pa_debug_gather")


def pa_debug_wait_timeout(limit_ns, done, stream=None, check=True):
    """Test-only: one kernel whose bounded mbarrier wait runs out after
    limit_ns (see include/pa.h); `done` is an int32 device tensor of one
    element that the kernel sets to 2 when it returns."""
    st = lib().pa_debug_wait_timeout(int(limit_ns), _ptr(done), _stream_ptr(stream))
    if check:
        _check(st, "pa_debug_wait_timeout")
    return st


# ---------------------------------------------------------------------------
# conveniences over the batches of paged_kv_attention_16_gb300.inputs
# ---------------------------------------------------------------------------

def to_device(batch, device="cuda"):
    """Copy every tensor field of a PagedBatch / MlaBatch to `device`."""
    import dataclasses
    fields = {}
    for f in dataclasses.fields(batch):
        v = getattr(batch, f.name)
        fields[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
    return type(batch)(**fields)


def forward(b, out=None, stream=None, kv_split_tokens=None, sinks=None, sliding_window=0,
            alibi_slopes=None, alibi_sqrt=False, max_query_len=0):
    """pa_forward on a device-resident PagedBatch (pa_forward_ex when an
    option is set: sinks / alibi_slopes as fp32 device tensors of num_heads
    values, a sliding window, sqrt ALiBi, the batch's HND layout); returns
    `out`."""
    if out is None:
        out = torch.empty_like(b.q)
    pa_forward(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens, b.query_start_loc,
               b.num_heads, b.num_kv_heads, b.head_dim, b.block_size, b.scale, out, stream,
               max_seq_len=b.max_seq_len,
               kv_split_tokens=b.kv_split_tokens if kv_split_tokens is None else kv_split_tokens,
               sinks=sinks, kv_layout=b.kv_layout, sliding_window=sliding_window,
               alibi_slopes=alibi_slopes, alibi_sqrt=alibi_sqrt, max_query_len=max_query_len)
    return out


def pa_mla_prefill(q, kv_cache, w_kv, block_table, seq_lens, query_start_loc, num_heads,
                   kv_lora_rank, qk_nope_dim, rope_dim, v_head_dim, block_size, scale, out,
                   stream=None, *, max_seq_len, max_total_kv, kv_split_tokens=0, num_blocks=None,
                   check=True):
    """Non-absorbed MLA prefill / extend (see include/pa.h)."""
    st = lib().pa_mla_prefill(
        _ptr(q), _ptr(kv_cache), _ptr(w_kv), _ptr(block_table), _ptr(seq_lens),
        _ptr(query_start_loc), int(num_heads), int(kv_lora_rank), int(qk_nope_dim),
        int(rope_dim), int(v_head_dim), int(block_size), float(scale), _ptr(out),
        _stream_ptr(stream), int(seq_lens.shape[0]), int(q.shape[0]), int(block_table.shape[1]),
        int(num_blocks if num_blocks is not None else kv_cache.shape[0]), int(max_seq_len),
        int(max_total_kv), int(kv_split_tokens))
    if check:
        _check(st, "pa_mla_prefill")
    return st


def mla_prefill(b, out=None, stream=None, kv_split_tokens=None):
    """pa_mla_prefill on a device-resident MlaPrefillBatch; returns `out`."""
    if out is None:
        out = torch.empty((b.num_tokens, b.num_heads, b.v_head_dim), dtype=b.q.dtype,
                          device=b.q.device)
    pa_mla_prefill(b.q, b.kv_cache, b.w_kv, b.block_table, b.seq_lens, b.query_start_loc,
                   b.num_heads, b.kv_lora_rank, b.qk_nope_dim, b.rope_dim, b.v_head_dim,
                   b.block_size, b.scale, out, stream, max_seq_len=b.max_seq_len,
                   max_total_kv=b.max_total_kv,
                   kv_split_tokens=b.kv_split_tokens if kv_split_tokens is None
                   else kv_split_tokens)
    return out


def mla_decode(b, out=None, stream=None):
    """pa_mla_decode on a device-resident MlaBatch; returns `out`."""
    if out is None:
        out = torch.empty((b.num_seqs, b.num_heads, b.kv_lora_rank), dtype=b.q.dtype,
                          device=b.q.device)
    pa_mla_decode(b.q, b.kv_cache, b.block_table, b.seq_lens, b.num_heads, b.kv_lora_rank,
                  b.rope_dim, b.block_size, b.scale, out, stream, max_seq_len=b.max_seq_len,
                  kv_split_tokens=b.kv_split_tokens)
    return out
