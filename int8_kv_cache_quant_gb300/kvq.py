"""Python binding of libkvq (include/kvq.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  torch supplies device
memory and the current stream; all arithmetic runs in libkvq's CUDA kernels.  There is no
CPU fallback: if libkvq.so is missing or the call fails, an exception is raised.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

BLOCK_SIZE = 16
PV_TILE = 128

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape or option",
           3: "device pointer not 16-byte aligned", 4: "workspace missing or too small",
           5: "CUDA launch or runtime error"}

DEV_BAD_BLOCK, DEV_BAD_POS, DEV_TIMEOUT, DEV_BAD_CELL, DEV_BAD_SEQ = 0x1, 0x2, 0x4, 0x8, 0x10


class KvqError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__("%s failed: %s (status %d)" % (fn, _STATUS.get(status, "?"), status))
        self.status = status


class _Cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class _DecodeOpts(ctypes.Structure):
    _fields_ = [("split_rows", ctypes.c_int32), ("route_threshold", ctypes.c_int32),
                ("force_route", ctypes.c_int32), ("stage1_event_begin", ctypes.c_void_p),
                ("stage1_event_end", ctypes.c_void_p), ("launches", ctypes.POINTER(ctypes.c_int32))]


_lib = None


def lib():
    """The loaded libkvq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkvq.so is not built (%s); run int8_kv_cache_quant_gb300.build.build()"
                               % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        cp = ctypes.POINTER(_Cache)
        L.kvq_version.restype = ctypes.c_int
        L.kvq_status_string.restype = ctypes.c_char_p
        L.kvq_status_string.argtypes = [ctypes.c_int]
        L.kvq_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        L.kvq_quant_write.argtypes = [cp, vp, vp, i32, vp, vp, vp, i32, i32, vp]
        L.kvq_rope_quant_write.argtypes = [cp, vp, i32, vp, vp, i32, vp, vp, vp, i32, i32, vp, i32, i32,
                                           vp, vp, vp, vp]
        L.kvq_attn_prefill_int8_qcodes.argtypes = [cp, vp, vp, i32, i32, i32, vp, i32, f32, vp, vp, sz, vp]
        L.kvq_decode_workspace_bytes.restype = sz
        L.kvq_decode_auto_split_rows.restype = i32
        L.kvq_decode_auto_split_rows.argtypes = [i32, i32, i32, i32, i32]
        L.kvq_prefill_split_tiles.restype = i32
        L.kvq_device_accessible.restype = i32
        L.kvq_device_accessible.argtypes = [ctypes.c_void_p]
        L.kvq_prefill_split_tiles.argtypes = [i32, i32, i32, i32]
        L.kvq_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, ctypes.POINTER(_DecodeOpts)]
        L.kvq_attn_decode_int8kv.argtypes = [cp, vp, i32, i32, vp, i32, vp, i32, f32, vp, vp, sz,
                                             ctypes.POINTER(_DecodeOpts), vp]
        L.kvq_attn_decode_int8kv_noalloc.argtypes = [cp, vp, i32, i32, vp, i32, vp, i32, f32, vp,
                                                     ctypes.POINTER(_DecodeOpts), vp]
        L.kvq_verify_workspace_bytes.restype = sz
        L.kvq_verify_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(_DecodeOpts)]
        L.kvq_attn_verify_int8kv.argtypes = [cp, vp, i32, i32, i32, vp, i32, vp, i32, f32, vp, vp, sz,
                                             ctypes.POINTER(_DecodeOpts), vp]
        L.kvq_decode_step_int8kv.argtypes = [cp, vp, vp, vp, i32, i32, i32, vp, i32, vp, i32, f32, vp, vp, sz,
                                             ctypes.POINTER(_DecodeOpts), vp]
        L.kvq_prefill_first_workspace_bytes.restype = sz
        L.kvq_prefill_first_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.kvq_attn_prefill_first_bf16.argtypes = [cp, vp, vp, vp, i32, i32, vp, i32, f32, vp, vp, sz, vp]
        L.kvq_prefill_workspace_bytes.restype = sz
        L.kvq_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.kvq_attn_prefill_int8.argtypes = [cp, vp, i32, i32, i32, vp, i32, f32, vp, vp, sz, vp]
        L.kvq_attn_sparse_int8kv.argtypes = [cp, vp, i32, i32, vp, vp, vp, i32, f32, vp, vp, sz, vp]
        L.kvq_sparse_workspace_bytes.restype = sz
        L.kvq_sparse_workspace_bytes.argtypes = [i32, i32, i32]
        L.kvq_debug_prefill_q_codes.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.kvq_debug_fault_inject.argtypes = [i32, ctypes.c_int64]
        L.kvq_debug_stream_floor.argtypes = [cp, i32, vp, i32, vp, i32, i32, vp]
        L.kvq_debug_prefill_qk_int32.argtypes = [cp, vp, vp, i32, i32, i32, vp, i32, f32, i32, i32, i32, i32, i32,
                                                 vp, vp, vp, sz, vp]
        _lib = L
    return _lib


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _p(t):
    """Device pointer of a CUDA tensor.  Anything else is refused before any launch: a kernel
    handed a host pointer would fault."""
    if t is None:
        return None
    if t.device.type != "cuda":
        raise ValueError("the library takes CUDA tensors here (got a %s tensor)" % t.device.type)
    return ctypes.c_void_p(t.data_ptr())


def _hp(t):
    """Pointer for the decode calls' zero-copy arguments (q, k_new, v_new, out): a CUDA tensor,
    or page-locked host memory mapped into the device's address space."""
    if t is None:
        return None
    if t.device.type != "cuda" and not kvq_device_accessible(t):
        raise ValueError("a host tensor must be page-locked memory mapped into the device's address space "
                         "(e.g. tensor.pin_memory())")
    return ctypes.c_void_p(t.data_ptr())


def _check(fn, status):
    if status != 0:
        raise KvqError(fn, status)


def kvq_device_accessible(t):
    """True when the kernels can dereference tensor t's storage (device memory, or page-locked
    host memory mapped into the device's address space)."""
    return bool(lib().kvq_device_accessible(ctypes.c_void_p(t.data_ptr())))


def _host_ok(fn, *tensors):
    """Host tensors passed to a decode call must be mapped page-locked memory (zero-copy): the
    kernels read and write them across the host link.  Anything else is refused before launch."""
    for t in tensors:
        if t is not None and t.device.type == "cpu" and not kvq_device_accessible(t):
            raise ValueError(fn + ": a host tensor must be page-locked memory mapped into the device's "
                             "address space (e.g. tensor.pin_memory())")


def _new_out(shape, q):
    # a host q (zero-copy) gets its result in page-locked host memory too
    return torch.empty(shape, dtype=torch.float32, device=q.device, pin_memory=q.device.type == "cpu")


class KVCache:
    """A paged int8 K/V cache on the GPU in the library's layout:
    k [num_blocks][n_kv_heads][head_dim/16][16][16] int8, v [num_blocks][n_kv_heads][head_dim][16]
    int8, k_scale / v_scale [num_blocks][n_kv_heads][16] fp32."""

    def __init__(self, num_blocks, n_kv_heads, head_dim, device="cuda"):
        self.num_blocks, self.n_kv_heads, self.head_dim = num_blocks, n_kv_heads, head_dim
        self.k = torch.zeros((num_blocks, n_kv_heads, head_dim // 16, BLOCK_SIZE, 16),
                             dtype=torch.int8, device=device)
        self.v = torch.zeros((num_blocks, n_kv_heads, head_dim, BLOCK_SIZE), dtype=torch.int8,
                             device=device)
        self.k_scale = torch.zeros((num_blocks, n_kv_heads, BLOCK_SIZE), dtype=torch.float32,
                                   device=device)
        self.v_scale = torch.zeros_like(self.k_scale)

    def struct(self):
        # every cache tensor goes through _p: a cache left in host memory is refused before any
        # launch (a kernel handed its pageable pointers would fault)
        ptrs = [_p(t).value for t in (self.k, self.v, self.k_scale, self.v_scale)]
        return _Cache(*ptrs, self.num_blocks, BLOCK_SIZE, self.n_kv_heads, self.head_dim)


def kvq_version():
    return lib().kvq_version()


def kvq_device_status(stream=None):
    flags = ctypes.c_uint32(0)
    _check("kvq_device_status", lib().kvq_device_status(ctypes.byref(flags), _stream(stream)))
    return flags.value


def kvq_quant_write(cache, k_new, v_new, seq_idx, pos, block_table, stream=None):
    """k_new, v_new: bf16 [T][Hkv][D]; seq_idx, pos: int32 [T]; block_table: int32 [S][M]."""
    bt = block_table if block_table.dim() == 2 else block_table.view(1, -1)
    c = cache.struct()
    _check("kvq_quant_write", lib().kvq_quant_write(
        ctypes.byref(c), _p(k_new), _p(v_new), int(seq_idx.numel()), _p(seq_idx), _p(pos), _p(bt),
        int(bt.shape[0]), int(bt.shape[1]), _stream(stream)))


def kvq_rope_quant_write(cache, q, k_new, v_new, seq_idx, pos, block_table, cos_sin, rotary_dim,
                         q_codes=None, q_scales=None, q_rot=None, stream=None):
    """Fused producer: RoPE on Q and K (cos_sin fp32 [max_pos][rotary_dim]), the quantisation
    rule on Q, K and V; K/V into the cache.  q: bf16 [T][Hq][D] or None.  Returns
    (q_codes int8 [T][Hq][D], q_scales fp32 [T][Hq], q_rot bf16 [T][Hq][D]), allocated when not
    given (None when q is None)."""
    bt = block_table if block_table.dim() == 2 else block_table.view(1, -1)
    T = int(seq_idx.numel())
    Hq = int(q.shape[1]) if q is not None else 0
    D = cache.head_dim
    if q is not None:
        dev = q.device
        if q_codes is None:
            q_codes = torch.empty((T, Hq, D), dtype=torch.int8, device=dev)
        if q_scales is None:
            q_scales = torch.empty((T, Hq), dtype=torch.float32, device=dev)
        if q_rot is None:
            q_rot = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    c = cache.struct()
    _check("kvq_rope_quant_write", lib().kvq_rope_quant_write(
        ctypes.byref(c), _p(q) if q is not None else None, Hq, _p(k_new), _p(v_new), T, _p(seq_idx), _p(pos),
        _p(bt), int(bt.shape[0]), int(bt.shape[1]), _p(cos_sin), int(cos_sin.shape[0]), int(rotary_dim),
        _p(q_codes) if q_codes is not None else None, _p(q_scales) if q_scales is not None else None,
        _p(q_rot) if q_rot is not None else None, _stream(stream)))
    return q_codes, q_scales, q_rot


def _decode_opts(split_rows, route_threshold, force_route, events=None, launches=None):
    ev0 = ev1 = None
    if events is not None:
        ev0, ev1 = (ctypes.c_void_p(e.cuda_event) for e in events)
    return _DecodeOpts(int(split_rows), int(route_threshold), int(force_route), ev0, ev1,
                       ctypes.pointer(launches) if launches is not None else None)


def kvq_decode_auto_split_rows(batch, n_kv_heads, head_dim, max_ctx, n_sms):
    return int(lib().kvq_decode_auto_split_rows(batch, n_kv_heads, head_dim, max_ctx, n_sms))


def kvq_prefill_split_tiles(n_tokens, n_q_heads, history_len, n_sms):
    return int(lib().kvq_prefill_split_tiles(n_tokens, n_q_heads, history_len, n_sms))


def kvq_decode_workspace_bytes(batch, n_q_heads, max_ctx, head_dim, split_rows=0,
                               route_threshold=0, force_route=0):
    o = _decode_opts(split_rows, route_threshold, force_route)
    return int(lib().kvq_decode_workspace_bytes(batch, n_q_heads, max_ctx, head_dim, ctypes.byref(o)))


def kvq_verify_workspace_bytes(batch, n_rows, n_q_heads, max_ctx, head_dim, split_rows=0,
                               route_threshold=0, force_route=0):
    o = _decode_opts(split_rows, route_threshold, force_route)
    return int(lib().kvq_verify_workspace_bytes(batch, n_rows, n_q_heads, max_ctx, head_dim, ctypes.byref(o)))


def kvq_attn_decode_int8kv(cache, q, block_table, ctx_lens, max_ctx, softmax_scale, out=None,
                           workspace=None, split_rows=0, route_threshold=0, force_route=0,
                           stream=None, stage1_events=None):
    """q: bf16 [B][Hq][D]; block_table int32 [B][M]; ctx_lens int32 [B] (device);
    max_ctx: host bound of ctx_lens.  Returns out fp32 [B][Hq][D].  stage1_events: optional
    pair of torch.cuda.Event recorded around the stage-1 kernel (profiling)."""
    B, Hq, D = q.shape
    if out is None:
        out = _new_out((B, Hq, D), q)
    _host_ok("kvq_attn_decode_int8kv", q, out)
    o = _decode_opts(split_rows, route_threshold, force_route, stage1_events)
    need = int(lib().kvq_decode_workspace_bytes(B, Hq, max(1, int(max_ctx)), D, ctypes.byref(o)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=cache.k.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    c = cache.struct()
    _check("kvq_attn_decode_int8kv", lib().kvq_attn_decode_int8kv(
        ctypes.byref(c), _hp(q), B, Hq, _p(block_table), int(block_table.shape[1]), _p(ctx_lens),
        int(max_ctx), float(softmax_scale), _hp(out), _p(workspace), wbytes, ctypes.byref(o),
        _stream(stream)))
    return out


def kvq_attn_verify_int8kv(cache, q, block_table, ctx_lens, max_ctx, softmax_scale, out=None,
                           workspace=None, split_rows=0, route_threshold=0, force_route=0,
                           stream=None, stage1_events=None):
    """q: bf16 [B][nq][Hq][D], the nq newest tokens of each sequence; row i of sequence b sees
    keys t < ctx_lens[b] - nq + 1 + i.  Returns out fp32 [B][nq][Hq][D]."""
    B, nq, Hq, D = q.shape
    if out is None:
        out = _new_out((B, nq, Hq, D), q)
    _host_ok("kvq_attn_verify_int8kv", q, out)
    o = _decode_opts(split_rows, route_threshold, force_route, stage1_events)
    need = int(lib().kvq_verify_workspace_bytes(B, nq, Hq, max(1, int(max_ctx)), D, ctypes.byref(o)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=cache.k.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    c = cache.struct()
    _check("kvq_attn_verify_int8kv", lib().kvq_attn_verify_int8kv(
        ctypes.byref(c), _hp(q), B, nq, Hq, _p(block_table), int(block_table.shape[1]), _p(ctx_lens),
        int(max_ctx), float(softmax_scale), _hp(out), _p(workspace), wbytes, ctypes.byref(o),
        _stream(stream)))
    return out


def kvq_decode_step_int8kv(cache, k_new, v_new, q, block_table, ctx_lens, max_ctx, softmax_scale, out=None,
                           workspace=None, split_rows=0, route_threshold=0, force_route=0,
                           stream=None, stage1_events=None, launches=None):
    """One decode step: write each sequence's nq newest tokens (k_new / v_new bf16
    [B][nq][Hkv][D], positions ctx_lens[b] - nq + j) into the cache, then attend with their
    query rows q bf16 [B][nq][Hq][D].  A 3-D q ([B][Hq][D]) with 3-D k_new / v_new
    ([B][Hkv][D]) is the one-token step.  Returns out fp32 shaped like q."""
    squeeze = q.dim() == 3
    if squeeze:
        q, k_new, v_new = q[:, None], k_new[:, None], v_new[:, None]
    B, nq, Hq, D = q.shape
    if out is None:
        out = _new_out((B, nq, Hq, D), q)
        ret = out[:, 0] if squeeze else out
    else:
        ret = out  # the caller's buffer, in the caller's shape ([B][Hq][D] for the one-token step)
    _host_ok("kvq_decode_step_int8kv", q, k_new, v_new, out)
    o = _decode_opts(split_rows, route_threshold, force_route, stage1_events, launches)
    need = int(lib().kvq_verify_workspace_bytes(B, nq, Hq, max(1, int(max_ctx)), D, ctypes.byref(o)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=cache.k.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    c = cache.struct()
    _check("kvq_decode_step_int8kv", lib().kvq_decode_step_int8kv(
        ctypes.byref(c), _hp(k_new), _hp(v_new), _hp(q), B, nq, Hq, _p(block_table), int(block_table.shape[1]),
        _p(ctx_lens), int(max_ctx), float(softmax_scale), _hp(out), _p(workspace), wbytes, ctypes.byref(o),
        _stream(stream)))
    return ret


NOALLOC_SCRATCH_BYTES = 16 << 20


def kvq_attn_decode_int8kv_noalloc(cache, q, block_table, ctx_lens, max_ctx, softmax_scale, out,
                                   split_rows=0, route_threshold=0, force_route=0, stream=None):
    """kvq_attn_decode_int8kv without a workspace argument, for callers that cannot allocate:
    the split-K partials live in a fixed scratch array inside the library.  `out` (fp32
    [B][Hq][D]) must be provided by the caller; nothing is allocated here."""
    B, Hq, D = q.shape
    _host_ok("kvq_attn_decode_int8kv_noalloc", q, out)
    o = _decode_opts(split_rows, route_threshold, force_route)
    c = cache.struct()
    _check("kvq_attn_decode_int8kv_noalloc", lib().kvq_attn_decode_int8kv_noalloc(
        ctypes.byref(c), _hp(q), B, Hq, _p(block_table), int(block_table.shape[1]), _p(ctx_lens),
        int(max_ctx), float(softmax_scale), _hp(out), ctypes.byref(o), _stream(stream)))
    return out


def kvq_debug_fault_inject(mode, wait_budget_cycles=0):
    """Test entry point of the failure path (see kvq.h): mode 0 none, 1 a decode stage-1 copy left
    un-issued, 2 a prefill piece left un-issued; every bounded wait gives up after
    wait_budget_cycles (<= 0: the default)."""
    _check("kvq_debug_fault_inject", lib().kvq_debug_fault_inject(int(mode), int(wait_budget_cycles)))


def kvq_prefill_workspace_bytes(n_tokens, n_q_heads, n_kv_heads, history_len, head_dim):
    return int(lib().kvq_prefill_workspace_bytes(n_tokens, n_q_heads, n_kv_heads, history_len, head_dim))


def kvq_prefill_first_workspace_bytes(n_tokens, n_q_heads, n_kv_heads, head_dim):
    return int(lib().kvq_prefill_first_workspace_bytes(n_tokens, n_q_heads, n_kv_heads, head_dim))


def kvq_attn_prefill_first_bf16(cache, q, k_new, v_new, block_table_row, softmax_scale, out=None, workspace=None,
                                stream=None):
    """The first prefill chunk: q bf16 [T][Hq][D], k_new / v_new bf16 [T][Hkv][D] (positions 0..T-1,
    written into the cache as int8); returns the high-precision causal attention, fp32 [T][Hq][D]."""
    T, Hq, D = q.shape
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(kvq_prefill_first_workspace_bytes(T, Hq, cache.n_kv_heads, D), dtype=torch.uint8,
                                device=q.device)
    c = cache.struct()
    _check("kvq_attn_prefill_first_bf16", lib().kvq_attn_prefill_first_bf16(
        ctypes.byref(c), _p(q), _p(k_new), _p(v_new), T, Hq, _p(block_table_row), int(block_table_row.numel()),
        float(softmax_scale), _p(out), _p(workspace), workspace.numel(), _stream(stream)))
    return out


def kvq_attn_prefill_int8(cache, q, history_len, block_table_row, softmax_scale, out=None,
                          workspace=None, stream=None):
    """q: bf16 [T][Hq][D]; block_table_row int32 [n]; returns out fp32 [T][Hq][D]."""
    T, Hq, D = q.shape
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=q.device)
    need = kvq_prefill_workspace_bytes(T, Hq, cache.n_kv_heads, int(history_len), D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    c = cache.struct()
    _check("kvq_attn_prefill_int8", lib().kvq_attn_prefill_int8(
        ctypes.byref(c), _p(q), T, Hq, int(history_len), _p(block_table_row),
        int(block_table_row.numel()), float(softmax_scale), _p(out), _p(workspace), wbytes,
        _stream(stream)))
    return out


def kvq_attn_prefill_int8_qcodes(cache, q_codes, q_scales, history_len, block_table_row, softmax_scale,
                                 out=None, workspace=None, stream=None):
    """q_codes int8 [T][Hq][D], q_scales fp32 [T][Hq] (from kvq_rope_quant_write); returns fp32 [T][Hq][D]."""
    T, Hq, D = q_codes.shape
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=q_codes.device)
    need = kvq_prefill_workspace_bytes(T, Hq, cache.n_kv_heads, int(history_len), D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_codes.device)
    wbytes = workspace.numel() * workspace.element_size()
    c = cache.struct()
    _check("kvq_attn_prefill_int8_qcodes", lib().kvq_attn_prefill_int8_qcodes(
        ctypes.byref(c), _p(q_codes), _p(q_scales), T, Hq, int(history_len), _p(block_table_row),
        int(block_table_row.numel()), float(softmax_scale), _p(out), _p(workspace), wbytes, _stream(stream)))
    return out


def kvq_sparse_workspace_bytes(n_blocks_row, n_kv_heads, head_dim):
    return int(lib().kvq_sparse_workspace_bytes(n_blocks_row, n_kv_heads, head_dim))


def kvq_attn_sparse_int8kv(cache, q, cell_offsets, cells, block_table_row, softmax_scale,
                           out=None, workspace=None, stream=None):
    """q: bf16 [N][Hq][D]; cell_offsets int32 [N+1]; cells int32; returns fp32 [N][Hq][D]."""
    N, Hq, D = q.shape
    if out is None:
        out = torch.empty((N, Hq, D), dtype=torch.float32, device=q.device)
    nb = int(block_table_row.numel())
    if workspace is None:
        workspace = torch.empty(kvq_sparse_workspace_bytes(nb, cache.n_kv_heads, D), dtype=torch.uint8,
                                device=q.device)
    c = cache.struct()
    _check("kvq_attn_sparse_int8kv", lib().kvq_attn_sparse_int8kv(
        ctypes.byref(c), _p(q), N, Hq, _p(cell_offsets), _p(cells), _p(block_table_row),
        nb, float(softmax_scale), _p(out), _p(workspace), workspace.numel(), _stream(stream)))
    return out


def kvq_debug_prefill_q_codes(q, stream=None):
    """Q quantisation step alone: returns (int8 codes [T][Hq][D], fp32 scales [T][Hq])."""
    T, Hq, D = q.shape
    codes = torch.empty((T, Hq, D), dtype=torch.int8, device=q.device)
    scales = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    _check("kvq_debug_prefill_q_codes", lib().kvq_debug_prefill_q_codes(
        _p(q), T, Hq, D, _p(codes), _p(scales), _stream(stream)))
    return codes, scales


def kvq_debug_prefill_qk_int32(cache, q_codes, q_scales, history_len, block_table_row, softmax_scale, q_head, q0,
                               k0, nk, split_tiles=-1, out=None, workspace=None, stream=None):
    """The production prefill (kvq_attn_prefill_int8_qcodes) that also exports the integer QK scores
    of one unit: returns (S int32 [128][nk] for query rows q0..q0+127 of q_head and keys
    k0..k0+nk-1, out fp32 [T][Hq][D]).  split_tiles: -1 the call's own key-range split, 0 none,
    r > 0 a forced tail of r key tiles."""
    T, Hq, D = q_codes.shape
    s = torch.empty((128, nk), dtype=torch.int32, device=q_codes.device)
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=q_codes.device)
    need = kvq_prefill_workspace_bytes(T, Hq, cache.n_kv_heads, int(history_len), D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_codes.device)
    c = cache.struct()
    _check("kvq_debug_prefill_qk_int32", lib().kvq_debug_prefill_qk_int32(
        ctypes.byref(c), _p(q_codes), _p(q_scales), T, Hq, int(history_len), _p(block_table_row),
        int(block_table_row.numel()), float(softmax_scale), int(split_tiles), int(q_head), int(q0), int(k0), int(nk),
        _p(s), _p(out), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return s, out


def kvq_debug_stream_floor(cache, block_table, ctx_lens, max_ctx, split_rows=0, stream=None):
    """The K/V stream of decode stage 1 alone (same grid, rings and copies, no arithmetic)."""
    c = cache.struct()
    _check("kvq_debug_stream_floor", lib().kvq_debug_stream_floor(
        ctypes.byref(c), int(block_table.shape[0]), _p(block_table), int(block_table.shape[1]), _p(ctx_lens),
        int(max_ctx), int(split_rows), _stream(stream)))
