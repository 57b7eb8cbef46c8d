"""ctypes marshalling for libpkv.so (argument checks and pointers only)."""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(PKG, "libpkv.so")
_lib = None

DEV_ERR_BITS = {
    "SLOT_RANGE": 1,
    "QSL": 2,
    "SEQ_LEN": 4,
    "BT_WIDTH": 8,
    "BLOCK_ID": 16,
    "TIMEOUT": 32,
    "INT8_PREFILL": 64,
    "CAPACITY": 128,
}

EXPORTS = ["pkv_write", "pkv_attention", "pkv_reserve_workspace", "pkv_get_error",
           "pkv_last_error_string", "pkv_num_sms", "pkv_trace_enable", "pkv_trace_read",
           "pkv_launch_count", "pkv_prepare_step", "pkv_write_int8", "pkv_attention_int8",
           "pkv_plan", "pkv_attention_planned", "pkv_workspace_size"]
TRACE_KINDS = ["write", "plan", "decode", "prefill", "combine", "prepare"]


class PkvError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("pkv error %d: %s" % (code, msg))
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load():
    """Loads libpkv.so (built by ``build.py`` / ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise PkvError(-100, "libpkv.so is not built (%s); run __graft_entry__.build()" % _LIB_PATH)
    L = ctypes.CDLL(_LIB_PATH)
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    L.pkv_write.restype = ctypes.c_int
    L.pkv_write.argtypes = [vp, i64, vp, i64, vp, vp, i64, i32, i32, i32, vp, i64, vp]
    L.pkv_attention.restype = ctypes.c_int
    L.pkv_attention.argtypes = [vp, i64, i64, i32, vp, vp, i64, i32, i32, i32, vp, vp, vp, i64,
                                i32, f32, vp, i64, vp]
    f32 = ctypes.c_float
    L.pkv_write_int8.restype = ctypes.c_int
    L.pkv_write_int8.argtypes = [vp, i64, vp, i64, vp, vp, f32, f32, i64, i32, i32, i32, vp, i64,
                                 vp]
    L.pkv_attention_int8.restype = ctypes.c_int
    L.pkv_attention_int8.argtypes = [vp, i64, i64, i32, vp, vp, f32, f32, i64, i32, i32, i32, vp,
                                     vp, vp, i64, i32, f32, vp, i64, vp]
    L.pkv_plan.restype = ctypes.c_int
    L.pkv_plan.argtypes = [i64, i32, i32, vp, vp, i64, i32, vp]
    L.pkv_attention_planned.restype = ctypes.c_int
    L.pkv_attention_planned.argtypes = [vp, i64, i32, vp, vp, i64, i32, i32, i32, vp, f32, vp,
                                        i64, vp]
    L.pkv_reserve_workspace.restype = ctypes.c_int
    L.pkv_reserve_workspace.argtypes = [i32, i64, i64, i32, i32]
    L.pkv_get_error.restype = ctypes.c_int
    L.pkv_get_error.argtypes = [vp, ctypes.POINTER(i32)]
    L.pkv_last_error_string.restype = ctypes.c_char_p
    L.pkv_last_error_string.argtypes = []
    L.pkv_num_sms.restype = ctypes.c_int
    L.pkv_num_sms.argtypes = []
    L.pkv_trace_enable.restype = ctypes.c_int
    L.pkv_trace_enable.argtypes = [ctypes.c_int]
    L.pkv_trace_read.restype = ctypes.c_int
    L.pkv_trace_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64),
                                 ctypes.c_int]
    L.pkv_launch_count.restype = i64
    L.pkv_launch_count.argtypes = []
    _lib = L
    return L


def _check(rc):
    if rc != 0:
        msg = load().pkv_last_error_string().decode(errors="replace")
        raise PkvError(rc, msg)


_torch = None
_raw_stream = None  # () -> the current device's current stream handle, as an int


def _T():
    """torch, imported on first use (the binding loads without it)."""
    global _torch, _raw_stream
    if _torch is None:
        import torch
        get_dev = getattr(torch._C, "_cuda_getDevice", None)
        get_raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if get_dev is not None and get_raw is not None:
            _raw_stream = lambda: get_raw(get_dev())  # noqa: E731
        else:
            _raw_stream = lambda: torch.cuda.current_stream().cuda_stream  # noqa: E731
        _torch = torch
    return _torch


def _stream(stream):
    """The stream handle for a call: torch's current stream when none is given
    (read through torch's raw getter: a Stream object costs microseconds)."""
    if stream is None:
        if _raw_stream is None:
            _T()
        return _raw_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _require(t, dtype, name, device=True):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)


def _per_row(t):
    """Elements in one row of a [rows, ...] tensor (also when it has no rows)."""
    n = 1
    for x in t.shape[1:]:
        n *= x
    return n


def _rows3(t, name):
    """Row stride of a [rows, heads, 128] tensor whose per-row block is contiguous."""
    st, sh = t.stride(), t.shape
    if len(st) == 2:
        if st[1] != 1:
            raise ValueError("%s: last dimension must be contiguous" % name)
        return st[0]
    if len(st) != 3 or st[2] != 1 or st[1] != sh[2]:
        raise ValueError("%s must be [rows, heads, head_size] with contiguous rows" % name)
    return st[0]


def _all_on_device(dtype, *ts):
    """True when every tensor has this dtype and lives on a CUDA device (the
    common case, tested in one pass; callers fall back to the per-argument
    checks, which name the culprit, when it is False)."""
    try:
        for t in ts:
            if t.dtype is not dtype or not t.is_cuda:
                return False
    except AttributeError:
        return False
    return True


def pkv_write(k, v, key_cache, value_cache, slot_mapping, n_tokens=None, stream=None):
    """Scatters k/v ([n, Hkv, 128] bf16) into the caches at slot_mapping (int64)."""
    torch = _T()
    if not (_all_on_device(torch.bfloat16, k, v, key_cache, value_cache) and
            _all_on_device(torch.int64, slot_mapping)):
        for t, n in ((k, "k"), (v, "v"), (key_cache, "key_cache"), (value_cache, "value_cache")):
            _require(t, torch.bfloat16, n)
        _require(slot_mapping, torch.int64, "slot_mapping")
    ks = key_cache.shape
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()) or len(ks) != 4:
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, head_size]")
    if ks != value_cache.shape:
        raise ValueError("key_cache and value_cache shapes differ")
    if not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous")
    nb, bs, hkv, d = ks
    n = slot_mapping.shape[0] if n_tokens is None else int(n_tokens)
    if n > slot_mapping.shape[0] or n > k.shape[0] or n > v.shape[0]:
        raise ValueError("n_tokens exceeds the rows of k/v/slot_mapping")
    _check(load().pkv_write(k.data_ptr(), _rows3(k, "k"), v.data_ptr(), _rows3(v, "v"),
                            key_cache.data_ptr(), value_cache.data_ptr(), nb, bs, hkv, d,
                            slot_mapping.data_ptr(), n, _stream(stream)))


def pkv_attention(q, key_cache, value_cache, query_start_loc, seq_lens, block_table, num_reqs,
                  scale, out, stream=None):
    """Causal varlen attention of q ([T, Hq, 128] bf16) over the paged cache
    into out ([T, Hq, 128] bf16); see include/pkv.h for the contract."""
    torch = _T()
    metadata = ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"),
                (block_table, "block_table"))
    if not (_all_on_device(torch.bfloat16, q, key_cache, value_cache, out) and
            _all_on_device(torch.int32, query_start_loc, seq_lens, block_table)):
        for t, n in ((q, "q"), (key_cache, "key_cache"), (value_cache, "value_cache"),
                     (out, "out")):
            _require(t, torch.bfloat16, n)
        for t, n in metadata:
            _require(t, torch.int32, n)
    for t, n in metadata:
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    ks = key_cache.shape
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()) or len(ks) != 4:
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, head_size]")
    if ks != value_cache.shape:
        raise ValueError("key_cache and value_cache shapes differ")
    nb, bs, hkv, d = ks
    qs = q.shape
    if len(qs) != 3:
        raise ValueError("q must be [rows, num_heads, head_size]")
    rows, hq, _ = qs
    if out.shape[0] < rows or _per_row(out) != hq * d:
        raise ValueError("out must hold [rows, num_heads * head_size]")
    bts = block_table.shape
    bt_width = bts[1] if len(bts) == 2 else bts[0]
    num_reqs = int(num_reqs)
    if num_reqs > 0 and (query_start_loc.numel() < num_reqs + 1 or
                         seq_lens.numel() < num_reqs or
                         (len(bts) == 2 and bts[0] < num_reqs)):
        raise ValueError("metadata shorter than num_reqs")
    _check(load().pkv_attention(q.data_ptr(), _rows3(q, "q"), rows, hq, key_cache.data_ptr(),
                                value_cache.data_ptr(), nb, bs, hkv, d,
                                query_start_loc.data_ptr(), seq_lens.data_ptr(),
                                block_table.data_ptr(), bt_width, num_reqs, float(scale),
                                out.data_ptr(), _rows3(out, "out"), _stream(stream)))


def _caches(key_cache, value_cache, dtype):
    import torch
    for t, n in ((key_cache, "key_cache"), (value_cache, "value_cache")):
        _require(t, dtype, n)
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()) or key_cache.dim() != 4:
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, head_size]")
    if key_cache.shape != value_cache.shape:
        raise ValueError("key_cache and value_cache shapes differ")
    return key_cache.shape


def pkv_write_int8(k, v, key_cache, value_cache, slot_mapping, k_scale, v_scale, n_tokens=None,
                   stream=None):
    """Quantises k/v ([n, Hkv, 128] bf16) into the int8 caches at slot_mapping:
    code = clamp(rne(x / scale), -127, 127), one fp32 scale per cache."""
    import torch
    _require(k, torch.bfloat16, "k")
    _require(v, torch.bfloat16, "v")
    nb, bs, hkv, d = _caches(key_cache, value_cache, torch.int8)
    _require(slot_mapping, torch.int64, "slot_mapping")
    if not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous")
    n = slot_mapping.shape[0] if n_tokens is None else int(n_tokens)
    if n > slot_mapping.shape[0] or n > k.shape[0] or n > v.shape[0]:
        raise ValueError("n_tokens exceeds the rows of k/v/slot_mapping")
    _check(load().pkv_write_int8(k.data_ptr(), _rows3(k, "k"), v.data_ptr(), _rows3(v, "v"),
                                 key_cache.data_ptr(), value_cache.data_ptr(), float(k_scale),
                                 float(v_scale), nb, bs, hkv, d, slot_mapping.data_ptr(), n,
                                 _stream(stream)))


def pkv_attention_int8(q, key_cache, value_cache, k_scale, v_scale, query_start_loc, seq_lens,
                       block_table, num_reqs, scale, out, stream=None):
    """pkv_attention over int8 caches (K = code * k_scale, V = code * v_scale),
    decode-path requests only; see include/pkv.h."""
    import torch
    _require(q, torch.bfloat16, "q")
    _require(out, torch.bfloat16, "out")
    nb, bs, hkv, d = _caches(key_cache, value_cache, torch.int8)
    for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"),
                 (block_table, "block_table")):
        _require(t, torch.int32, n)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    if q.dim() != 3:
        raise ValueError("q must be [rows, num_heads, head_size]")
    rows, hq, _ = q.shape
    if out.shape[0] < rows or _per_row(out) != hq * d:
        raise ValueError("out must hold [rows, num_heads * head_size]")
    bt_width = block_table.shape[1] if block_table.dim() == 2 else block_table.shape[0]
    if int(num_reqs) > 0 and (query_start_loc.numel() < int(num_reqs) + 1 or
                              seq_lens.numel() < int(num_reqs) or
                              (block_table.dim() == 2 and block_table.shape[0] < int(num_reqs))):
        raise ValueError("metadata shorter than num_reqs")
    _check(load().pkv_attention_int8(q.data_ptr(), _rows3(q, "q"), rows, hq, key_cache.data_ptr(),
                                     value_cache.data_ptr(), float(k_scale), float(v_scale), nb,
                                     bs, hkv, d, query_start_loc.data_ptr(), seq_lens.data_ptr(),
                                     block_table.data_ptr(), bt_width, int(num_reqs),
                                     float(scale), out.data_ptr(), _rows3(out, "out"),
                                     _stream(stream)))


def pkv_plan(q_rows, num_heads, num_kv_heads, query_start_loc, seq_lens, block_table_width,
             num_reqs, stream=None):
    """Builds one step plan on the current device, for pkv_attention_planned
    calls (one per layer) that follow it; see include/pkv.h."""
    import torch
    for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens")):
        _require(t, torch.int32, n)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    if int(num_reqs) > 0 and (query_start_loc.numel() < int(num_reqs) + 1 or
                              seq_lens.numel() < int(num_reqs)):
        raise ValueError("metadata shorter than num_reqs")
    _check(load().pkv_plan(int(q_rows), int(num_heads), int(num_kv_heads),
                           query_start_loc.data_ptr(), seq_lens.data_ptr(),
                           int(block_table_width), int(num_reqs), _stream(stream)))


def pkv_attention_planned(q, key_cache, value_cache, block_table, scale, out, stream=None):
    """One layer's attention on the current step plan (pkv_plan)."""
    torch = _T()
    if not (_all_on_device(torch.bfloat16, q, key_cache, value_cache, out) and
            _all_on_device(torch.int32, block_table)):
        for t, n in ((q, "q"), (key_cache, "key_cache"), (value_cache, "value_cache"),
                     (out, "out")):
            _require(t, torch.bfloat16, n)
        _require(block_table, torch.int32, "block_table")
    if not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous")
    nb, bs, hkv, d = _caches(key_cache, value_cache, torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [rows, num_heads, head_size]")
    rows, hq, _ = q.shape
    if out.shape[0] < rows or _per_row(out) != hq * d:
        raise ValueError("out must hold [rows, num_heads * head_size]")
    _check(load().pkv_attention_planned(q.data_ptr(), _rows3(q, "q"), hq, key_cache.data_ptr(),
                                        value_cache.data_ptr(), nb, bs, hkv, d,
                                        block_table.data_ptr(), float(scale), out.data_ptr(),
                                        _rows3(out, "out"), _stream(stream)))


def pkv_reserve_workspace(max_reqs, max_q_rows, block_table_width, num_heads, num_kv_heads):
    _check(load().pkv_reserve_workspace(int(max_reqs), int(max_q_rows), int(block_table_width),
                                        int(num_heads), int(num_kv_heads)))


class WorkspaceInfo(ctypes.Structure):
    """Mirror of pkv_workspace_info (include/pkv.h)."""
    _fields_ = [("bytes", ctypes.c_int64), ("decode_units", ctypes.c_int64),
                ("prefill_tiles", ctypes.c_int64), ("split_pairs", ctypes.c_int64),
                ("partial_rows", ctypes.c_int64), ("decode_workers", ctypes.c_int32),
                ("decode_workers_int8", ctypes.c_int32)]


def pkv_workspace_size(max_reqs, max_q_rows, block_table_width, num_heads, num_kv_heads,
                       num_sms) -> dict:
    """Bytes and plan capacities of the workspace pkv_reserve_workspace would
    hold for these sizes on a device with num_sms SMs (host-only)."""
    L = load()
    fn = L.pkv_workspace_size
    if fn.argtypes is None:
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                       ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(WorkspaceInfo)]
    info = WorkspaceInfo()
    _check(fn(int(max_reqs), int(max_q_rows), int(block_table_width), int(num_heads),
              int(num_kv_heads), int(num_sms), ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in WorkspaceInfo._fields_}


def pkv_get_error(stream=None) -> int:
    """Synchronises the stream; returns and clears the device error words
    (the allocating calls' and pkv_attention_noalloc's)."""
    bits = ctypes.c_int32(0)
    _check(load().pkv_get_error(_stream(stream), ctypes.byref(bits)))
    return bits.value


def pkv_num_sms() -> int:
    return load().pkv_num_sms()


def pkv_trace_enable(on: bool) -> None:
    load().pkv_trace_enable(1 if on else 0)


def pkv_trace_read():
    """{kind: (total ms, launches)} of the traced launches since the last read."""
    n = len(TRACE_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    rc = load().pkv_trace_read(ms, cnt, n)
    if rc < 0:
        _check(rc)
    return {k: (ms[i], cnt[i]) for i, k in enumerate(TRACE_KINDS)}


def pkv_launch_count() -> int:
    return load().pkv_launch_count()


def pkv_attention_noalloc(q, key_cache, value_cache, query_start_loc, seq_lens, block_table,
                          num_reqs, scale, out, stream=None):
    """pkv_attention computed with the library's static scratch array instead
    of a cudaMalloc'd workspace, for callers that cannot allocate device
    memory (see include/pkv.h).  Same arguments and result; raises PkvError
    with the return code when a host check refuses the call."""
    import torch
    L = load()
    fn = L.pkv_attention_noalloc
    if fn.argtypes is None:
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
        fn.restype = ctypes.c_int
        fn.argtypes = [vp, i64, i64, i32, vp, vp, i64, i32, i32, i32, vp, vp, vp, i64, i32, f32,
                       vp, i64, vp]
    for t, n in ((q, "q"), (key_cache, "key_cache"), (value_cache, "value_cache"), (out, "out")):
        _require(t, torch.bfloat16, n)
    for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"),
                 (block_table, "block_table")):
        _require(t, torch.int32, n)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()) or key_cache.dim() != 4:
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, head_size]")
    nb, bs, hkv, d = key_cache.shape
    rows, hq, _ = q.shape
    bt_width = block_table.shape[1] if block_table.dim() == 2 else block_table.shape[0]
    rc = fn(q.data_ptr(), _rows3(q, "q"), rows, hq, key_cache.data_ptr(), value_cache.data_ptr(),
            nb, bs, hkv, d, query_start_loc.data_ptr(), seq_lens.data_ptr(),
            block_table.data_ptr(), bt_width, int(num_reqs), float(scale), out.data_ptr(),
            _rows3(out, "out"), _stream(stream))
    if rc != 0:
        raise PkvError(rc, "pkv_attention_noalloc refused the call")


def pkv_prepare_step(query_start_loc, num_computed, persistent_block_table, num_reqs,
                     num_tokens_padded, positions, seq_lens, slot_mapping, block_table=None,
                     idx_mapping=None, stream=None):
    """Positions, seq_lens, slot mapping and the batch-order block table on
    the device (see include/pkv.h)."""
    import torch
    L = load()
    fn = L.pkv_prepare_step
    if fn.argtypes is None:
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        fn.restype = ctypes.c_int
        fn.argtypes = [vp, vp, vp, vp, i64, i64, i32, i64, vp, vp, vp, vp, vp]
    for t, n, dt in ((query_start_loc, "query_start_loc", torch.int32),
                     (num_computed, "num_computed", torch.int32),
                     (persistent_block_table, "persistent_block_table", torch.int32),
                     (positions, "positions", torch.int64), (seq_lens, "seq_lens", torch.int32),
                     (slot_mapping, "slot_mapping", torch.int64)):
        _require(t, dt, n)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % n)
    if block_table is not None:
        _require(block_table, torch.int32, "block_table")
    if idx_mapping is not None:
        _require(idx_mapping, torch.int32, "idx_mapping")
    rows, width = persistent_block_table.shape
    _check(fn(query_start_loc.data_ptr(), num_computed.data_ptr(),
              idx_mapping.data_ptr() if idx_mapping is not None else None,
              persistent_block_table.data_ptr(), rows, width, int(num_reqs),
              int(num_tokens_padded), positions.data_ptr(), seq_lens.data_ptr(),
              slot_mapping.data_ptr(), block_table.data_ptr() if block_table is not None else None,
              _stream(stream)))
