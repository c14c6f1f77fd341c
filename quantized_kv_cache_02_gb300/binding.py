"""ctypes binding of libkvq.so (include/kvq.h): the same entry points under the
same names, plus ``KVQCache``, a small owner object that allocates the arena
with torch and passes torch's current CUDA stream.  Argument marshalling only:
all work runs in the library's CUDA kernels.  Importing fails loudly when the
library has not been built; there is no other implementation to fall back on.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK, KVQ_EINVAL, KVQ_ECAPACITY, KVQ_ENOMEM, KVQ_ECUDA, KVQ_EUNSUPPORTED, KVQ_EDEVICE = range(7)
KVQ_BF16, KVQ_FP32 = 0, 1
STATUS_NAMES = {0: "KVQ_OK", 1: "KVQ_EINVAL", 2: "KVQ_ECAPACITY", 3: "KVQ_ENOMEM", 4: "KVQ_ECUDA",
                5: "KVQ_EUNSUPPORTED", 6: "KVQ_EDEVICE"}

# Every function include/kvq.h declares.
EXPORTED = ("kvq_required_bytes", "kvq_create", "kvq_append", "kvq_decode_attention",
            "kvq_decode_attention_ex", "kvq_bytes", "kvq_ledger", "kvq_seq_state", "kvq_export_unit",
            "kvq_export_pages", "kvq_device_status", "kvq_page_bytes", "kvq_kernel_launches", "kvq_destroy",
            "kvq_last_error", "kvq_decode_attention_noalloc", "kvq_restore", "kvq_dense_decode_attention",
            "kvq_compare", "kvq_required_bytes_paged", "kvq_create_paged", "kvq_release", "kvq_pool_state",
            "kvq_required_bytes_segmented", "kvq_create_segmented", "kvq_decode_step")


class kvq_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("residual_len", ctypes.c_int32), ("group", ctypes.c_int32),
                ("qmax", ctypes.c_int32), ("dtype", ctypes.c_int32), ("eps", ctypes.c_float)]


class kvq_bytes_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("code_bytes", "n_scales", "scale_bytes", "window_elems",
                                              "window_bytes", "total", "allocated")]


class kvq_seq_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("total", "quantized", "window", "last_flushed", "n_groups",
                                              "capacity")]


class kvq_unit_view(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("v_scales", ctypes.c_void_p), ("window_k", ctypes.c_void_p), ("window_v", ctypes.c_void_p)]


class kvq_decode_opts(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("chunk_pages", ctypes.c_int32), ("split_start", ctypes.c_void_p),
                ("split_stop", ctypes.c_void_p)]


class kvq_compare_t(ctypes.Structure):
    _fields_ = [("key_mse", ctypes.c_double), ("value_mse", ctypes.c_double)] + [
        (n, ctypes.c_int64) for n in ("n_key_scales", "n_value_scales", "raw_bytes", "container_quantized_bytes",
                                      "packed_quantized_bytes")]


class KVQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvq.so and declare its signatures (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, V, I32, I64, SZ = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sigs = {
        "kvq_required_bytes": ([P(kvq_config), P(I64), P(SZ)], ctypes.c_int),
        "kvq_create": ([P(kvq_config), P(I64), V, SZ, P(V)], ctypes.c_int),
        "kvq_append": ([V, V, V, I64, I32, I32, V], ctypes.c_int),
        "kvq_decode_attention": ([V, V, V, V], ctypes.c_int),
        "kvq_decode_attention_ex": ([V, V, V, V, P(kvq_decode_opts)], ctypes.c_int),
        "kvq_bytes": ([V, P(kvq_bytes_t)], ctypes.c_int),
        "kvq_ledger": ([P(kvq_config), P(I64), P(kvq_bytes_t)], ctypes.c_int),
        "kvq_seq_state": ([V, I32, P(kvq_seq_info)], ctypes.c_int),
        "kvq_export_unit": ([V, I32, I32, P(kvq_unit_view), V], ctypes.c_int),
        "kvq_export_pages": ([V, I32, I32, V, SZ, V], ctypes.c_int),
        "kvq_device_status": ([V, P(I32), V], ctypes.c_int),
        "kvq_page_bytes": ([P(kvq_config)], SZ),
        "kvq_kernel_launches": ([], ctypes.c_uint64),
        "kvq_decode_attention_noalloc": ([V, V, V, V], ctypes.c_int),
        "kvq_decode_step": ([V, V, V, V, V, V, P(kvq_decode_opts)], ctypes.c_int),
        "kvq_restore": ([V, I32, I32, V, V, I64, ctypes.c_int, V], ctypes.c_int),
        "kvq_dense_decode_attention": ([V, V, V, I64, V, V, V], ctypes.c_int),
        "kvq_compare": ([V, V, I64, I32, I64, I32, ctypes.c_int, I32, ctypes.c_float, I32, V, P(kvq_compare_t), V],
                        ctypes.c_int),
        "kvq_required_bytes_paged": ([P(kvq_config), P(I64), I64, P(SZ)], ctypes.c_int),
        "kvq_create_paged": ([P(kvq_config), P(I64), I64, V, SZ, P(V)], ctypes.c_int),
        "kvq_required_bytes_segmented": ([P(kvq_config), P(I64), P(SZ)], ctypes.c_int),
        "kvq_create_segmented": ([P(kvq_config), P(I64), V, SZ, P(V)], ctypes.c_int),
        "kvq_release": ([V, I32, I32], ctypes.c_int),
        "kvq_pool_state": ([V, P(I64), P(I64)], ctypes.c_int),
        "kvq_destroy": ([V], None),
        "kvq_last_error": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != KVQ_OK:
        raise KVQError(status, load_library().kvq_last_error().decode())


def make_config(batch, n_kv_heads, n_q_heads, head_dim, residual_len, group, qmax, dtype=KVQ_BF16, eps=1e-8):
    return kvq_config(batch, n_kv_heads, n_q_heads, head_dim, residual_len, group, qmax, dtype, eps)


def _i64_array(values):
    values = [int(v) for v in values]
    return (ctypes.c_int64 * len(values))(*values)


# ---- thin wrappers with the C names --------------------------------------------

def kvq_required_bytes(cfg: kvq_config, capacity) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().kvq_required_bytes(ctypes.byref(cfg), _i64_array(capacity), ctypes.byref(out)))
    return out.value


def kvq_ledger(cfg: kvq_config, tokens) -> dict:
    out = kvq_bytes_t()
    _check(load_library().kvq_ledger(ctypes.byref(cfg), _i64_array(tokens), ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in kvq_bytes_t._fields_}


def kvq_page_bytes(cfg: kvq_config) -> int:
    return load_library().kvq_page_bytes(ctypes.byref(cfg))


def kvq_required_bytes_paged(cfg: kvq_config, capacity, pool_blocks: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().kvq_required_bytes_paged(ctypes.byref(cfg), _i64_array(capacity), pool_blocks,
                                                   ctypes.byref(out)))
    return out.value


def kvq_create_paged(cfg: kvq_config, capacity, pool_blocks: int, device_ptr: int, device_bytes: int) -> int:
    handle = ctypes.c_void_p()
    _check(load_library().kvq_create_paged(ctypes.byref(cfg), _i64_array(capacity), pool_blocks,
                                           ctypes.c_void_p(device_ptr), device_bytes, ctypes.byref(handle)))
    return handle.value


def kvq_required_bytes_segmented(cfg: kvq_config, capacity) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().kvq_required_bytes_segmented(ctypes.byref(cfg), _i64_array(capacity), ctypes.byref(out)))
    return out.value


def kvq_create_segmented(cfg: kvq_config, capacity, device_ptr: int, device_bytes: int) -> int:
    handle = ctypes.c_void_p()
    _check(load_library().kvq_create_segmented(ctypes.byref(cfg), _i64_array(capacity), ctypes.c_void_p(device_ptr),
                                               device_bytes, ctypes.byref(handle)))
    return handle.value


def kvq_release(handle, seq_begin: int, n_seqs: int) -> None:
    _check(load_library().kvq_release(handle, seq_begin, n_seqs))


def kvq_pool_state(handle) -> tuple:
    free, total = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(load_library().kvq_pool_state(handle, ctypes.byref(free), ctypes.byref(total)))
    return free.value, total.value


def kvq_create(cfg: kvq_config, capacity, device_ptr: int, device_bytes: int) -> int:
    handle = ctypes.c_void_p()
    _check(load_library().kvq_create(ctypes.byref(cfg), _i64_array(capacity), ctypes.c_void_p(device_ptr),
                                     device_bytes, ctypes.byref(handle)))
    return handle.value


def kvq_append(handle, new_k_ptr, new_v_ptr, n_tokens, seq_begin, n_seqs, stream) -> None:
    _check(load_library().kvq_append(handle, new_k_ptr, new_v_ptr, n_tokens, seq_begin, n_seqs, stream))


def kvq_decode_attention(handle, q_ptr, out_ptr, stream) -> None:
    _check(load_library().kvq_decode_attention(handle, q_ptr, out_ptr, stream))


def kvq_decode_attention_ex(handle, q_ptr, out_ptr, stream, kernel=0, chunk_pages=0, split_start=None,
                            split_stop=None) -> None:
    opts = kvq_decode_opts(kernel, chunk_pages, split_start, split_stop)
    _check(load_library().kvq_decode_attention_ex(handle, q_ptr, out_ptr, stream, ctypes.byref(opts)))


def kvq_decode_step(handle, k_ptr, v_ptr, q_ptr, out_ptr, stream, kernel=0, split_start=None, split_stop=None):
    opts = kvq_decode_opts(kernel, 0, split_start, split_stop)
    _check(load_library().kvq_decode_step(handle, k_ptr, v_ptr, q_ptr, out_ptr, stream, ctypes.byref(opts)))


def kvq_decode_attention_noalloc(handle, q_ptr, out_ptr, stream) -> None:
    """Decode attention with the split scratch in the library's fixed device
    array (for callers that cannot allocate device memory at call time)."""
    _check(load_library().kvq_decode_attention_noalloc(handle, q_ptr, out_ptr, stream))


def kvq_bytes(handle) -> dict:
    out = kvq_bytes_t()
    _check(load_library().kvq_bytes(handle, ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in kvq_bytes_t._fields_}


def kvq_seq_state(handle, seq: int) -> dict:
    out = kvq_seq_info()
    _check(load_library().kvq_seq_state(handle, seq, ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in kvq_seq_info._fields_}


def kvq_export_unit(handle, seq, kv_head, view: kvq_unit_view, stream) -> None:
    _check(load_library().kvq_export_unit(handle, seq, kv_head, ctypes.byref(view), stream))


def kvq_export_pages(handle, seq, kv_head, dst_ptr, dst_bytes, stream) -> None:
    _check(load_library().kvq_export_pages(handle, seq, kv_head, dst_ptr, dst_bytes, stream))


def kvq_device_status(handle, stream) -> int:
    word = ctypes.c_int32(0)
    status = load_library().kvq_device_status(handle, ctypes.byref(word), stream)
    if status not in (KVQ_OK, KVQ_EDEVICE):
        _check(status)
    return word.value


def kvq_restore(handle, seq_begin, n_seqs, k_ptr, v_ptr, t_stride, out_dtype, stream) -> None:
    _check(load_library().kvq_restore(handle, seq_begin, n_seqs, k_ptr, v_ptr, t_stride, out_dtype, stream))


def kvq_dense_decode_attention(handle, k_ptr, v_ptr, t_stride, q_ptr, out_ptr, stream) -> None:
    _check(load_library().kvq_dense_decode_attention(handle, k_ptr, v_ptr, t_stride, q_ptr, out_ptr, stream))


def kvq_compare(key_ptr, value_ptr, batch, heads, tokens, head_dim, dtype, qmax, eps, group, workspace_ptr,
                stream) -> dict:
    out = kvq_compare_t()
    _check(load_library().kvq_compare(key_ptr, value_ptr, batch, heads, tokens, head_dim, dtype, qmax, eps, group,
                                      workspace_ptr, ctypes.byref(out), stream))
    return {n: getattr(out, n) for n, _ in kvq_compare_t._fields_}


def compare(key, value, qmax=7, eps=1e-8, group=0) -> dict:
    """The page's compare on device tensors key, value [batch, heads, tokens,
    head_dim] (bf16 or fp32, contiguous, same shape and dtype)."""
    import torch
    assert key.is_cuda and key.shape == value.shape and key.dtype == value.dtype
    assert key.is_contiguous() and value.is_contiguous() and key.dim() == 4
    dt = {torch.bfloat16: KVQ_BF16, torch.float32: KVQ_FP32}[key.dtype]
    ws = torch.empty(2, dtype=torch.float64, device=key.device)
    b, h, t, d = key.shape
    return kvq_compare(key.data_ptr(), value.data_ptr(), b, h, t, d, dt, qmax, eps, group, ws.data_ptr(),
                       torch.cuda.current_stream(key.device).cuda_stream)


def kvq_kernel_launches() -> int:
    return load_library().kvq_kernel_launches()


def kvq_destroy(handle) -> None:
    if handle:
        load_library().kvq_destroy(handle)


# ---- owner object ------------------------------------------------------------

class KVQCache:
    """One layer's quantized cache on the current CUDA device.  The arena is a
    torch uint8 tensor kept alive by this object; every call runs on torch's
    current stream."""

    def __init__(self, batch, n_kv_heads, n_q_heads, head_dim, residual_len, group, qmax, capacity,
                 dtype="bf16", eps=1e-8, device=None, pool_blocks=0, segmented=False):
        """pool_blocks > 0 makes a paged cache: ``capacity`` then bounds each
        sequence's length and the pool of blocks is shared.  segmented=True
        makes a cache that flushes each append's whole overflow as one segment
        (``group`` is then unused)."""
        import torch
        self.torch = torch
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.dtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.cfg = make_config(batch, n_kv_heads, n_q_heads, head_dim, residual_len, group, qmax,
                               KVQ_BF16 if dtype == "bf16" else KVQ_FP32, eps)
        if isinstance(capacity, int):
            capacity = [capacity] * batch
        self.capacity = list(capacity)
        self.pool_blocks = pool_blocks
        self.segmented = segmented
        if segmented:
            self.nbytes = kvq_required_bytes_segmented(self.cfg, self.capacity)
        elif pool_blocks:
            self.nbytes = kvq_required_bytes_paged(self.cfg, self.capacity, pool_blocks)
        else:
            self.nbytes = kvq_required_bytes(self.cfg, self.capacity)
        self.arena = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=self.device)
        base = self.arena.data_ptr()
        self._base = (base + 255) // 256 * 256
        with torch.cuda.device(self.device):
            if segmented:
                self.handle = kvq_create_segmented(self.cfg, self.capacity, self._base, self.nbytes)
            elif pool_blocks:
                self.handle = kvq_create_paged(self.cfg, self.capacity, pool_blocks, self._base, self.nbytes)
            else:
                self.handle = kvq_create(self.cfg, self.capacity, self._base, self.nbytes)

    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def _check_input(self, t, shape):
        assert t.is_cuda and t.device == self.device, "input must live on the cache's device"
        assert t.dtype == self.dtype and t.is_contiguous(), f"input must be contiguous {self.dtype}"
        assert tuple(t.shape) == tuple(shape), f"expected shape {tuple(shape)}, got {tuple(t.shape)}"

    def append(self, new_k, new_v, seq_begin=0):
        """new_k, new_v: [n_seqs, n_kv_heads, n_tokens, head_dim] on the device."""
        n_seqs, _, n, _ = new_k.shape
        shape = (n_seqs, self.cfg.n_kv_heads, n, self.cfg.head_dim)
        self._check_input(new_k, shape)
        self._check_input(new_v, shape)
        kvq_append(self.handle, new_k.data_ptr(), new_v.data_ptr(), n, seq_begin, n_seqs, self._stream())

    def decode_attention(self, q, out=None, kernel=0, chunk_pages=0, split_start=None, split_stop=None):
        """q: [batch, n_q_heads, head_dim]; returns float32 [batch, n_q_heads, head_dim]."""
        shape = (self.cfg.batch, self.cfg.n_q_heads, self.cfg.head_dim)
        self._check_input(q, shape)
        if out is None:
            out = self.torch.empty(shape, dtype=self.torch.float32, device=self.device)
        if kernel == 0 and chunk_pages == 0 and split_start is None and split_stop is None:
            kvq_decode_attention(self.handle, q.data_ptr(), out.data_ptr(), self._stream())
        else:
            kvq_decode_attention_ex(self.handle, q.data_ptr(), out.data_ptr(), self._stream(), kernel, chunk_pages,
                                    split_start, split_stop)
        return out

    def restore(self, seq_begin=0, n_seqs=None, t_stride=None, out_dtype="bf16", k_out=None, v_out=None):
        """Dense restored Keys and Values [n_seqs, n_kv_heads, t_stride, head_dim]
        (rows past each sequence's length are left as allocated)."""
        n_seqs = self.cfg.batch - seq_begin if n_seqs is None else n_seqs
        if t_stride is None:
            t_stride = max(1, max(self.seq_state(b)["total"] for b in range(seq_begin, seq_begin + n_seqs)))
        dt = self.torch.bfloat16 if out_dtype == "bf16" else self.torch.float32
        shape = (n_seqs, self.cfg.n_kv_heads, t_stride, self.cfg.head_dim)
        if k_out is None:
            k_out = self.torch.zeros(shape, dtype=dt, device=self.device)
        if v_out is None:
            v_out = self.torch.zeros(shape, dtype=dt, device=self.device)
        assert tuple(k_out.shape) == shape and tuple(v_out.shape) == shape
        assert k_out.dtype == dt and v_out.dtype == dt and k_out.is_contiguous() and v_out.is_contiguous()
        kvq_restore(self.handle, seq_begin, n_seqs, k_out.data_ptr(), v_out.data_ptr(), t_stride,
                    KVQ_BF16 if out_dtype == "bf16" else KVQ_FP32, self._stream())
        return k_out, v_out

    def dense_decode_attention(self, k, v, q, out=None):
        """Standard decode attention over dense restored k, v [batch, n_kv_heads,
        t_stride, head_dim] (bf16), lengths from this cache."""
        shape = (self.cfg.batch, self.cfg.n_q_heads, self.cfg.head_dim)
        self._check_input(q, shape)
        assert k.shape == v.shape and k.dim() == 4 and k.shape[:2] == (self.cfg.batch, self.cfg.n_kv_heads)
        assert k.dtype == self.dtype and v.dtype == self.dtype and k.is_contiguous() and v.is_contiguous()
        if out is None:
            out = self.torch.empty(shape, dtype=self.torch.float32, device=self.device)
        kvq_dense_decode_attention(self.handle, k.data_ptr(), v.data_ptr(), k.shape[2], q.data_ptr(), out.data_ptr(),
                                   self._stream())
        return out

    def decode_step(self, new_k, new_v, q, out=None, kernel=0, split_start=None, split_stop=None):
        """Append one token per sequence (new_k, new_v: [batch, n_kv_heads, 1,
        head_dim]) and attend with q [batch, n_q_heads, head_dim]."""
        shape = (self.cfg.batch, self.cfg.n_kv_heads, 1, self.cfg.head_dim)
        self._check_input(new_k, shape)
        self._check_input(new_v, shape)
        qshape = (self.cfg.batch, self.cfg.n_q_heads, self.cfg.head_dim)
        self._check_input(q, qshape)
        if out is None:
            out = self.torch.empty(qshape, dtype=self.torch.float32, device=self.device)
        kvq_decode_step(self.handle, new_k.data_ptr(), new_v.data_ptr(), q.data_ptr(), out.data_ptr(), self._stream(),
                        kernel, split_start, split_stop)
        return out

    def bytes(self):
        return kvq_bytes(self.handle)

    def release(self, seq_begin=0, n_seqs=1):
        kvq_release(self.handle, seq_begin, n_seqs)

    def pool_state(self):
        """(free blocks, pool blocks) of a paged cache."""
        return kvq_pool_state(self.handle)

    def seq_state(self, seq):
        return kvq_seq_state(self.handle, seq)

    def export_unit(self, seq, kv_head):
        """Host numpy copies of one unit: dict of k_codes, v_codes, k_scales,
        v_scales, window_k, window_v (token order)."""
        import numpy as np
        st = self.seq_state(seq)
        Q, W, D = st["quantized"], st["window"], self.cfg.head_dim
        arrs = {"k_codes": np.zeros((Q, D), np.int8), "v_codes": np.zeros((Q, D), np.int8),
                "k_scales": np.zeros((st["n_groups"], D), np.float32), "v_scales": np.zeros((Q,), np.float32),
                "window_k": np.zeros((W, D), np.float32), "window_v": np.zeros((W, D), np.float32)}
        view = kvq_unit_view(*[a.ctypes.data for a in arrs.values()])
        kvq_export_unit(self.handle, seq, kv_head, view, self._stream())
        return arrs

    def export_pages(self, seq, kv_head):
        import numpy as np
        st = self.seq_state(seq)
        n = (st["quantized"] // self.cfg.group) * kvq_page_bytes(self.cfg)
        buf = np.zeros(max(n, 1), np.uint8)
        kvq_export_pages(self.handle, seq, kv_head, buf.ctypes.data, buf.nbytes, self._stream())
        return buf[:n].tobytes()

    def device_status(self):
        return kvq_device_status(self.handle, self._stream())

    def close(self):
        if getattr(self, "handle", None):
            kvq_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
