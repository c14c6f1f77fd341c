"""Host-only checks of the C ABI: the library loads, exports every function
include/kvq.h declares, and its pure host functions (sizes, ledger,
validation) agree with the oracle's accounting.  No GPU needed."""

import ctypes
import os
import re

import pytest

from oracle import kvq_oracle as O
from oracle import layout as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")

kvq = pytest.importorskip("quantized_kv_cache_02_gb300")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kvq_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_function():
    lib = kvq.load_library()
    declared = _declared_functions()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(declared) == sorted(kvq.EXPORTED)


def test_page_bytes_matches_layout_definition():
    for G, D, qmax in ((32, 128, 7), (64, 128, 127), (128, 128, 7), (8, 16, 7), (32, 128, 1), (8, 16, 1)):
        cfg = kvq.make_config(1, 1, 1, D, 8, G, qmax)
        assert kvq.kvq_page_bytes(cfg) == L.page_bytes(G, D, O.code_bits(qmax))


@pytest.mark.parametrize("tokens", [[0], [40, 64, 7], [4096], [8192, 8320, 1, 159]])
@pytest.mark.parametrize("R,G,qmax,dtype", [(8, 8, 7, kvq.KVQ_FP32), (128, 32, 7, kvq.KVQ_BF16),
                                            (128, 64, 127, kvq.KVQ_BF16), (256, 128, 7, kvq.KVQ_BF16),
                                            (128, 32, 1, kvq.KVQ_BF16)])
def test_ledger_matches_oracle(tokens, R, G, qmax, dtype):
    cfg = kvq.make_config(len(tokens), 8, 32, 128, R, G, qmax, dtype)
    got = kvq.kvq_ledger(cfg, tokens)
    ref = O.held_ledger(tokens, n_kv_heads=8, head_dim=128, residual_length=R, group=G, qmax=qmax,
                        window_element_bytes=2 if dtype == kvq.KVQ_BF16 else 4)
    for k in ("code_bytes", "n_scales", "scale_bytes", "window_elems", "window_bytes", "total"):
        assert got[k] == ref[k], k


def test_ledger_explainer_window_case():
    """32 layers of an 8-head, d=128 cache holding 4096 tokens with R = G = 128:
    124 MiB of 4-bit codes plus a 16 MiB bf16 window (the explainer's 140 MiB)."""
    cfg = kvq.make_config(1, 8, 32, 128, 128, 128, 7, kvq.KVQ_BF16)
    led = kvq.kvq_ledger(cfg, [4096])
    assert 32 * led["code_bytes"] == 124 << 20
    assert 32 * led["window_bytes"] == 16 << 20


def test_required_bytes_grows_with_capacity():
    cfg = kvq.make_config(4, 8, 32, 128, 128, 32, 7)
    small = kvq.kvq_required_bytes(cfg, [1024] * 4)
    large = kvq.kvq_required_bytes(cfg, [8192] * 4)
    page = kvq.kvq_page_bytes(cfg)
    assert large - small >= 4 * 8 * (8192 - 1024) // 32 * page
    assert small % 256 == 0 and large % 256 == 0


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, kvq.binding.KVQ_EINVAL),
    ("n_q_heads", 12, kvq.binding.KVQ_EINVAL),
    ("n_q_heads", 8 * 16, kvq.binding.KVQ_EUNSUPPORTED),
    ("head_dim", 120, kvq.binding.KVQ_EUNSUPPORTED),
    ("residual_len", 0, kvq.binding.KVQ_EINVAL),
    ("group", 12, kvq.binding.KVQ_EUNSUPPORTED),
    ("qmax", 0, kvq.binding.KVQ_EINVAL),
    ("qmax", 128, kvq.binding.KVQ_EINVAL),
    ("dtype", 7, kvq.binding.KVQ_EINVAL),
    ("eps", 0.0, kvq.binding.KVQ_EINVAL),
])
def test_config_validation(field, value, status):
    cfg = kvq.make_config(2, 8, 32, 128, 128, 32, 7)
    setattr(cfg, field, value)
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_required_bytes(cfg, [64, 64])
    assert e.value.status == status


def test_capacity_validation_and_null_handles():
    cfg = kvq.make_config(2, 8, 32, 128, 128, 32, 7)
    with pytest.raises(kvq.KVQError):
        kvq.kvq_required_bytes(cfg, [64, 0])
    lib = kvq.load_library()
    assert lib.kvq_append(None, None, None, 1, 0, 1, None) == kvq.binding.KVQ_EINVAL
    assert b"NULL" in lib.kvq_last_error()
    assert lib.kvq_decode_attention(None, None, None, None) == kvq.binding.KVQ_EINVAL
    lib.kvq_destroy(None)
    # a host pointer is not an arena
    buf = ctypes.create_string_buffer(1 << 16)
    handle = ctypes.c_void_p()
    caps = (ctypes.c_int64 * 2)(64, 64)
    rc = lib.kvq_create(ctypes.byref(cfg), caps, ctypes.cast(buf, ctypes.c_void_p), 16, ctypes.byref(handle))
    assert rc != kvq.binding.KVQ_OK and handle.value is None


def test_restore_dense_and_compare_validate_before_any_launch():
    lib = kvq.load_library()
    assert lib.kvq_restore(None, 0, 1, None, None, 8, 0, None) == kvq.binding.KVQ_EINVAL
    assert lib.kvq_dense_decode_attention(None, None, None, 8, None, None, None) == kvq.binding.KVQ_EINVAL
    out = kvq.binding.kvq_compare_t()
    ws = ctypes.c_void_p(64)  # never dereferenced: every case below fails validation first
    good = dict(batch=1, heads=2, tokens=32, head_dim=16, dtype=0, qmax=7, eps=1e-8, group=0)

    def call(**kw):
        a = {**good, **kw}
        return lib.kvq_compare(ws, ws, a["batch"], a["heads"], a["tokens"], a["head_dim"], a["dtype"], a["qmax"],
                               a["eps"], a["group"], ws, ctypes.byref(out), None)

    for bad in [dict(batch=0), dict(tokens=0), dict(head_dim=0), dict(dtype=5), dict(qmax=0), dict(qmax=128),
                dict(eps=0.0), dict(group=-1), dict(group=5)]:
        assert call(**bad) == kvq.binding.KVQ_EINVAL, bad
    assert call(batch=70000) == kvq.binding.KVQ_EUNSUPPORTED
    assert lib.kvq_compare(None, ws, 1, 2, 32, 16, 0, 7, 1e-8, 0, ws, ctypes.byref(out), None) == kvq.binding.KVQ_EINVAL
    assert lib.kvq_compare(ws, ws, 1, 2, 32, 16, 0, 7, 1e-8, 0, ws, None, None) == kvq.binding.KVQ_EINVAL


def test_paged_sizes_and_validation():
    cfg = kvq.make_config(2, 8, 32, 128, 128, 32, 7)
    small = kvq.binding.kvq_required_bytes_paged(cfg, [4096, 4096], 10)
    big = kvq.binding.kvq_required_bytes_paged(cfg, [4096, 4096], 1000)
    # the pool grows by whole blocks: n_kv_heads group pages each
    assert big - small >= 990 * 8 * kvq.kvq_page_bytes(cfg) - 256
    with pytest.raises(kvq.KVQError) as e:
        kvq.binding.kvq_required_bytes_paged(cfg, [4096, 4096], 0)
    assert e.value.status == kvq.binding.KVQ_EINVAL
    lib = kvq.load_library()
    assert lib.kvq_release(None, 0, 1) == kvq.binding.KVQ_EINVAL
    free, total = ctypes.c_int64(), ctypes.c_int64()
    assert lib.kvq_pool_state(None, ctypes.byref(free), ctypes.byref(total)) == kvq.binding.KVQ_EINVAL
