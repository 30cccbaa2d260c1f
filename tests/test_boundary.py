"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects bad configurations on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def kvq():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    from bit_asymmetric_kv_kvq_gb300 import _build
    try:
        _build.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    return kvq


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ["kvq_create", "kvq_prefill_quantize", "kvq_append", "kvq_decode_attention", "kvq_destroy"]:
        assert n in names


def test_library_exports_every_declared_symbol(kvq):
    L = ctypes.CDLL(kvq.kvq.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    # and the binding knows the signature of each one
    assert set(declared_functions()) <= set(kvq.kvq.SIGNATURES)


def test_status_strings(kvq):
    for s in range(-6, 1):
        assert kvq.status_string(s) and kvq.status_string(s) != "unknown status"
    assert kvq.status_string(-99) == "unknown status"
    assert kvq.lib().kvq_version() >> 16 == 1


def _status(kvq, **over):
    cfg = kvq.make_config(2, 4, 8, 128, 4096, 2, 2, 32, 128)
    for k, v in over.items():
        setattr(cfg, k, v)
    h = ctypes.c_void_p(123)
    st = kvq.lib().kvq_create(ctypes.byref(cfg), 0, ctypes.byref(h))
    assert h.value is None  # *out is cleared on failure
    return st


@pytest.mark.parametrize("field,value,expect", [
    ("batch", 0, -1), ("num_kv_heads", 0, -1), ("num_q_heads", 6, -1), ("head_dim", 0, -1), ("max_tokens", 0, -1),
    ("k_bits", 1, -1), ("k_bits", 5, -1), ("v_bits", 8, -1), ("group_size", 48, -1), ("residual", 100, -1),
    ("k_sparse", -1, -1), ("rope", 2, -1), ("softmax_scale", 0.0, -1), ("softmax_scale", float("inf"), -1),
    ("head_dim", 64, -2), ("group_size", 16, -2), ("residual", 256, -2), ("k_sparse", 5, -2),
    ("num_q_heads", 32, -2),  # 8 query heads per kv head: not in this build
    ("sink_tokens", -1, -1), ("sink_tokens", 129, -2),  # more sink tokens than R: not in this build
])
def test_bad_configs_are_rejected_on_the_host(kvq, field, value, expect):
    assert _status(kvq, **{field: value}) == expect


def test_null_arguments(kvq):
    L = kvq.lib()
    assert L.kvq_destroy(None) == 0
    assert L.kvq_create(None, 0, ctypes.byref(ctypes.c_void_p())) == -1
    cfg = kvq.make_config(1, 1, 1, 128, 16, 2, 2, 32, 128)
    assert L.kvq_create(ctypes.byref(cfg), 0, None) == -1
    assert L.kvq_prefill_quantize(None, None, None, 1, None) == -1
    assert L.kvq_append(None, None, None, None) == -1
    assert L.kvq_decode_attention(None, None, None, None) == -1
    assert L.kvq_get_state(None, None, None, None) == -1
    assert L.kvq_set_splits(None, 0) == -1
    assert L.kvq_sync_status(None, None) == -1
    assert L.kvq_launch_count(None) == -1
    assert L.kvq_reset(None) == -1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import bit_asymmetric_kv_kvq_gb300.kvq as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        b.lib()


def test_axis_calls_check_arguments_on_the_host(kvq):
    L = kvq.lib()
    p = 256  # any 16-byte aligned non-null address: the checks run before any launch
    assert L.kvq_axis_quantize(None, 1, 64, 128, 2, 32, 0, p, p, p, None) == -1
    assert L.kvq_axis_quantize(p, 1, 64, 128, 5, 32, 0, p, p, p, None) == -1   # bits
    assert L.kvq_axis_quantize(p, 1, 64, 128, 2, 32, 2, p, p, p, None) == -1   # axis
    assert L.kvq_axis_quantize(p, 1, 65, 128, 2, 32, 0, p, p, p, None) == -1   # tokens not a multiple of G
    assert L.kvq_axis_quantize(p, 1, 64, 64, 2, 32, 0, p, p, p, None) == -2    # head_dim
    assert L.kvq_axis_quantize(p, 1, 64, 128, 2, 16, 1, p, p, p, None) == -2   # group
    assert L.kvq_axis_dequantize(p, p, p, 0, 64, 128, 32, 0, p, None) == -1
    assert L.kvq_axis_attention(p, p, 1, p, 1, 3, 64, 128, 0.1, None, p, None) == -2  # heads per unit
    assert L.kvq_axis_attention(p, p, 1, p, 1, 1, 64, 128, 0.0, None, p, None) == -1  # scale


def _r16(x):
    return (x + 15) // 16 * 16


@pytest.mark.parametrize("bk,bv,G,R,nsp,rope,cb", [
    (2, 2, 32, 128, 0, 0, 0), (4, 2, 32, 128, 0, 0, 0), (4, 4, 64, 128, 0, 0, 0), (3, 3, 64, 128, 2, 1, 0),
    (2, 2, 32, 64, 1, 0, 0), (3, 3, 32, 96, 3, 0, 0), (2, 2, 32, 128, 0, 1, 0), (4, 4, 32, 128, 0, 0, 1),
])
def test_page_layout_on_the_host(kvq, bk, bv, G, R, nsp, rope, cb):
    """kvq_page_layout: the sections the header lists, in order, each padded to 16 bytes; fragment
    order exactly for 2/4-bit codes with keys stored after RoPE and uniform levels."""
    hg = 4 if (rope or cb) and (bk, bv) == (3, 3) else 1
    cfg = kvq.make_config(2, 2, 2 * hg, 128, 4096, bk, bv, G, R, k_sparse=nsp, rope=rope, codebook=cb)
    lay = kvq.kvq.kvq_page_layout(cfg)
    D = 128
    sizes = [R * D * bk // 8, (R // G) * D * 4, R * D * bv // 8, R * (D // G) * 4, R * nsp, R * nsp * 2]
    offs = [lay[k] for k in ("kcodes_offset", "kmeta_offset", "vcodes_offset", "vmeta_offset", "sp_idx_offset",
                             "sp_val_offset")] + [lay["page_bytes"]]
    assert offs[0] == 0
    for i, n in enumerate(sizes):
        assert offs[i + 1] - offs[i] == _r16(n), (i, offs, sizes)
    assert lay["tokens_per_page"] == R
    assert lay["fragment_order"] == int(bk in (2, 4) and bv in (2, 4) and not rope and not cb)


def test_page_layout_errors(kvq):
    L = kvq.lib()
    cfg = kvq.make_config(1, 1, 1, 128, 16, 2, 2, 32, 128)
    info = kvq.kvq.kvq_page_info()
    assert L.kvq_page_layout(None, ctypes.byref(info)) == -1
    assert L.kvq_page_layout(ctypes.byref(cfg), None) == -1
    cfg.k_bits = 5
    assert L.kvq_page_layout(ctypes.byref(cfg), ctypes.byref(info)) == -1
    cfg.k_bits, cfg.head_dim = 2, 64
    assert L.kvq_page_layout(ctypes.byref(cfg), ctypes.byref(info)) == -2
