"""C-ABI checks that need no GPU: the library loads, exports every function include/oscar.h declares,
and rejects invalid arguments on the host (status codes) before any launch."""
import ctypes as C

import pytest

import __graft_entry__
from bit_rotated_kv_02_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), f"{n} declared in oscar.h but not exported"
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_version_and_error_string(lib):
    assert b"sm_103a" in lib.oscar_version()
    assert lib.oscar_last_error_string() is not None


FAKE = C.c_void_p(0x10000)  # never dereferenced: validation fails first


def _pool(**kw):
    p = _lib.oscar_pool()
    p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.group_size = 1, 8, 2, 128, 128
    p.num_pages, p.max_pages = 4, 4
    for name, _ in _lib.oscar_pool._fields_[7:]:
        setattr(p, name, 0x10000)
    p.codebook_k = p.codebook_v = None  # the uniform levels unless a test sets a codebook
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2), (dict(group_size=48), 2), (dict(num_q_heads=7), 1), (dict(num_q_heads=32, num_kv_heads=2), 2),
    (dict(batch=0), 1), (dict(codes_k=None), 1), (dict(err=None), 1), (dict(R_k=0x10004), 1),
])
def test_pool_validation(lib, kw, status):
    p = _pool(**kw)
    assert lib.oscar_demote(C.byref(p), None, None) == status
    assert lib.oscar_last_error_string()


def test_decode_rejects_missing_workspace(lib):
    p = _pool()
    n = C.c_size_t(0)
    assert lib.oscar_decode_workspace_size(C.byref(p), 4, C.byref(n)) == 0 and n.value > 0
    assert lib.oscar_decode_attention(C.byref(p), FAKE, FAKE, 0.088, 4, None, 0, None) == 3
    assert lib.oscar_decode_attention(C.byref(p), FAKE, FAKE, 0.088, 4, FAKE, 4096, None) == 3
    assert lib.oscar_decode_attention(C.byref(p), FAKE, FAKE, -1.0, 4, FAKE, n.value, None) == 1
    assert lib.oscar_decode_attention(C.byref(p), None, FAKE, 0.088, 4, FAKE, n.value, None) == 1
    # q and out must be memory the kernels can reach: a bad pointer is refused on the host
    assert lib.oscar_decode_attention(C.byref(p), FAKE, FAKE, 0.088, 4, FAKE, n.value, None) == 1
    assert b"page-locked" in lib.oscar_last_error_string()


def test_quantize_validation(lib):
    args = (FAKE,) * 3 + (FAKE,) * 3
    assert lib.oscar_quantize_kv(16, 2, 64, 32, *args, None, None) == 2
    assert lib.oscar_quantize_kv(16, 2, 128, 16, *args, None, None) == 2
    assert lib.oscar_quantize_kv(-1, 2, 128, 32, *args, None, None) == 1
    assert lib.oscar_quantize_kv(0, 2, 128, 32, *args, None, None) == 0   # empty input is a no-op
    assert lib.oscar_quantize_kv(16, 2, 128, 32, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 1


def test_prefill_and_rotation_validation(lib):
    p = _pool()
    assert lib.oscar_prefill_pool(C.byref(p), 1, 100, FAKE, FAKE, None, None) == 1          # seq out of range
    assert lib.oscar_prefill_pool(C.byref(p), 0, 320 + 4 * 64 + 1, FAKE, FAKE, None, None) == 1  # too long
    assert lib.oscar_make_rotation(96, 0, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 2
    assert lib.oscar_make_rotation(128, 7, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == 1
    assert lib.oscar_make_rotation(128, 0, FAKE, FAKE, FAKE, FAKE, 16, None) == 3
    assert lib.oscar_make_rotation_workspace_size(128) >= 128 * 128 * 8
    assert lib.oscar_calib_covariance_v(100, 2, 128, FAKE, FAKE, FAKE, 0.0, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.oscar_append_kv(C.byref(p), None, FAKE, None) == 1


def _cache(**kw):
    c = _lib.oscar_bf16_cache()
    c.batch, c.num_q_heads, c.num_kv_heads, c.head_dim, c.num_pages, c.max_pages = 2, 8, 2, 128, 16, 8
    for name, _ in _lib.oscar_bf16_cache._fields_[6:]:
        setattr(c, name, 0x10000)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2), (dict(num_q_heads=7), 1), (dict(num_q_heads=32), 2), (dict(batch=0), 1),
    (dict(num_pages=0), 1), (dict(k_pages=None), 1), (dict(seq_len=None), 1), (dict(v_pages=0x10008), 1),
    (dict(num_pages=1 << 24), 1),
])
def test_bf16_cache_validation(lib, kw, status):
    c = _cache(**kw)
    assert lib.oscar_bf16_append_kv(C.byref(c), FAKE, FAKE, None) == status
    assert lib.oscar_last_error_string()


def test_bf16_cache_call_validation(lib):
    c = _cache()
    n = C.c_size_t(0)
    assert lib.oscar_bf16_decode_workspace_size(C.byref(c), C.byref(n)) == 0 and n.value > 0
    assert lib.oscar_bf16_decode_attention(C.byref(c), FAKE, FAKE, 0.088, None, 0, None) == 3
    assert lib.oscar_bf16_decode_attention(C.byref(c), FAKE, FAKE, 0.088, FAKE, n.value - 1, None) == 3
    assert lib.oscar_bf16_decode_attention(C.byref(c), FAKE, FAKE, 0.0, FAKE, n.value, None) == 1
    assert lib.oscar_bf16_decode_attention(C.byref(c), None, FAKE, 0.088, FAKE, n.value, None) == 1
    assert lib.oscar_bf16_decode_step(C.byref(c), None, FAKE, FAKE, FAKE, 0.088, FAKE, n.value, None) == 1
    assert lib.oscar_bf16_decode_step(C.byref(c), C.c_void_p(0x10008), FAKE, FAKE, FAKE, 0.088, FAKE, n.value,
                                      None) == 1
    assert lib.oscar_bf16_prefill(C.byref(c), 2, 10, FAKE, FAKE, None) == 1          # seq out of range
    assert lib.oscar_bf16_prefill(C.byref(c), 0, 8 * 64 + 1, FAKE, FAKE, None) == 1  # longer than max_pages*64
    assert lib.oscar_bf16_prefill(C.byref(c), 0, 10, None, FAKE, None) == 1


def test_codebook_validation(lib):
    """Codebook pools and the codebook calls reject bad arguments before any launch."""
    assert lib.oscar_demote(C.byref(_pool(codebook_k=0x10004)), None, None) == 1   # codebooks 16-byte aligned
    assert lib.oscar_demote(C.byref(_pool(codebook_v=0x10008)), None, None) == 1
    n = C.c_size_t(0)
    assert lib.oscar_decode_workspace_size(C.byref(_pool(codebook_k=0x10000, codebook_v=0x10000)), 0,
                                           C.byref(n)) == 0 and n.value > 0
    src, dst = (FAKE,) * 3, (FAKE,) * 3
    assert lib.oscar_quantize_kv_codebook(16, 2, 128, 128, *src, None, *dst, None, None) == 1
    assert lib.oscar_quantize_kv_codebook(16, 2, 128, 128, *src, C.c_void_p(0x10004), *dst, None, None) == 1
    assert lib.oscar_quantize_kv_codebook(16, 2, 128, 48, *src, FAKE, *dst, None, None) == 2
    assert lib.oscar_quantize_kv_codebook(16, 2, 64, 128, *src, FAKE, *dst, None, None) == 2
    assert lib.oscar_quantize_kv_codebook(0, 2, 128, 128, *src, FAKE, *dst, None, None) == 0  # empty: no-op
    # Lloyd-Max calibration: the workspace query, a missing workspace, bad sizes
    assert lib.oscar_lloyd_max_workspace_size(10, 2, C.byref(n)) == 0 and n.value == 10 * 2 * 128 * 4
    assert lib.oscar_lloyd_max_workspace_size(-1, 2, C.byref(n)) == 1
    assert lib.oscar_lloyd_max_workspace_size(10, 2, None) == 1
    assert lib.oscar_lloyd_max_codebook(10, 2, 128, 128, FAKE, FAKE, FAKE, 200, FAKE, FAKE, 16, None) == 3
    assert lib.oscar_lloyd_max_codebook(10, 2, 128, 128, FAKE, FAKE, FAKE, -1, FAKE, FAKE, 10240, None) == 1
    assert lib.oscar_lloyd_max_codebook(10, 2, 64, 128, FAKE, FAKE, FAKE, 200, FAKE, FAKE, 10240, None) == 2
    assert lib.oscar_lloyd_max_codebook(10, 2, 128, 128, FAKE, FAKE, FAKE, 200, None, FAKE, 10240, None) == 1


def test_debug_build_is_a_separate_library_with_the_checks_compiled_in():
    """The debug build compiles the same sources with OSCAR_DEBUG into liboscar_debug.so; the binding loads it
    only when the environment asks for it (OSCAR_DEBUG=1)."""
    from bit_rotated_kv_02_gb300 import build
    assert "-DOSCAR_DEBUG" in build.DEBUG_FLAGS
    assert build.LIB_DEBUG != build.LIB and build.LIB_DEBUG.endswith("liboscar_debug.so")
    src = open(build.os.path.join(build.CSRC, "oscar_internal.cuh")).read()
    assert "#ifdef OSCAR_DEBUG" in src and "OSCAR_DEVERR_DEBUG_CHECK" in src and "__trap" not in src
