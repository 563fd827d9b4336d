"""GPU check of the allocation-free decode entry point (oscar_decode_attention_noalloc).

Callers that cannot allocate device memory (an engine that reserved all of it up front, or a decode
loop that must not block on the allocator) use this entry point: its scratch is a fixed array inside
the library.  It must give what oscar_decode_attention gives with a caller-allocated workspace, on
consecutive calls that reuse the same array, and refuse pools whose scratch would not fit.
This file is collected last so that a run stopping at the first failure has run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import __graft_entry__
import bit_rotated_kv_02_gb300 as ok
import synth
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _pool(lens, Hq, Hkv, g, seed):
    pages = [max(0, -(-(L - 320) // 64)) for L in lens]
    _, P = helpers.make_pools(len(lens), Hq, Hkv, g, pages, seed)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for b, L in enumerate(lens):
        K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
        V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    return P, ch


@pytest.mark.parametrize("g", [128, 32])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(g):
    Hq, Hkv = 8, 2
    P, ch = _pool([1024, 3000], Hq, Hkv, g, 700 + g)
    lib = ok.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    scale = 1.0 / np.sqrt(128.0)
    for call in range(2):
        q = helpers.to_dev_bf16(synth.outlier_q(800 + call, 2, Hq, Hkv, 128, ch))
        ref = ok.oscar_decode_attention(P, q)
        out = torch.full_like(ref, float("nan"))
        st = lib.oscar_decode_attention_noalloc(P.ref, C.c_void_p(q.data_ptr()), C.c_void_p(out.data_ptr()),
                                                scale, stream)
        assert st == 0, lib.oscar_last_error_string().decode()
        torch.cuda.synchronize()
        helpers.assert_attention_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64))
    assert P.err() == 0


def test_noalloc_rejects_a_pool_whose_scratch_does_not_fit():
    B, Hq, Hkv = 64, 64, 8
    R = torch.from_numpy(np.stack([np.eye(128, dtype=np.float32)] * Hkv))
    clip = torch.full((Hkv,), 0.9)
    P = ok.Pool(B, Hq, Hkv, 128, 1, 1, R, R, clip, clip)
    assert ok.oscar_decode_workspace_size(P) > ok.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    lib = ok.lib()
    st = lib.oscar_decode_attention_noalloc(P.ref, C.c_void_p(q.data_ptr()), C.c_void_p(out.data_ptr()), 0.088,
                                            C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3
    assert b"static" in lib.oscar_last_error_string()
