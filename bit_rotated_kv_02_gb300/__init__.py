"""Python binding of liboscar.so — the GB300 (sm_103a) OSCAR INT2 KV-cache hot path.

The functions below carry the C ABI's names (include/oscar.h) and only marshal arguments: torch
tensors provide device memory and streams, every computation runs in the library's CUDA kernels.
If liboscar.so has not been built the first call raises; there is no fallback implementation.

Three-segment pool "BF16 sink (64 tokens) | INT2 history | BF16 recent (256 tokens)", rotation
R = U · Hadamard · bit-reversal, 4 two-bit codes per byte ("超越TurboQuant！OSCAR：面向真实服务的2-bit
KV Cache量化", section "OSCAR 的设计").
"""
from __future__ import annotations

import ctypes as C
import math

import torch

from . import _lib
from ._lib import OscarError

HEAD_DIM, PAGE, SINK, RECENT = 128, 64, 64, 256
ROT_HAAR, ROT_COVARIANCE = 0, 1
DEVERR_PAGE_INDEX, DEVERR_HISTORY_FULL, DEVERR_COUNTERS, DEVERR_TIMEOUT, DEVERR_DEBUG_CHECK = 1, 2, 4, 8, 16

__all__ = ["OscarError", "Pool", "oscar_version", "oscar_make_rotation", "oscar_calib_covariance_k",
           "oscar_calib_covariance_v", "oscar_quantize_kv", "oscar_quantize_kv_codebook", "oscar_lloyd_max_codebook", "oscar_prefill_pool", "oscar_prefill_pool_shared", "oscar_demote", "oscar_append_kv",
           "oscar_decode_workspace_size", "oscar_decode_attention", "oscar_profile_events",
           "oscar_decode_attention_noalloc", "NOALLOC_SCRATCH_BYTES", "lib", "BF16Cache", "oscar_bf16_prefill",
           "oscar_bf16_append_kv", "oscar_bf16_decode_workspace_size", "oscar_bf16_decode_attention",
           "oscar_bf16_decode_step"]
NOALLOC_SCRATCH_BYTES = 8 << 20
PROFILE_HISTORY, PROFILE_DEMOTE = 0, 1


def lib() -> C.CDLL:
    return _lib.load()


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _s(stream):
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t, dtype, name, host_ok=False):
    """Check a tensor argument: a contiguous CUDA tensor of `dtype` (or, where host_ok, a page-locked host
    tensor, which the kernels read or write in place over the host link)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (host_ok and t.is_pinned())):
        raise TypeError(f"{name} must be a CUDA tensor" + (" or a pinned host tensor" if host_ok else ""))
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def oscar_version() -> str:
    return lib().oscar_version().decode()


def oscar_make_rotation(M: torch.Tensor, mode: int, stream=None):
    """R = U·H·P from a d x d fp64 device matrix M (Gaussian draws for ROT_HAAR, covariance for
    ROT_COVARIANCE).  Returns (R64 fp64, R32 fp32).  Synchronous."""
    _dev(M, torch.float64, "M")
    d = M.shape[0]
    R64 = torch.empty((d, d), dtype=torch.float64, device=M.device)
    R32 = torch.empty((d, d), dtype=torch.float32, device=M.device)
    ws = torch.empty(lib().oscar_make_rotation_workspace_size(d), dtype=torch.uint8, device=M.device)
    _lib.check(lib().oscar_make_rotation(d, mode, _p(M), _p(R64), _p(R32), _p(ws), ws.numel(), _s(stream)),
               "oscar_make_rotation")
    return R64, R32


def oscar_calib_covariance_k(Q: torch.Tensor, stream=None) -> torch.Tensor:
    """C = sum_h Q_h^T Q_h for bf16 Q [T][heads][d]; fp64 [d][d]."""
    _dev(Q, torch.bfloat16, "Q")
    T, H, d = Q.shape
    C_ = torch.empty((d, d), dtype=torch.float64, device=Q.device)
    _lib.check(lib().oscar_calib_covariance_k(T, H, d, _p(Q), _p(C_), _s(stream)), "oscar_calib_covariance_k")
    return C_


def oscar_calib_covariance_v(Q, K, V, softmax_scale=None, stream=None) -> torch.Tensor:
    """C = sum_h (S_h V)^T (S_h V), S_h = causal softmax(Q_h K^T * scale); Q [T][heads][d], K, V [T][d] bf16."""
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _dev(t, torch.bfloat16, n)
    T, H, d = Q.shape
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    C_ = torch.empty((d, d), dtype=torch.float64, device=Q.device)
    ws = torch.empty(lib().oscar_calib_covariance_v_workspace_size(T, H, d), dtype=torch.uint8, device=Q.device)
    _lib.check(lib().oscar_calib_covariance_v(T, H, d, _p(Q), _p(K), _p(V), scale, _p(C_), _p(ws), ws.numel(),
                                              _s(stream)), "oscar_calib_covariance_v")
    return C_


def oscar_quantize_kv(x, R32, clip, group_size, codes=None, scale=None, zero=None, stats=None, stream=None):
    """Bulk rotate/clip/quantize/pack: x bf16 [N][Hkv][128] -> (codes u8 [N][Hkv][32], scale, zero bf16 [N][Hkv][ng])."""
    _dev(x, torch.bfloat16, "x")
    _dev(R32, torch.float32, "R32")
    _dev(clip, torch.float32, "clip")
    N, Hkv, d = x.shape
    ng = d // group_size
    codes = torch.empty((N, Hkv, d // 4), dtype=torch.uint8, device=x.device) if codes is None else codes
    scale = torch.empty((N, Hkv, ng), dtype=torch.bfloat16, device=x.device) if scale is None else scale
    zero = torch.empty((N, Hkv, ng), dtype=torch.bfloat16, device=x.device) if zero is None else zero
    _lib.check(lib().oscar_quantize_kv(N, Hkv, d, group_size, _p(x), _p(R32), _p(clip), _p(codes), _p(scale),
                                       _p(zero), _p(stats), _s(stream)), "oscar_quantize_kv")
    return codes, scale, zero


def oscar_quantize_kv_codebook(x, R32, clip, codebook, group_size=HEAD_DIM, codes=None, scale=None, zero=None,
                               stats=None, stream=None):
    """oscar_quantize_kv with the four levels codebook fp32 [Hkv][4] in place of the uniform 0, 1, 2, 3."""
    _dev(x, torch.bfloat16, "x")
    _dev(R32, torch.float32, "R32")
    _dev(clip, torch.float32, "clip")
    _dev(codebook, torch.float32, "codebook")
    N, Hkv, d = x.shape
    ng = d // group_size
    codes = torch.empty((N, Hkv, d // 4), dtype=torch.uint8, device=x.device) if codes is None else codes
    scale = torch.empty((N, Hkv, ng), dtype=torch.bfloat16, device=x.device) if scale is None else scale
    zero = torch.empty((N, Hkv, ng), dtype=torch.bfloat16, device=x.device) if zero is None else zero
    _lib.check(lib().oscar_quantize_kv_codebook(N, Hkv, d, group_size, _p(x), _p(R32), _p(clip), _p(codebook),
                                                _p(codes), _p(scale), _p(zero), _p(stats), _s(stream)),
               "oscar_quantize_kv_codebook")
    return codes, scale, zero


def oscar_lloyd_max_codebook(x, R32, clip, group_size=HEAD_DIM, max_iters=200, codebook=None, ws=None, stream=None):
    """Lloyd-Max levels fp32 [Hkv][4] per KV head from the calibration rows x bf16 [n][Hkv][128]."""
    _dev(x, torch.bfloat16, "x")
    _dev(R32, torch.float32, "R32")
    _dev(clip, torch.float32, "clip")
    N, Hkv, d = x.shape
    codebook = torch.empty((Hkv, 4), dtype=torch.float32, device=x.device) if codebook is None else codebook
    n = C.c_size_t(0)
    _lib.check(lib().oscar_lloyd_max_workspace_size(N, Hkv, C.byref(n)), "oscar_lloyd_max_workspace_size")
    if ws is None:
        ws = torch.empty(max(n.value, 16), dtype=torch.uint8, device=x.device)
    _lib.check(lib().oscar_lloyd_max_codebook(N, Hkv, d, group_size, _p(x), _p(R32), _p(clip), max_iters,
                                              _p(codebook), _p(ws), ws.numel(), _s(stream)),
               "oscar_lloyd_max_codebook")
    return codebook


class Pool:
    """Device storage of one layer's three-segment pool plus its C struct (see include/oscar.h).
    codebook_k, codebook_v: optional fp32 [Hkv][4] Lloyd-Max levels (None: the uniform INT2 levels)."""

    def __init__(self, batch, num_q_heads, num_kv_heads, group_size, num_pages, max_pages, R_k, R_v, clip_k, clip_v,
                 device="cuda", head_dim=HEAD_DIM, codebook_k=None, codebook_v=None):
        dev = torch.device(device)
        self.device = dev
        self.B, self.Hq, self.Hkv, self.d, self.g = batch, num_q_heads, num_kv_heads, head_dim, group_size
        self.ng = head_dim // group_size
        self.num_pages, self.max_pages = num_pages, max_pages
        bf = torch.bfloat16
        z = lambda *shape, dt: torch.zeros(shape, dtype=dt, device=dev)
        self.sink_k, self.sink_v = z(batch, num_kv_heads, SINK, head_dim, dt=bf), z(batch, num_kv_heads, SINK, head_dim, dt=bf)
        self.recent_k = z(batch, num_kv_heads, RECENT, head_dim, dt=bf)
        self.recent_v = z(batch, num_kv_heads, RECENT, head_dim, dt=bf)
        self.codes_k = z(num_pages, num_kv_heads, PAGE, head_dim // 4, dt=torch.uint8)
        self.codes_v = z(num_pages, num_kv_heads, PAGE, head_dim // 4, dt=torch.uint8)
        self.scale_k, self.zero_k = z(num_pages, num_kv_heads, PAGE, self.ng, dt=bf), z(num_pages, num_kv_heads, PAGE, self.ng, dt=bf)
        self.scale_v, self.zero_v = z(num_pages, num_kv_heads, PAGE, self.ng, dt=bf), z(num_pages, num_kv_heads, PAGE, self.ng, dt=bf)
        self.page_table = torch.full((batch, max(max_pages, 1)), -1, dtype=torch.int32, device=dev)
        self.sink_len, self.hist_len = z(batch, dt=torch.int32), z(batch, dt=torch.int32)
        self.recent_start, self.recent_len = z(batch, dt=torch.int32), z(batch, dt=torch.int32)
        self.R_k = _dev(R_k.to(dev, torch.float32).contiguous(), torch.float32, "R_k")
        self.R_v = _dev(R_v.to(dev, torch.float32).contiguous(), torch.float32, "R_v")
        self.clip_k = clip_k.to(dev, torch.float32).contiguous()
        self.clip_v = clip_v.to(dev, torch.float32).contiguous()
        self.err_word = z(1, dt=torch.int32)
        self.sync = z(batch, dt=torch.int32)
        cbk = lambda cb: None if cb is None else torch.as_tensor(cb, dtype=torch.float32).to(dev).reshape(
            num_kv_heads, 4).contiguous()
        self.codebook_k, self.codebook_v = cbk(codebook_k), cbk(codebook_v)
        self.struct = _lib.oscar_pool(
            batch, num_q_heads, num_kv_heads, head_dim, group_size, num_pages, max_pages,
            *(t.data_ptr() for t in (self.sink_k, self.sink_v, self.recent_k, self.recent_v, self.codes_k,
                                     self.codes_v, self.scale_k, self.zero_k, self.scale_v, self.zero_v,
                                     self.page_table, self.sink_len, self.hist_len, self.recent_start,
                                     self.recent_len, self.R_k, self.R_v, self.clip_k, self.clip_v, self.err_word,
                                     self.sync)),
            *(None if t is None else t.data_ptr() for t in (self.codebook_k, self.codebook_v)))

    @property
    def ref(self):
        return C.byref(self.struct)

    def set_page_table(self, pt):
        self.page_table.copy_(torch.as_tensor(pt, dtype=torch.int32).reshape(self.page_table.shape))

    def err(self) -> int:
        return int(self.err_word.item()) & 0xffffffff

    def counters(self):
        return {k: getattr(self, k).cpu().numpy().copy() for k in ("sink_len", "hist_len", "recent_start", "recent_len")}


def oscar_prefill_pool(pool: Pool, seq: int, k, v, stats=None, stream=None):
    _dev(k, torch.bfloat16, "k")
    _dev(v, torch.bfloat16, "v")
    _lib.check(lib().oscar_prefill_pool(pool.ref, seq, k.shape[0], _p(k), _p(v), _p(stats), _s(stream)),
               "oscar_prefill_pool")


def oscar_prefill_pool_shared(pool: Pool, seq: int, k, v, shared_pages: int, stats=None, stream=None):
    """Prefill whose first `shared_pages` history pages are already in the pool (shared prefix pages that
    the sequence's page table points at); they are not written."""
    _dev(k, torch.bfloat16, "k")
    _dev(v, torch.bfloat16, "v")
    _lib.check(lib().oscar_prefill_pool_shared(pool.ref, seq, k.shape[0], _p(k), _p(v), shared_pages, _p(stats),
                                               _s(stream)), "oscar_prefill_pool_shared")


def oscar_demote(pool: Pool, mask=None, stream=None):
    if mask is not None:
        _dev(mask, torch.int32, "mask")
    _lib.check(lib().oscar_demote(pool.ref, _p(mask), _s(stream)), "oscar_demote")


def oscar_append_kv(pool: Pool, k_new, v_new, stream=None):
    _dev(k_new, torch.bfloat16, "k_new")
    _dev(v_new, torch.bfloat16, "v_new")
    _lib.check(lib().oscar_append_kv(pool.ref, _p(k_new), _p(v_new), _s(stream)), "oscar_append_kv")


def oscar_decode_workspace_size(pool: Pool, num_splits: int = 0) -> int:
    n = C.c_size_t(0)
    _lib.check(lib().oscar_decode_workspace_size(pool.ref, num_splits, C.byref(n)), "oscar_decode_workspace_size")
    return n.value


def oscar_decode_attention(pool: Pool, q, out=None, softmax_scale=None, num_splits=0, ws=None, stream=None):
    """fp32 out [B][Hq][128] of bf16 q [B][Hq][128] over the pool."""
    _dev(q, torch.bfloat16, "q")
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out is None else out
    if ws is None:
        ws = torch.empty(oscar_decode_workspace_size(pool, num_splits), dtype=torch.uint8, device=q.device)
    scale = 1.0 / math.sqrt(pool.d) if softmax_scale is None else float(softmax_scale)
    _lib.check(lib().oscar_decode_attention(pool.ref, _p(q), _p(out), scale, num_splits, _p(ws), ws.numel(),
                                            _s(stream)), "oscar_decode_attention")
    return out


def oscar_decode_step(pool: Pool, k_new, v_new, q, out=None, softmax_scale=None, ws=None, stream=None):
    """One decode step (append k_new/v_new bf16 [B][Hkv][128], demote, attention of q bf16 [B][Hq][128]):
    what oscar_append_kv then oscar_decode_attention give, in fewer launches.  Returns fp32 out."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (q, "q")):
        _dev(t, torch.bfloat16, n, host_ok=True)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device, pin_memory=not q.is_cuda) if out is None else out
    _dev(out, torch.float32, "out", host_ok=True)
    if ws is None:
        ws = torch.empty(oscar_decode_workspace_size(pool, 0), dtype=torch.uint8, device=pool.device)
    scale = 1.0 / math.sqrt(pool.d) if softmax_scale is None else float(softmax_scale)
    _lib.check(lib().oscar_decode_step(pool.ref, _p(k_new), _p(v_new), _p(q), _p(out), scale, _p(ws), ws.numel(),
                                       _s(stream)), "oscar_decode_step")
    return out


def oscar_profile_events(which: int, start=None, stop=None):
    """Arm the timing hook: the next launch of kernel kind `which` on this thread records torch.cuda.Event
    `start` before and `stop` after that kernel (on the call's stream)."""
    sp = None if start is None else C.c_void_p(start.cuda_event)
    ep = None if stop is None else C.c_void_p(stop.cuda_event)
    _lib.check(lib().oscar_profile_events(which, sp, ep), "oscar_profile_events")


def oscar_decode_attention_noalloc(pool: Pool, q, out, softmax_scale=None, stream=None):
    """Decode attention with the library's fixed device scratch (no allocation by the library or here):
    q bf16 [B][Hq][128], out fp32 [B][Hq][128] caller-provided."""
    _dev(q, torch.bfloat16, "q")
    _dev(out, torch.float32, "out")
    scale = 1.0 / math.sqrt(pool.d) if softmax_scale is None else float(softmax_scale)
    _lib.check(lib().oscar_decode_attention_noalloc(pool.ref, _p(q), _p(out), scale, _s(stream)),
               "oscar_decode_attention_noalloc")
    return out


# ---- BF16 paged cache: the baseline INT2 decoding is compared against ----------------------------------
class BF16Cache:
    """Device storage of a BF16 paged KV cache plus its C struct (see include/oscar.h)."""

    def __init__(self, batch, num_q_heads, num_kv_heads, num_pages, max_pages, device="cuda", head_dim=HEAD_DIM):
        dev = torch.device(device)
        self.B, self.Hq, self.Hkv, self.d = batch, num_q_heads, num_kv_heads, head_dim
        self.num_pages, self.max_pages = num_pages, max_pages
        self.k_pages = torch.zeros((num_pages, num_kv_heads, PAGE, head_dim), dtype=torch.bfloat16, device=dev)
        self.v_pages = torch.zeros_like(self.k_pages)
        self.page_table = torch.full((batch, max_pages), -1, dtype=torch.int32, device=dev)
        self.seq_len = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.err_word = torch.zeros(1, dtype=torch.int32, device=dev)
        self.struct = _lib.oscar_bf16_cache(
            batch, num_q_heads, num_kv_heads, head_dim, num_pages, max_pages,
            *(t.data_ptr() for t in (self.k_pages, self.v_pages, self.page_table, self.seq_len, self.err_word)))

    @property
    def ref(self):
        return C.byref(self.struct)

    def set_page_table(self, pt):
        self.page_table.copy_(torch.as_tensor(pt, dtype=torch.int32).reshape(self.page_table.shape))

    def err(self) -> int:
        return int(self.err_word.item()) & 0xffffffff


def oscar_bf16_prefill(cache: BF16Cache, seq: int, k, v, stream=None):
    """Tokens [0, len) of sequence `seq` from bf16 k, v [len][Hkv][128]."""
    _dev(k, torch.bfloat16, "k")
    _dev(v, torch.bfloat16, "v")
    _lib.check(lib().oscar_bf16_prefill(cache.ref, seq, k.shape[0], _p(k), _p(v), _s(stream)), "oscar_bf16_prefill")


def oscar_bf16_append_kv(cache: BF16Cache, k_new, v_new, stream=None):
    _dev(k_new, torch.bfloat16, "k_new")
    _dev(v_new, torch.bfloat16, "v_new")
    _lib.check(lib().oscar_bf16_append_kv(cache.ref, _p(k_new), _p(v_new), _s(stream)), "oscar_bf16_append_kv")


def oscar_bf16_decode_workspace_size(cache: BF16Cache) -> int:
    n = C.c_size_t(0)
    _lib.check(lib().oscar_bf16_decode_workspace_size(cache.ref, C.byref(n)), "oscar_bf16_decode_workspace_size")
    return n.value


def oscar_bf16_decode_attention(cache: BF16Cache, q, out=None, softmax_scale=None, ws=None, stream=None):
    """fp32 out [B][Hq][128] of bf16 q [B][Hq][128] over the BF16 cache."""
    _dev(q, torch.bfloat16, "q")
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out is None else out
    if ws is None:
        ws = torch.empty(oscar_bf16_decode_workspace_size(cache), dtype=torch.uint8, device=q.device)
    scale = 1.0 / math.sqrt(cache.d) if softmax_scale is None else float(softmax_scale)
    _lib.check(lib().oscar_bf16_decode_attention(cache.ref, _p(q), _p(out), scale, _p(ws), ws.numel(), _s(stream)),
               "oscar_bf16_decode_attention")
    return out


def oscar_bf16_decode_step(cache: BF16Cache, k_new, v_new, q, out=None, softmax_scale=None, ws=None, stream=None):
    """Append k_new/v_new bf16 [B][Hkv][128], then attention of q bf16 [B][Hq][128]; returns fp32 out."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (q, "q")):
        _dev(t, torch.bfloat16, n)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out is None else out
    if ws is None:
        ws = torch.empty(oscar_bf16_decode_workspace_size(cache), dtype=torch.uint8, device=q.device)
    scale = 1.0 / math.sqrt(cache.d) if softmax_scale is None else float(softmax_scale)
    _lib.check(lib().oscar_bf16_decode_step(cache.ref, _p(k_new), _p(v_new), _p(q), _p(out), scale, _p(ws),
                                            ws.numel(), _s(stream)), "oscar_bf16_decode_step")
    return out
