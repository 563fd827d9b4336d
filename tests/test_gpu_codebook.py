"""GPU parity: the 4-level Lloyd-Max codebook in place of the uniform INT2 levels
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", closing comparison with TurboQuant).
Group 128 decodes on the tensor-core kernels (indicator planes), other group sizes on the CUDA-core
kernels (a 4-entry table); both are held to the oracle.

Codes, scales and zero points must equal the oracle's bit for bit (nearest level, ties to the even
code, with the uniform quantizer's bf16 scale and zero); the levels (0, 1, 2, 3) must reproduce the
uniform pool; decode attention over a codebook pool is held to the usual tolerance; the GPU's Lloyd-Max
calibration must land on the oracle's levels.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import bit_rotated_kv_02_gb300 as ok
import synth
from oracle import codebook as ocb
from oracle import rotation as orot
from tests import helpers

pytestmark = pytest.mark.gpu

# two hand-picked non-uniform codebooks (one per KV head) and the uniform levels
SKEWED = np.array([[0.2, 1.05, 1.95, 2.8], [-0.1, 0.9, 2.1, 3.2]], np.float32)


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _rows(seed, n, Hkv=2):
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    return synth.outlier_kv(seed + 1, n, Hkv, 128, ch), ch


@pytest.mark.parametrize("g", [128, 64, 32])
@pytest.mark.parametrize("n", [1, 37, 1000])
def test_quantize_kv_codebook_matches_oracle(g, n):
    Hkv = 2
    X, _ = _rows(1100 + n + g, n, Hkv)
    R = helpers.oracle_rotations(1101, Hkv)
    clip = np.array([0.9, 0.85], np.float32)
    codes, scale, zero = ok.oscar_quantize_kv_codebook(helpers.to_dev_bf16(X), torch.from_numpy(R).cuda(),
                                                       torch.from_numpy(clip).cuda(),
                                                       torch.from_numpy(SKEWED).cuda(), g)
    for h in range(Hkv):
        oc, os_, oz = ocb.quantize_vectors_cb(X[:, h], R[h], clip[h], g, SKEWED[h])
        assert np.array_equal(codes[:, h].cpu().numpy(), oc), h
        assert np.array_equal(helpers.bits_of(scale[:, h]), os_), h
        assert np.array_equal(helpers.bits_of(zero[:, h]), oz), h


@pytest.mark.parametrize("g", [128, 32])
def test_uniform_codebook_reproduces_the_uniform_pool(g):
    """The levels (0, 1, 2, 3) through the codebook kernels give the uniform pool's bytes and an attention
    output within the oracle's tolerance, like the uniform pool's."""
    Hkv, Hq, lens = 2, 8, [900, 1700]
    uni = np.stack([ocb.UNIFORM] * Hkv)
    pages = [-(-(L - 320) // 64) for L in lens]
    Ou, Pu = helpers.make_pools(len(lens), Hq, Hkv, g, pages, 1200, extra_pages=1)
    _, Pc = helpers.make_pools(len(lens), Hq, Hkv, g, pages, 1200, extra_pages=1, codebook_k=uni, codebook_v=uni)
    ch = synth.outlier_channels(1200, Hkv, 128, 4)
    for b, L in enumerate(lens):
        Kn, Vn = synth.outlier_kv(1210 + b, L, Hkv, 128, ch), synth.outlier_kv(1220 + b, L, Hkv, 128, ch)
        K, V = helpers.to_dev_bf16(Kn), helpers.to_dev_bf16(Vn)
        Ou.prefill(b, Kn, Vn)
        ok.oscar_prefill_pool(Pu, b, K, V)
        ok.oscar_prefill_pool(Pc, b, K, V)
    for t in range(5):
        knn, vnn = synth.outlier_kv(1230 + t, 2, Hkv, 128, ch), synth.outlier_kv(1240 + t, 2, Hkv, 128, ch)
        kn, vn = helpers.to_dev_bf16(knn), helpers.to_dev_bf16(vnn)
        Ou.append(knn, vnn)
        ok.oscar_append_kv(Pu, kn, vn)
        ok.oscar_append_kv(Pc, kn, vn)
    torch.cuda.synchronize()
    for name in helpers.POOL_ARRAYS:
        assert np.array_equal(helpers.device_array(Pu, name), helpers.device_array(Pc, name)), name
    qn = synth.outlier_q(1250, len(lens), Hq, Hkv, 128, ch)
    q = helpers.to_dev_bf16(qn)
    # group 32 decodes the two pools on different paths (tensor cores for the uniform levels, CUDA cores for a
    # codebook): each is held to the oracle's tolerance, and to the same tolerance against each other
    ref = Ou.decode(qn)
    oc, ou = ok.oscar_decode_attention(Pc, q).cpu().numpy(), ok.oscar_decode_attention(Pu, q).cpu().numpy()
    helpers.assert_attention_close(oc, ref)
    helpers.assert_attention_close(ou, ref)
    helpers.assert_attention_close(oc, ou.astype(np.float64))


def _codebooks_from_oracle(seed, Hkv, Rk, Rv, clip):
    """Lloyd-Max levels of each head computed by the oracle on calibration rows of the same distribution."""
    Kc, ch = _rows(seed, 400, Hkv)
    Vc = synth.outlier_kv(seed + 2, 400, Hkv, 128, ch)
    cbk = np.stack([ocb.lloyd_max(ocb.calibration_values(Kc[:, h], Rk[h], clip, 128)) for h in range(Hkv)])
    cbv = np.stack([ocb.lloyd_max(ocb.calibration_values(Vc[:, h], Rv[h], clip, 128)) for h in range(Hkv)])
    return cbk, cbv


@pytest.mark.parametrize("G,g", [(4, 128), (8, 128), (1, 128), (2, 64)])
def test_codebook_pool_prefill_steps_and_attention_match_oracle(G, g):
    seed, Hkv = 1300 + G + g, 2
    Hq, lens = G * Hkv, [350, 1400]
    Rk, Rv = helpers.oracle_rotations(seed, Hkv), helpers.oracle_rotations(seed + 1000, Hkv)
    cbk, cbv = _codebooks_from_oracle(seed + 50, Hkv, Rk, Rv, 0.9)
    assert not np.array_equal(cbk[0], ocb.UNIFORM)
    pages = [-(-(L - 320) // 64) for L in lens]
    O, P = helpers.make_pools(len(lens), Hq, Hkv, g, pages, seed, extra_pages=2, codebook_k=cbk, codebook_v=cbv)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for b, L in enumerate(lens):
        K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
        V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
        O.prefill(b, K, V)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    q = synth.outlier_q(seed + 7, len(lens), Hq, Hkv, 128, ch)
    helpers.assert_attention_close(ok.oscar_decode_attention(P, helpers.to_dev_bf16(q)).cpu().numpy(), O.decode(q))
    for t in range(40):   # demotions into history pages (sequence 0 crosses a page boundary)
        kn = synth.outlier_kv(seed + 2000 + t, 2, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, 2, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, 2, Hq, Hkv, 128, ch)
        O.append(kn, vn)
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        if t % 13 == 0 or t == 39:
            helpers.assert_attention_close(out.cpu().numpy(), O.decode(qt))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0


@pytest.mark.parametrize("g", [128, 32])
def test_lloyd_max_calibration_matches_oracle(g):
    Hkv = 2
    X, _ = _rows(1400 + g, 1500, Hkv)
    R = np.stack([orot.to_f32(orot.hadamard(128) @ orot.bitrev_matrix(128)), helpers.oracle_rotations(1401, 1)[0]])
    clip = np.array([0.9, 1.0], np.float32)
    cb = ok.oscar_lloyd_max_codebook(helpers.to_dev_bf16(X), torch.from_numpy(R).cuda(),
                                     torch.from_numpy(clip).cuda(), group_size=g).cpu().numpy()
    for h in range(Hkv):
        ref = ocb.lloyd_max(ocb.calibration_values(X[:, h], R[h], clip[h], g))
        np.testing.assert_allclose(cb[h], ref, rtol=0, atol=1e-4)
        assert np.all(np.diff(cb[h]) > 0)


def test_lloyd_max_without_rows_and_without_iterations_keeps_uniform_levels():
    Hkv = 2
    R = torch.from_numpy(helpers.oracle_rotations(1450, Hkv)).cuda()
    clip = torch.full((Hkv,), 0.9, device="cuda")
    x0 = torch.empty((0, Hkv, 128), dtype=torch.bfloat16, device="cuda")
    uni = np.stack([ocb.UNIFORM] * Hkv)
    assert np.array_equal(ok.oscar_lloyd_max_codebook(x0, R, clip).cpu().numpy(), uni)
    X, _ = _rows(1451, 50, Hkv)
    assert np.array_equal(ok.oscar_lloyd_max_codebook(helpers.to_dev_bf16(X), R, clip, max_iters=0).cpu().numpy(), uni)


def test_codebook_alignment_is_checked():
    Hkv = 2
    X, _ = _rows(1460, 4, Hkv)
    R = torch.from_numpy(helpers.oracle_rotations(1461, Hkv)).cuda()
    clip = torch.full((Hkv,), 0.9, device="cuda")
    buf = torch.zeros(4 * Hkv + 1, dtype=torch.float32, device="cuda")
    with pytest.raises(ok.OscarError):
        ok.oscar_quantize_kv_codebook(helpers.to_dev_bf16(X), R, clip, buf[1:].view(Hkv, 4))
