"""GPU parity: rotation construction R = U·H·P and the calibration covariances against the oracle.

R = U · Hadamard · bit-reversal; U from Q^T Q (keys) and V^T S^T S V (values)
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计";
"OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract).
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import bit_rotated_kv_02_gb300 as ok
from oracle import rotation as orot
import synth
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _f32_agrees(R32_gpu, R64_ref):
    """R32 is the nearest float32 to R64; entries may differ only where R64 sits next to a midpoint."""
    ref32 = orot.to_f32(R64_ref)
    bad = R32_gpu != ref32
    if bad.any():
        r = R64_ref[bad]
        mid = (ref32[bad].astype(np.float64) + R32_gpu[bad].astype(np.float64)) / 2
        assert np.all(np.abs(r - mid) < 1e-12)


@pytest.mark.parametrize("d", [8, 32, 128])
def test_haar_rotation(d):
    G = synth.gaussian_matrix(100 + d, d)
    R64, R32 = ok.oscar_make_rotation(torch.from_numpy(G).cuda(), ok.ROT_HAAR)
    R64, R32 = R64.cpu().numpy(), R32.cpu().numpy()
    ref = orot.rotation_from_gaussian(G)
    assert np.max(np.abs(R64 - ref)) < 1e-10
    assert np.max(np.abs(R64 @ R64.T - np.eye(d))) < 1e-12
    _f32_agrees(R32, ref)


@pytest.mark.parametrize("d", [16, 128])
def test_covariance_rotation(d):
    V0 = orot.haar_orthogonal(synth.gaussian_matrix(200 + d, d))
    lam = 2.0 / (np.arange(d) + 1.0) + 0.1
    C = (V0 * lam) @ V0.T
    R64, R32 = ok.oscar_make_rotation(torch.from_numpy(C).cuda(), ok.ROT_COVARIANCE)
    R64 = R64.cpu().numpy()
    ref = orot.rotation_from_covariance(C)
    assert np.max(np.abs(R64 - ref)) < 1e-10
    _f32_agrees(R32.cpu().numpy(), ref)
    # U = R P H (H, P involutions) diagonalises C with descending eigenvalues
    U = R64 @ orot.bitrev_matrix(d) @ orot.hadamard(d)
    assert np.max(np.abs(C @ U - U * lam)) <= 1e-10 * np.max(np.abs(C))


def test_calibration_covariances():
    T, H, d = 300, 4, 128
    ch = synth.outlier_channels(7, 1, d, 4)
    Q = synth.calib_samples(8, T, H, d, ch, heads_per_channel_set=H)
    KV = synth.calib_samples(9, T, 2, d, ch, heads_per_channel_set=2)
    f = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)
    Ck = ok.oscar_calib_covariance_k(helpers.to_dev_bf16(Q)).cpu().numpy()
    ref_k = orot.covariance_k(f(Q))
    assert np.max(np.abs(Ck - ref_k)) <= 1e-12 * np.max(np.abs(ref_k))
    Cv = ok.oscar_calib_covariance_v(helpers.to_dev_bf16(Q), helpers.to_dev_bf16(np.ascontiguousarray(KV[:, 0])),
                                     helpers.to_dev_bf16(np.ascontiguousarray(KV[:, 1]))).cpu().numpy()
    ref_v = orot.covariance_v(f(Q), f(KV[:, 0]), f(KV[:, 1]))
    assert np.max(np.abs(Cv - ref_v)) <= 1e-11 * np.max(np.abs(ref_v))


def test_rotation_from_calibration_matches_oracle():
    """Covariance-aligned rotation from synthetic anisotropic calibration samples, end to end."""
    T, H, d = 512, 4, 128
    ch = synth.outlier_channels(11, 1, d, 4)
    Q = synth.calib_samples(12, T, H, d, ch, heads_per_channel_set=H)
    Ck = ok.oscar_calib_covariance_k(helpers.to_dev_bf16(Q))
    R64, _ = ok.oscar_make_rotation(Ck, ok.ROT_COVARIANCE)
    ref_C = orot.covariance_k(synth.bf16_bits_to_f32(Q).astype(np.float64))
    w, _ = orot.canonical_eigenvectors(ref_C)
    gaps = np.min(np.abs(np.diff(w))) / np.max(np.abs(w))
    ref = orot.rotation_from_covariance(ref_C)
    tol = max(1e-10, 1e-14 / gaps)
    assert np.max(np.abs(R64.cpu().numpy() - ref)) < tol
