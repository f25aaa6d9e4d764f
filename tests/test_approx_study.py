"""The approximation study's grid (oracle only, CPU)."""
import numpy as np

import approx_study as S


def test_grid_is_complete_and_finite():
    errs = S.approx_errors("clustered", 256, 16, [16, 64], [0, 6], heads=1)
    assert set(errs) == {(m, key) for m in (16, 64) for key in (0, 6, "svd")}
    assert all(np.isfinite(list(errs.values())))


def test_one_landmark_per_token_with_the_svd_inverse_is_exact():
    """m = n: every landmark is one token, the three softmax factors are the
    same matrix S, and S S^+ S = S (a Penrose condition), so the product is
    exact attention (Proposed method, bullet 3)."""
    errs = S.approx_errors("normal", 32, 16, [32], [0], heads=2)
    assert errs[(32, "svd")] < 1e-9
    assert errs[(32, 0)] > 1e-3  # Z_0 alone is not the inverse


def test_families_differ_only_by_the_segment_drift():
    qn, kn, vn = S.draw("normal", 256, 16, 1, 3)
    qc, kc, vc = S.draw("clustered", 256, 16, 1, 3)
    drift = qc - qn
    assert np.abs(drift).max() > 0.1
    # the drift is constant over each of the 128 segments and shared by Q, K, V
    seg = drift.reshape(1, 128, 2, 16)
    np.testing.assert_allclose(seg[:, :, 0], seg[:, :, 1], atol=1e-6)
    np.testing.assert_allclose(kc - kn, drift, atol=1e-5)
    np.testing.assert_allclose(vc - vn, drift, atol=1e-5)
