"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks
that the pin suite in test_oracle.py rejects every one of them."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "update_multiplies_from_right": ("return 0.25 * (z @ outer)", "return 0.25 * (outer @ z)"),
    "constant_13": ("13.0 * eye", "12.0 * eye"),
    "constant_7_sign": ("inner = 7.0 * eye - az", "inner = 7.0 * eye + az"),
    "init_not_transposed": ("return a.T / (norm1 * norminf)", "return a / (norm1 * norminf)"),
    "init_frobenius": ("norminf = np.abs(a).sum(axis=1).max()", "norminf = np.sqrt((a * a).sum())"),
    "one_update_too_many": ("for _ in range(iters):\n        z = pinv_step(a, z)",
                            "for _ in range(iters + 1):\n        z = pinv_step(a, z)"),
    "softmax_wrong_axis": ("e = np.exp(s - s.max(axis=1, keepdims=True))\n    return e / e.sum(axis=1, keepdims=True)",
                           "e = np.exp(s - s.max(axis=0, keepdims=True))\n    return e / e.sum(axis=0, keepdims=True)"),
    "landmark_scale_1_over_d": ("return softmax_rows(q_tilde @ k_tilde.T / np.sqrt(d))",
                                "return softmax_rows(q_tilde @ k_tilde.T / d)"),
    "left_factor_unscaled": ("return softmax_rows(q @ k_tilde.T / np.sqrt(d)) @ w",
                             "return softmax_rows(q @ k_tilde.T) @ w"),
    "right_factor_scale": ("return softmax_rows(q_tilde @ k.T / np.sqrt(d)) @ v",
                           "return softmax_rows(q_tilde @ k.T / d) @ v"),
    "conv_flipped": ("out[lo:hi] += w[j] * v[lo + shift:hi + shift]",
                     "out[lo:hi] += w[ks - 1 - j] * v[lo + shift:hi + shift]"),
    "conv_off_by_one": ("shift = j - r", "shift = j - r - 1"),
    "strided_segments": ("out[i] = x[lo:hi].mean(axis=0)",
                         "out[i] = x[i::m].mean(axis=0)"),
    "remainder_in_last_segment": (
        "return [(i * n // m, (i + 1) * n // m) for i in range(m)]",
        "return [(i * (n // m), (i + 1) * (n // m) if i < m - 1 else n) for i in range(m)]"),
    "remainder_in_first_segments": (
        "return [(i * n // m, (i + 1) * n // m) for i in range(m)]",
        "return [(i * (n // m) + min(i, n % m), (i + 1) * (n // m) + min(i + 1, n % m))"
        " for i in range(m)]"),
    "z_transposed": ("w_mat = z @ g", "w_mat = z.T @ g"),
    "padding_keys_unmasked": ("g = masked_softmax_rows(q_tilde @ k.T / np.sqrt(d), valid) @ v",
                              "g = softmax_rows(q_tilde @ k.T / np.sqrt(d)) @ v"),
    "padding_read_by_conv": ("conv = conv_of(np.where(valid[:, None], v, 0.0), w)",
                             "conv = conv_of(v, w)"),
    "padded_landmarks_over_all_rows": ("q_tilde = segment_means(q[:length], m)",
                                       "q_tilde = segment_means(q, m)"),
    "channel_filters_shared": ("out[t] += w[:, j] * v[u]", "out[t] += w[0, j] * v[u]"),
    "conv_dropped": ('"out": att + conv', '"out": att'),
}


@pytest.fixture(scope="module")
def source():
    return open(os.path.join(ROOT, "oracle", "nystrom_ref.py")).read()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutation(name, source, tmp_path):
    old, new = MUTATIONS[name]
    assert old in source, f"mutation site for {name} not found"
    repo = tmp_path / "repo"
    (repo / "oracle").mkdir(parents=True)
    shutil.copytree(os.path.join(ROOT, "tests"), repo / "tests",
                    ignore=shutil.ignore_patterns("test_oracle_mutations.py", "__pycache__"))
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), repo / "oracle" / "__init__.py")
    (repo / "oracle" / "nystrom_ref.py").write_text(source.replace(old, new, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-W", "ignore", "tests/test_oracle.py"],
                       cwd=repo, capture_output=True, text=True, timeout=300)
    assert r.returncode == 1, f"pins did not catch {name}:\n{r.stdout[-2000:]}"
