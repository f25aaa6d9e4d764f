"""Write closed_form_n4_m2.json: a worked example of Nyström attention whose
every value follows from a hand derivation (uses only ``math``; neither the
oracle nor the CUDA library).

The Nyströmformer review page prints no worked example, so this fixture is
derived instead. Setup (one head, d = 64, so 1/sqrt(d) = 1/8):

    Q = K = 4 * [e0, e0, e1, e1]   (n = 4 rows; e_i = i-th unit vector)
    m = 2 segments of 2 rows  ->  Q~ = K~ = 4 * [e0, e1]

Every score matrix then has entries 16/8 = 2 (same unit vector) or 0, so
with a = e^2/(1+e^2) and b = 1/(1+e^2) (a + b = 1, a - b = tanh 1):

    A_S = softmax(Q~ K~^T/8) = [[a, b], [b, a]]
    F   = softmax(Q K~^T/8)  : rows 0,1 = [a, b]; rows 2,3 = [b, a]
    B   = softmax(Q~ K^T/8)  : row 0 = [a, a, b, b]/2; row 1 = [b, b, a, a]/2

A_S is symmetric with eigenvectors (1, 1)/sqrt2, (1, -1)/sqrt2 and
eigenvalues s1 = 1, s2 = tanh 1. ||A_S||_1 = ||A_S||_inf = 1, so
Z_0 = A_S^T = A_S. Every update keeps the eigenvectors; with the residual
e = 1 - s z of an eigenvalue s, one update of
Z <- 1/4 Z (13I - A Z (15I - A Z (7I - A Z))) maps e to 3/4 e^3 + 1/4 e^4
(expand 1 - x(13 - 15x + 7x^2 - x^3)/4 at x = 1 - e). From e_0 = 1 - s^2:
z_k = (1 - e_k) / s, and Z_k = 1/2 [[z1 + z2, z1 - z2], [z1 - z2, z1 + z2]].

Then G = B V, W = Z_k G, att = F W, and with a 3-tap filter (w0, w1, w2)
conv[t] = w0 V[t-1] + w1 V[t] + w2 V[t+1] (zero outside 0..3).
Only columns 0..3 of V are non-zero; the other 60 are zero.

Second fixture, closed_form_n8_m3.json: n = 8 rows, m = 3, where m does not
divide n. Segment i is rows [floor(i n/m), floor((i+1) n/m)), so the
segments are rows {0, 1}, {2, 3, 4} and {5, 6, 7} (lengths 2, 3, 3; putting
the remainder last would give 2, 2, 4, and giving it to the first segments
3, 3, 2). With

    Q = K = 4 * [e0, e0, e1, e1, e1, e2, e2, e2]

every segment is constant and Q~ = K~ = 4 * [e0, e1, e2]. With E = e^2,
a' = E/(E+2), b' = 1/(E+2): A_S has a' on the diagonal and b' elsewhere; it
is symmetric with eigenvalue 1 on (1, 1, 1)/sqrt3 and (E-1)/(E+2) on the
plane orthogonal to it, ||A_S||_1 = ||A_S||_inf = 1, so Z_0 = A_S and
Z_k = z1 P + z2 (I - P) with P = 1 1^T / 3 and z from the same residual map
as above. Row t of F is b' everywhere but a' at t's segment; row i of B
gives weight E / c_i to the keys of segment i and 1 / c_i to the others,
c_i = len_i E + (n - len_i).
"""
import json
import math
import os

D = 64
V_SMALL = [[1.0, 0.0, 2.0, -1.0],
           [0.0, 3.0, -2.0, 1.0],
           [2.0, 1.0, 0.0, 4.0],
           [-1.0, 2.0, 1.0, 0.0]]
W3 = [0.25, 1.0, -0.5]


def main():
    a = math.exp(2.0) / (1.0 + math.exp(2.0))
    b = 1.0 / (1.0 + math.exp(2.0))
    s = [1.0, math.tanh(1.0)]
    V = [row + [0.0] * (D - 4) for row in V_SMALL]
    half = [[a / 2, a / 2, b / 2, b / 2], [b / 2, b / 2, a / 2, a / 2]]
    G = [[sum(half[i][t] * V[t][c] for t in range(4)) for c in range(D)] for i in range(2)]
    F = [[a, b], [a, b], [b, a], [b, a]]
    conv = [[sum(W3[j] * V[t + j - 1][c] for j in range(3) if 0 <= t + j - 1 < 4)
             for c in range(D)] for t in range(4)]
    cases = []
    for iters in (0, 1, 2, 6, 12):
        z = []
        for sv in s:
            e = 1.0 - sv * sv
            for _ in range(iters):
                e = 0.75 * e ** 3 + 0.25 * e ** 4
            z.append((1.0 - e) / sv)
        Z = [[(z[0] + z[1]) / 2, (z[0] - z[1]) / 2], [(z[0] - z[1]) / 2, (z[0] + z[1]) / 2]]
        Wm = [[sum(Z[i][j] * G[j][c] for j in range(2)) for c in range(D)] for i in range(2)]
        att = [[sum(F[t][i] * Wm[i][c] for i in range(2)) for c in range(D)] for t in range(4)]
        cases.append({"iters": iters, "z": Z, "w": Wm, "att": att,
                      "out": [[att[t][c] + conv[t][c] for c in range(D)] for t in range(4)]})
    q = [[0.0] * D for _ in range(4)]
    for t in range(4):
        q[t][0 if t < 2 else 1] = 4.0
    fixture = {
        "source": "hand derivation (see make_closed_form.py); the Nyströmformer review "
                  "page, Proposed method bullets 1-6, defines the computation",
        "n": 4, "d": D, "m": 2, "conv_w": W3,
        "q": q, "k": q, "v": V,
        "a_s": [[a, b], [b, a]], "g": G, "conv": conv, "cases": cases,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_form_n4_m2.json")
    with open(path, "w") as f:
        json.dump(fixture, f)
    print("wrote", path)


V8_SMALL = V_SMALL + [[3.0, -1.0, 1.0, 2.0],
                      [0.5, 0.0, -3.0, 1.0],
                      [-2.0, 1.0, 2.0, -1.0],
                      [1.0, 1.0, 1.0, 3.0]]


def ragged():
    """closed_form_n8_m3.json (see the module docstring)."""
    n, m = 8, 3
    seg_of = [0, 0, 1, 1, 1, 2, 2, 2]
    lens = [2, 3, 3]
    E = math.exp(2.0)
    ap, bp = E / (E + 2.0), 1.0 / (E + 2.0)
    s = [1.0, (E - 1.0) / (E + 2.0)]
    V = [row + [0.0] * (D - 4) for row in V8_SMALL]
    Bm = [[(E if seg_of[t] == i else 1.0) / (lens[i] * E + (n - lens[i])) for t in range(n)]
          for i in range(m)]
    G = [[sum(Bm[i][t] * V[t][c] for t in range(n)) for c in range(D)] for i in range(m)]
    F = [[ap if i == seg_of[t] else bp for i in range(m)] for t in range(n)]
    A = [[ap if i == j else bp for j in range(m)] for i in range(m)]
    conv = [[sum(W3[j] * V[t + j - 1][c] for j in range(3) if 0 <= t + j - 1 < n)
             for c in range(D)] for t in range(n)]
    cases = []
    for iters in (0, 1, 6):
        z = []
        for sv in s:
            e = 1.0 - sv * sv
            for _ in range(iters):
                e = 0.75 * e ** 3 + 0.25 * e ** 4
            z.append((1.0 - e) / sv)
        Z = [[z[0] / 3 + z[1] * ((1.0 if i == j else 0.0) - 1.0 / 3) for j in range(m)]
             for i in range(m)]
        Wm = [[sum(Z[i][j] * G[j][c] for j in range(m)) for c in range(D)] for i in range(m)]
        att = [[sum(F[t][i] * Wm[i][c] for i in range(m)) for c in range(D)] for t in range(n)]
        cases.append({"iters": iters, "z": Z, "w": Wm, "att": att,
                      "out": [[att[t][c] + conv[t][c] for c in range(D)] for t in range(n)]})
    q = [[0.0] * D for _ in range(n)]
    for t in range(n):
        q[t][seg_of[t]] = 4.0
    fixture = {
        "source": "hand derivation (see make_closed_form.py); the Nyströmformer review "
                  "page, Proposed method bullets 1-6, defines the computation; segments "
                  "of 2, 3 and 3 rows by the even-split reading of segment means",
        "n": n, "d": D, "m": m, "conv_w": W3,
        "q": q, "k": q, "v": V,
        "a_s": A, "g": G, "conv": conv, "cases": cases,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_form_n8_m3.json")
    with open(path, "w") as f:
        json.dump(fixture, f)
    print("wrote", path)


if __name__ == "__main__":
    main()
    ragged()
