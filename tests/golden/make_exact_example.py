"""Write exact_a0_T4_d2.json: a tiny worked example of the 2Mamba mixer in exact
rational arithmetic, straight from the definition in "2Mamba2Furious" Sec. 5
(squared QK inner product, softplus A-mask applied to the squared scores,
"softmax" normalisation read as o_i = N_i / Z_i).

With a_t = 0 every step's decay is exp(-softplus(0)) = exp(-log 2) = 1/2 exactly,
so the A-mask between tokens j <= i is 2^-(i-j) and every output is a rational
number.  q, k, v are small integers.  Nothing here calls the oracle or the CUDA
path: the expected values come from Fractions only.

Run:  python tests/golden/make_exact_example.py
"""
import json
import os
from fractions import Fraction

T, d, dv = 4, 2, 2
q = [[1, 2], [-1, 1], [2, 0], [1, -3]]
k = [[1, 0], [2, -1], [0, 1], [-1, 1]]
v = [[3, -1], [1, 2], [-2, 5], [4, 0]]


def main():
    o_norm, o_raw, Z = [], [], []
    for i in range(T):
        num = [Fraction(0)] * dv
        den = Fraction(0)
        for j in range(i + 1):
            s = sum(q[i][m] * k[j][m] for m in range(d))
            w = Fraction(1, 2 ** (i - j)) * s * s
            den += w
            for c in range(dv):
                num[c] += w * v[j][c]
        o_raw.append([str(x) for x in num])
        o_norm.append([str(x / den) for x in num])
        Z.append(str(den))
    out = {
        "source": "2Mamba2Furious, Sec. 5: w_ij = exp(cumA_i - cumA_j) (q_i.k_j)^2, "
                  "cumA_t = sum_{u<=t} -softplus(a_u); a = 0 gives decay 1/2 per step",
        "T": T, "d": d, "dv": dv, "a": [0.0] * T, "q": q, "k": k, "v": v,
        "o_normalized": o_norm, "o_unnormalized": o_raw, "Z": Z,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "exact_a0_T4_d2.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(path)


if __name__ == "__main__":
    main()
