"""Writes rope_freqs.txt: the float64 nearest to theta^(-2j/D) for the rotary
layouts the workloads and tests use, evaluated with mpmath at 200 bits (an
independent high-precision evaluation, so that the platform pow of either side
is checked, not trusted).

    python tests/golden/make_rope_freqs.py
"""
import os

import mpmath

LAYOUTS = [(1e4, 64), (1e4, 128), (1e4, 256), (1e4, 512), (1e6, 64), (1e6, 128), (1e6, 256), (1e6, 512)]


def main():
    mpmath.mp.prec = 200
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rope_freqs.txt")
    with open(out, "w") as f:
        f.write("# theta head_dim j nearest-float64(theta^(-2j/head_dim)) as a hex float; mpmath, 200 bits\n")
        for theta, D in LAYOUTS:
            for j in range(D // 2):
                v = mpmath.power(mpmath.mpf(theta), mpmath.mpf(-2 * j) / D)
                f.write(f"{theta:g} {D} {j} {float(v).hex()}\n")


if __name__ == "__main__":
    main()
