"""Coefficients of the FMA-pipe 2^x in ssm_common.cuh (`ex2_fma`).

2^f on [-0.5, 0.5] by the degree-6 polynomial that interpolates it at the
seven Chebyshev nodes of the interval (close to the minimax polynomial),
rounded to float32. Prints the coefficients (c0 first) and the largest
relative error of the float32 Horner evaluation on a dense grid, with each
step rounded (the device fuses them, which is no worse).

    python selective_state_space_07_gb300/csrc/exp2_poly.py
"""
import numpy as np

DEG = 6


def coefficients(deg=DEG):
    k = np.arange(deg + 1)
    nodes = 0.5 * np.cos((2 * k + 1) * np.pi / (2 * (deg + 1)))
    return np.linalg.solve(np.vander(nodes, deg + 1, increasing=True), 2.0 ** nodes).astype(np.float32)


def horner32(c, f):
    acc = np.full_like(f, c[-1])
    for j in range(len(c) - 2, -1, -1):
        acc = (acc * f + c[j]).astype(np.float32)
    return acc


if __name__ == "__main__":
    c = coefficients()
    f = np.linspace(-0.5, 0.5, 400001).astype(np.float32)
    err = np.max(np.abs(horner32(c, f).astype(np.float64) / 2.0 ** f.astype(np.float64) - 1.0))
    for j, v in enumerate(c):
        print(f"c{j} = {float(v)!r}f  (0x{np.float32(v).view(np.uint32):08x})")
    print(f"max relative error on [-0.5, 0.5]: {err:.3e}")
