"""Fit the polynomial used by the FMA-only exp2 in the softmax.

The FlashAttention-4 paper (Section 3.1.3, "Emulation of the exponential
function") computes 2^x on the FMA units for part of the softmax entries:
Cody-Waite range reduction x = n + f with n = floor(x), f in [0, 1), a short
polynomial p(f) ~ 2^f evaluated by Horner's rule, and the scaling by 2^n done
as an integer add on the exponent field. The pages give no coefficients, so
this script fits them: a minimax (Remez exchange) fit of the RELATIVE error
of p(f) = 1 + c1 f + ... + cn f^n against 2^f on [0, 1], with p(0) = 1
pinned so that 2^0 and every power of two come out exact. The coefficients
are then rounded to fp32 and the error of the fp32 Horner evaluation is
measured on a dense grid.

    python fit_exp2_poly.py            # prints the coefficient table for degrees 3 and 4
"""
from __future__ import annotations

import numpy as np


def remez(deg: int, iters: int = 60, grid: int = 200001):
    xs = np.linspace(0.0, 1.0, grid)
    # initial reference: deg+1 points in (0, 1], endpoint included
    ref = 0.5 - 0.5 * np.cos(np.pi * (np.arange(1, deg + 2)) / (deg + 1))
    coef = None
    for _ in range(iters):
        # unknowns c1..c_deg and E:  sum_k c_k x^k - s_i E 2^x = 2^x - 1
        A = np.zeros((deg + 1, deg + 1))
        rhs = np.exp2(ref) - 1.0
        for i, x in enumerate(ref):
            A[i, :deg] = [x ** k for k in range(1, deg + 1)]
            A[i, deg] = -((-1) ** i) * np.exp2(x)
        sol = np.linalg.solve(A, rhs)
        coef = np.concatenate([[1.0], sol[:deg]])
        err = np.polyval(coef[::-1], xs) / np.exp2(xs) - 1.0
        # new reference: the extremum of each sign run, deg+1 of them, largest first
        sign = np.sign(err)
        sign[sign == 0] = 1
        runs, start = [], 1   # skip x = 0 where the error is pinned to zero
        for j in range(2, len(xs) + 1):
            if j == len(xs) or sign[j] != sign[start]:
                seg = slice(start, j)
                k = start + int(np.argmax(np.abs(err[seg])))
                runs.append(k)
                start = j
        runs = sorted(runs, key=lambda k: -abs(err[k]))[: deg + 1]
        new_ref = np.sort(xs[runs])
        if len(new_ref) < deg + 1 or np.allclose(new_ref, ref, atol=1e-12):
            break
        ref = new_ref
    return coef


def horner_fp32(coef32: np.ndarray, f: np.ndarray) -> np.ndarray:
    """fp32 Horner evaluation (each step rounded to fp32, as an FMA chain does)."""
    acc = np.full_like(f, coef32[-1], dtype=np.float32)
    for c in coef32[-2::-1]:
        acc = (acc.astype(np.float64) * f.astype(np.float64) + np.float64(c)).astype(np.float32)
    return acc


def report(deg: int):
    coef = remez(deg)
    c32 = coef.astype(np.float32)
    c32[0] = np.float32(1.0)
    f = np.linspace(0.0, 1.0, 1_000_001, dtype=np.float32)
    approx = horner_fp32(c32, f).astype(np.float64)
    rel = np.abs(approx / np.exp2(f.astype(np.float64)) - 1.0)
    return c32, float(rel.max())


if __name__ == "__main__":
    for deg in (3, 4):
        c32, err = report(deg)
        print(f"degree {deg}: max relative error {err:.3e} (bf16 half-ulp 1.95e-03)")
        for k, c in enumerate(c32):
            print(f"  c{k} = {float(c):.9e}f  /* 0x{np.float32(c).view(np.uint32):08x} */")
