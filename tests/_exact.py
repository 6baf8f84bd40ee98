"""Exact integration over a uniform u in (0, 1) for decisions that are monotone in u.

A decision taken by comparing u against fixed fp64 thresholds partitions (0, 1)
into intervals. The boundaries are located by bisection down to adjacent
doubles, so each outcome's measure is exact to ~1e-16.
"""
import numpy as np

U_LO = 2.0 ** -60
U_HI = 1.0 - 2.0 ** -53


def outcome_measures(f):
    """{outcome: measure of {u : f(u) == outcome}} for f monotone (piecewise constant) in u."""
    res = {}
    start = 0.0
    u = U_LO
    fu = f(u)
    f_hi = f(U_HI)
    while fu != f_hi:
        a, b = u, U_HI
        while np.nextafter(a, 1.0) < b:
            m = 0.5 * (a + b)
            if m <= a or m >= b:
                break
            if f(m) == fu:
                a = m
            else:
                b = m
        res[fu] = res.get(fu, 0.0) + (b - start)
        start = b
        u = b
        fu = f(b)
    res[fu] = res.get(fu, 0.0) + (1.0 - start)
    return res
