"""Coefficients of the software exp2 used by the forward kernel's optional path.

2^x = 2^n * 2^f with n = floor(x) and f in [0, 1); 2^f is approximated by the cubic
p(f) = 1 + c1 f + c2 f^2 + c3 f^3 that minimises the maximum relative error on [0, 1] under
p(0) = 1 ("B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams", Chapter 9 and its
appendix on how the software exp2 works: a low-degree polynomial for the fractional part, the
integer part added to the exponent field).  The fit is a Remez exchange on the relative error;
`python -m dense_attention_forward_attn_gb300.soft_exp2_fit` prints the coefficients written
into attn_fwd_kernel.cuh (kExp2C1..kExp2C3).
"""
import numpy as np


def relative_error(c, f):
    """(p(f) - 2^f) / 2^f for coefficients c = (c1, c2, c3), in fp64."""
    c1, c2, c3 = c
    t = np.exp2(f)
    return (1.0 + f * (c1 + f * (c2 + f * c3)) - t) / t


def fit(iterations: int = 40, grid_points: int = 200001):
    """Minimax (c1, c2, c3) and the maximum relative error on [0, 1]."""
    grid = np.linspace(0.0, 1.0, grid_points)
    pts = np.array([0.1, 0.4, 0.75, 1.0])   # alternation points; f = 0 is exact by construction
    c = np.zeros(3)
    for _ in range(iterations):
        a = np.zeros((4, 4))
        b = np.zeros(4)
        for r, f in enumerate(pts):
            t = 2.0 ** f
            a[r, :3] = [f / t, f * f / t, f ** 3 / t]
            a[r, 3] = -((-1.0) ** r)      # error alternates in sign
            b[r] = (t - 1.0) / t
        sol = np.linalg.solve(a, b)
        c = sol[:3]
        err = relative_error(c, grid)
        turn = np.diff(np.sign(np.diff(err))) != 0
        ext = [e for e in list(grid[1:-1][turn]) + [1.0] if e > 1e-6]
        if len(ext) == 4:
            pts = np.array(ext)
    return tuple(float(x) for x in c), float(np.abs(relative_error(c, grid)).max())


if __name__ == "__main__":
    (c1, c2, c3), e = fit()
    f32 = [np.format_float_positional(np.float32(x), unique=True) for x in (c1, c2, c3)]
    print(f"kExp2C1 = {f32[0]}f, kExp2C2 = {f32[1]}f, kExp2C3 = {f32[2]}f  (max relative error {e:.3g})")
