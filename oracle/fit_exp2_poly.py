"""Fit of the polynomial inside the oracle's exp2_det (test infrastructure, like the rest of oracle/).

exp2_det(x) = 2^n * p(f) with n = rint(x), f = x - n in [-1/2, 1/2], and
p(f) = 1 + c1 f + c2 f^2 + c3 f^3 + c4 f^4 (Horner in fp32 fma).  The constant term is fixed at 1
so that integer arguments are exact.  c1..c4 minimise the largest relative error
|p(f) / 2^f - 1| on [-1/2, 1/2]; this script finds them by the Remez exchange algorithm (the
relative-error form: at each reference set solve p(f_i) - 2^f_i = (-1)^i E 2^f_i for c1..c4 and E,
then move the reference to the extrema of the error), rounds them to fp32, and reports the error of
the rounded polynomial in exact arithmetic and of oracle.exp2_det itself, the fp32 evaluation.
With p(0) = 1 the relative error is e(f) = f 2^-f (q(f) - (2^f - 1) / f), q the cubic c1 + c2 f +
c3 f^2 + c4 f^3: a weighted approximation of (2^f - 1) / f by q with the weight |f| 2^-f, which
vanishes at f = 0.  The alternation that characterises the optimum is that of the weighted error
e(f) sign(f), not of e(f) itself (e changes sign at f = 0 whether or not q - (2^f - 1) / f does).

Run: python -m oracle.fit_exp2_poly   (only numpy and the oracle are used)
"""
import numpy as np

DEGREE = 4


def _err(c, f):
    p = 1.0 + sum(ci * f ** (i + 1) for i, ci in enumerate(c))
    return p / np.exp2(f) - 1.0


def remez(iters=30):
    n = DEGREE + 1  # unknowns c1..c4 and E, as many reference points
    # Chebyshev points of [-1/2, 1/2] as the first reference
    ref = 0.5 * np.cos(np.pi * (np.arange(n) + 0.5) / n)[::-1]
    grid = np.linspace(-0.5, 0.5, 200001)
    c = np.zeros(DEGREE)
    E = 0.0
    for _ in range(iters):
        A = np.zeros((n, n))
        rhs = np.exp2(ref) - 1.0
        for i, f in enumerate(ref):
            A[i, :DEGREE] = [f ** (k + 1) for k in range(DEGREE)]
            A[i, DEGREE] = -((-1) ** i) * np.sign(f) * np.exp2(f)
        sol = np.linalg.solve(A, rhs)
        c, E = sol[:DEGREE], sol[DEGREE]
        e = _err(c, grid) * np.sign(grid)  # the weighted error
        # new reference: the extremum of each sign-alternating segment of the error (e(0) = 0 for
        # every candidate, since p(0) = 1: that zero takes the sign of its neighbour instead of
        # cutting a segment)
        sign = np.sign(e)
        for i in np.flatnonzero(sign == 0):
            sign[i] = sign[i - 1] if i > 0 else sign[i + 1]
        cuts = np.flatnonzero(np.diff(sign) != 0) + 1
        segs = np.split(np.arange(grid.size), cuts)
        ext = [s[np.argmax(np.abs(e[s]))] for s in segs]
        if len(ext) < n:
            break
        # keep n alternating extrema with the largest magnitudes, in order
        while len(ext) > n:
            drop = min(range(len(ext)), key=lambda k: abs(e[ext[k]]))
            ext.pop(drop)
        ref = grid[np.array(ext)]
    return c, abs(E)


def main():
    c, E = remez()
    c32 = c.astype(np.float32)
    grid = np.linspace(-0.5, 0.5, 200001)
    err_exact = np.abs(_err(c32.astype(np.float64), grid)).max()
    print("minimax relative error (exact coefficients): %.3e" % E)
    print("fp32 coefficients c1..c4: %s" % " ".join("%.9g" % x for x in c32))
    print("relative error of the fp32-rounded polynomial (exact arithmetic): %.3e" % err_exact)
    try:
        import oracle
        xs = np.concatenate([np.linspace(-124.9, 0.0, 20001), np.linspace(-1, 1, 2001)]).astype(np.float32)
        got = np.array([oracle.exp2_det(float(x)) for x in xs])
        rel = np.abs(got / np.exp2(xs.astype(np.float64)) - 1.0).max()
        print("relative error of oracle.exp2_det (fp32 evaluation): %.3e" % rel)
    except Exception as e:  # the fit itself needs numpy only
        print("oracle not available: %s" % e)
    return c32, E


if __name__ == "__main__":
    main()
