"""Per-step Polar Express coefficients: greedy minimax odd quintics, computed in fp64.

[P3] "dtensor-muon 0.1.0", section "What is Muon?", names the Polar Express scheme
(arXiv 2505.16932): per-step precomputed coefficients instead of one fixed quintic.
No page prints the coefficients, so this module computes them from the method's
principle as we read it:

  * After Frobenius normalisation every singular value lies in [l_0, 1]; l_0 = 1e-3
    is the assumed lower bound (a parameter).
  * Step t uses the odd quintic p_t(x) = a x + b x^3 + c x^5 that minimises
    max_{x in [l_t, u_t]} |1 - p_t(x)| (a best uniform approximation of the constant 1).
  * If E_t is that minimal error, p_t maps [l_t, u_t] onto [1 - E_t, 1 + E_t], which is
    the next step's interval.

The minimax problem is solved with the Remez exchange: a best approximation from the
3-dimensional space span{x, x^3, x^5} equioscillates on 4 points (Chebyshev's
alternation theorem for Haar spaces on [l, u] with l > 0). The interior extrema of the
error are the roots of p'(x) = a + 3 b x^2 + 5 c x^4, a quadratic in x^2, so each
exchange finds them in closed form.

Each step's polynomial is applied at x / safety (coefficients rescaled: a/s, b/s^3, c/s^5),
safety = 1.01 by default: our reading of the scheme's safeguard against round-off. The
polynomials of the middle steps are steep at the top of their interval, so a singular value
that rounding pushes slightly past it is amplified step after step and the iteration diverges
in bf16; evaluating at x / 1.01 keeps a 1% overshoot inside the interval the next step was
designed for. With the margin, step t maps [l_t, u_t] into [q_t(l_t), 1 + E_t], which is the
next interval (q_t the rescaled polynomial, E_t the minimax error).

Parity of the GPU path never depends on these values (oracle and kernels receive the same
table). Fidelity to the published table is parity unpinned; the solver itself is pinned
by the alternation property and by the degree-1 closed form (tests/test_oracle_pins.py).

Run ``python -m oracle.polar_express`` to rewrite tests/golden/polar_express_{5,8}step.json.
"""
from __future__ import annotations

import json
import os
import sys
from typing import List, Tuple

import numpy as np

LIMIT = (15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0)   # p(1)=1, p'(1)=p''(1)=0: the limit as the interval shrinks to {1}


def _solve_reference(pts: np.ndarray) -> Tuple[np.ndarray, float]:
    """a x_i + b x_i^3 + c x_i^5 + (-1)^i E = 1 on the 4 reference points."""
    M = np.stack([pts, pts ** 3, pts ** 5, (-1.0) ** np.arange(4)], axis=1)
    sol = np.linalg.solve(M, np.ones(4))
    return sol[:3], float(sol[3])


def _critical_points(coef: np.ndarray, lo: float, hi: float) -> np.ndarray:
    a, b, c = coef
    ys = np.roots([5.0 * c, 3.0 * b, a]) if c != 0 else np.array([-a / (3.0 * b)])
    xs = [np.sqrt(y.real) for y in np.atleast_1d(ys) if abs(y.imag) < 1e-300 and lo * lo < y.real < hi * hi]
    return np.sort(np.array(xs))


def minimax_odd_quintic(lo: float, hi: float, iters: int = 100, tol: float = 1e-15):
    """Best uniform odd-quintic approximation of 1 on [lo, hi]. Returns ((a, b, c), E, reference points)."""
    if hi - lo < 1e-9 * hi:
        return LIMIT, 0.0, np.array([lo, lo, hi, hi])
    k = np.arange(4)
    pts = lo + (hi - lo) * (1.0 - np.cos(k * np.pi / 3.0)) / 2.0
    coef, E = _solve_reference(pts)
    for _ in range(iters):
        crit = _critical_points(coef, lo, hi)
        if len(crit) != 2:
            # error not yet shaped like the alternant; keep the current reference, nudge it inward
            break
        new = np.array([lo, crit[0], crit[1], hi])
        coef_new, E_new = _solve_reference(new)
        moved = np.max(np.abs(new - pts))
        pts, coef, E = new, coef_new, E_new
        if moved < tol * hi:
            break
    return tuple(float(v) for v in coef), abs(E), pts


def polar_express_table(steps: int, l0: float = 1e-3, safety: float = 1.01) -> List[Tuple[float, float, float]]:
    lo, hi = l0, 1.0
    table = []
    for _ in range(steps):
        (a, b, c), E, _ = minimax_odd_quintic(lo, hi)
        a, b, c = a / safety, b / safety ** 3, c / safety ** 5
        table.append((a, b, c))
        lo, hi = a * lo + b * lo ** 3 + c * lo ** 5, 1.0 + E
    return table


def _golden_path(steps: int) -> str:
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return os.path.join(root, "tests", "golden", f"polar_express_{steps}step.json")


def main(argv=None) -> int:
    for steps in (5, 8):
        table = polar_express_table(steps)
        doc = {
            "source": "oracle/polar_express.py: greedy per-step minimax odd quintics on [l_t, u_t], l_0=1e-3, u_0=1, "
                      "each applied at x/1.01 "
                      "(Polar Express scheme, arXiv 2505.16932, named by the dtensor-muon 0.1.0 package description, "
                      "section 'What is Muon?'; the pages print no coefficients)",
            "l0": 1e-3,
            "safety": 1.01,
            "steps": steps,
            "coeffs": [list(abc) for abc in table],
        }
        with open(_golden_path(steps), "w") as f:
            json.dump(doc, f, indent=1)
            f.write("\n")
        print(_golden_path(steps))
    return 0


if __name__ == "__main__":
    sys.exit(main())
