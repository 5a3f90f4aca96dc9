"""The error budget of the kernels' weights and race quotients.

Each constant bounds the relative error of one factor over its whole input
domain; tests/weight_error_scan.cu measures each one on the GPU (all inputs of
the domain, except softmax_weight's two-argument form, which is bounded by its
parts: expf of the rounded difference, measured on every float, times
(1 + lo) with the rounding error lo of the difference, plus one fma rounding).

Top-p-only rows of the row kernel weigh an element of bin b as
w24 * 2^-24 * exp(-b/32) (w24 from ex2.approx, exp(-b/32) from a table) and race it
as fl(fl(w24 * rcp(fl(q + eps))) * 2^-24 exp(-b/32)).  Top-k rows (and every row
of the cluster kernel and of the row kernel's exact selection) weigh y as
softmax_weight(y, M) = expf(fl(y - M)) (1 + lo), sum masses in 2^-40 fixed point,
and race by IEEE division weight / fl(q + eps).
"""

NEAR = 1e-6  # the parity rule's near-tie band (relative)

U = 2.0 ** -24  # one fp32 rounding (relative)
EPS_W24 = 1.15e-7  # w24_weight over frac in [0, 1/32]
EPS_EXP_BIN = 2.0 ** -24 * (1 + 2.0 ** -10)  # the table exp(-b/32): nearest float (+ its compile-time error)
EPS_FRAC = 2.0 ** -30  # the rounding of frac = c - y (|frac| < 1/16), as a relative mass error
EPS_RCP = 1.0e-7  # rcp.approx.f32 over every normal float
EPS_EXPF = 1.55e-7  # expf over every float in [-87, 0]
LO_MAX = 87.0 * 2.0 ** -24  # the largest rounding error of y - M (|y - M| <= 87) carried as lo
EPS_SOFTMAX_WEIGHT = (1 + EPS_EXPF) * (1 + U) * (1 + LO_MAX ** 2) - 1  # expf, the fma, lo to first order


def _compose(*eps):
    r = 1.0
    for e in eps:
        r *= 1.0 + e
    return r - 1.0


def mass_error_wide() -> float:
    """An element's mass in a top-p-only row of the row kernel."""
    return _compose(EPS_W24, EPS_EXP_BIN, EPS_FRAC)


def race_error_wide() -> float:
    """An element's race score there: its mass, fl(q + eps), rcp, and two products."""
    return _compose(mass_error_wide(), U, EPS_RCP, U, U)


def mass_error_topk(n: int = 262144) -> float:
    """An element's mass in rows weighed by softmax_weight with 2^-40 fixed-point sums of up to n
    elements (as a relative error against a total S >= 1: n * 2^-41 added to each side)."""
    return EPS_SOFTMAX_WEIGHT + n * 2.0 ** -41


def race_error_topk() -> float:
    """A race score there: the weight, fl(q + eps), and the IEEE division."""
    return _compose(EPS_SOFTMAX_WEIGHT, U, U)


def topp_flip_band(eps: float, p: float) -> float:
    """Relative distance of the exact boundary mass from p * S within which masses each off by at
    most eps can change the top-p count."""
    return 2.0 * (1.0 - p) * eps / (1.0 - eps)


def race_flip_band(eps: float) -> float:
    """Relative gap of the two best race scores within which scores each off by at most eps can
    change the winner."""
    return 2.0 * eps / (1.0 - eps)
