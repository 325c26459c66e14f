"""Error budget of the FastMTP draft block's GPU path against the block's exact definition.

The oracle evaluates the block in float64 with no rounding at all.  The GPU path sums in fp32
and stores every value that passes between its kernels in bf16.  The fp32 sums differ from
float64 by ~1e-6 relative, so the difference between the two is the bf16 storage, and this
module bounds it before any GPU run.

One store.  Round-to-nearest bf16 (8 significant bits) leaves an error that is uniform within
half a unit in the last place.  Over a vector of roughly Gaussian values that is a relative
L2 error EPS_STORE = 1.66e-3 (2^-7 / sqrt(12), weighted by the distribution of mantissas).

One step, first order.  The block's values are projections of unit-RMS vectors by weights
N(0, std), so a projection over n inputs has RMS std * sqrt(n) and passes a relative error on
unchanged.  The stores that count are:
  - the block input and u = W_p [..] (both at the scale of u, std * sqrt(2H)) and u after the
    attention.  The attention branch adds very little: an average over hundreds of cache
    entries has RMS ~0.04, so its stores are left out;
  - the FFN input f (unit RMS), the activation and the FFN output (at the FFN output's scale);
  - u after the FFN (the state).
An error in u reaches the state directly and also through the FFN, whose linearisation has gain
J = std * sqrt(I) * J_swiglu * s (s = std * sqrt(H), J_swiglu the RMS Jacobian of
silu(g) * v at g, v ~ N(0, s^2)).  Independent errors add in quadrature.
Across steps, the previous state enters through the half of W_p that reads it, gain s, amplified
by the FFN factor and normalised by the state's RMS.

At the decoder shape (H 1280, FFN 7,168, std 0.02, K = 3) the estimate is a relative L2 error of
5.4e-3 for the state; a bf16-storage simulation on the CPU gives 5.5e-3.  The bounds are:
  - state: rel-L2 <= STATE_REL = 1e-2, the layers' bound (1.85 times the estimate), and every
    element within 6 * STATE_REL * rms(ref);
  - drafts: a logit v is w_v . hn with w_v ~ N(0, std), so an error of relative L2 e in the
    unit-RMS normalised state moves it by e * sigma_logit, sigma_logit = std * sqrt(H).  At the
    bound, e = sqrt(STATE_REL^2 + EPS_STORE^2) (one more store).  Two logits then differ by
    sqrt(2) e sigma_logit at one standard deviation.  A draft is therefore compared bit for bit
    wherever the exact top-two logits are GAP_STDS = 6 of those apart at every step.
"""
from __future__ import annotations

import math

import numpy as np

EPS_STORE = 1.66e-3
STATE_REL = 1e-2
ELEMENT_STDS = 6.0
GAP_STDS = 6.0


def swiglu_gains(s: float) -> tuple[float, float]:
    """(RMS of silu(g) * v, RMS Jacobian of it per unit perturbation of g and v) for independent
    g, v ~ N(0, s^2), by Gauss-Hermite quadrature."""
    z, w = np.polynomial.hermite_e.hermegauss(80)
    w = w / w.sum()
    g = s * z
    sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    dsilu = sig * (1.0 + g * (1.0 - sig))
    e_silu2 = float((w * silu ** 2).sum())
    e_dsilu2 = float((w * dsilu ** 2).sum())
    func = math.sqrt(e_silu2 * s * s)
    jac = math.sqrt(e_dsilu2 * s * s + e_silu2)
    return func, jac


def state_rel_estimate(H: int, I: int, K: int, std: float = 0.02) -> float:
    """First-order relative L2 error of the block's state after K steps due to bf16 storage."""
    s = std * math.sqrt(H)                     # a projection of a unit-RMS H-vector
    u0 = std * math.sqrt(2 * H)                # u = W_p [two unit-RMS halves]
    f_g, j_g = swiglu_gains(s)
    p_d = std * math.sqrt(I) * f_g             # FFN output
    j_ffn = std * math.sqrt(I) * j_g * s       # its gain for a relative error of its input
    state = math.sqrt(u0 * u0 + p_d * p_d)
    amp2 = 1.0 + j_ffn * j_ffn                 # an error in u also reaches the state through the FFN
    step2 = EPS_STORE ** 2 * (amp2 * 3 * u0 * u0 + j_ffn ** 2 + 2 * p_d ** 2 + state ** 2)
    carry2 = (s * s * amp2) / (state * state)  # previous state's error, through W_p and the FFN
    var = 0.0
    for _ in range(K):
        var = step2 + carry2 * var
    return math.sqrt(var) / state


def draft_gap(w_vocab_values: np.ndarray) -> float:
    """Smallest exact top-two logit difference at which the GPU's draft must equal the oracle's."""
    H = w_vocab_values.shape[1]
    sigma_logit = float(np.sqrt((w_vocab_values.astype(np.float64) ** 2).mean())) * math.sqrt(H)
    e = math.sqrt(STATE_REL ** 2 + EPS_STORE ** 2)
    return GAP_STDS * math.sqrt(2.0) * e * sigma_logit


def assert_state_close(got, ref, what):
    """The block's state (or a projection of it) against the exact value, within the budget."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    rms = float(np.sqrt((ref ** 2).mean()))
    worst = float(np.abs(got - ref).max()) if got.size else 0.0
    assert rel <= STATE_REL and worst <= ELEMENT_STDS * STATE_REL * rms, (
        "%s rel-L2 %.3e (bound %.1e), worst %.3e (bound %.3e)" % (what, rel, STATE_REL, worst,
                                                                   ELEMENT_STDS * STATE_REL * rms))
    return rel, worst
