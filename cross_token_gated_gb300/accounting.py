"""Work accounting for the gate-aggregation path: the paper's analytical counts and
the algorithmic flops / bytes the benchmark divides by.

Paper conventions ("TANGO: Token-Aggregated Nonlinear Gating Operators for Natural
and Formal Language Modeling"):
  * parameters outside the tied embedding (sec. 2.3 "Parameter matching", Table 1):
    W_q, W_k (d x d), W_g, W_v (d x F), W_o (F x d), the block and the final RMSNorm
    gains, one temperature and one null bias per head;
  * analytical forward MACs (sec. 3 "Compute accounting"; sec. 4.2 Table 5;
    sec. 6.1): learned projections, token pairs and the vocabulary projection, with
    every one of the T^2 token pairs counted at (F + d) MACs, for R applications.

Build conventions (what the benchmark's roofline numbers mean):
  * flops count a multiply-add as 2 and only CAUSAL pairs j <= i;
  * bytes count each operand read once and each output written once.
"""
from __future__ import annotations


def paper_block_params(d: int, F: int, H: int) -> int:
    """Non-embedding parameters of one TANGO/WANGO block plus the final RMSNorm."""
    return 2 * d * d + 3 * d * F + 2 * d + 2 * H


def paper_macs_tango(T: int, d: int, F: int, vocab: int, R: int = 4) -> int:
    """Analytical forward MACs of the R-application TANGO model on one sequence."""
    return R * (T * (2 * d * d + 3 * d * F) + T * T * (F + d)) + T * d * vocab


def paper_macs_wango_estimate(T: int, d: int, F: int, vocab: int, W: int, H: int,
                              R: int = 4, C: int = 64) -> float:
    """An estimate of the WANGO count: projections; (W + C) pairs per token at
    (F + d) MACs, as a blockwise evaluation with blocks of C = 64 positions touches
    (sec. 2.2); and 4 * d_h * F MACs per token for the feature-map state (update and
    read-out of S).

    The pages do not spell out their WANGO accounting; this reading reproduces the
    printed 1.90T (T = 8192) and 52.91B (T = 256) to about 0.1 %, not exactly."""
    d_h = d // H
    return (R * (T * (2 * d * d + 3 * d * F) + T * (W + C) * (F + d) + 4 * T * d_h * F)
            + T * d * vocab)


# ------------------------------------------------------------------ build units

def causal_pairs(T: int) -> int:
    return T * (T + 1) // 2


def window_pairs(T: int, W: int) -> int:
    """sum_i min(i + 1, W) over i < T."""
    if W >= T:
        return causal_pairs(T)
    return W * (W + 1) // 2 + (T - W) * W


def tango_agg_flops(B: int, T: int, dqk: int, m: int) -> int:
    """Scores (dqk MACs summed over heads) + gate aggregation (m MACs) per causal pair."""
    return 2 * B * causal_pairs(T) * (dqk + m)


def wango_agg_flops(B: int, T: int, dqk: int, m: int, H: int, W: int) -> int:
    """Window pairs as in TANGO, plus for every destination with a non-empty older
    prefix one read-out phi(q)^T [S | z] and for every source leaving the window one
    update of S and z (d_h * m + dqk MACs each)."""
    d_h = dqk // H
    n_old = max(0, T - W)
    return 2 * B * (window_pairs(T, W) * (dqk + m) + 2 * n_old * (d_h * m + dqk))


def agg_bytes(B: int, T: int, dqk: int, m: int, elem: int = 2) -> int:
    """q, k, g, v read once and u written once."""
    return B * T * (2 * dqk + 3 * m) * elem


def proj_flops(B: int, T: int, d: int, dqk: int, m: int) -> int:
    return 2 * B * T * d * (2 * dqk + 2 * m)


def out_flops(B: int, T: int, d: int, m: int) -> int:
    return 2 * B * T * m * d


def block_flops(B: int, T: int, d: int, dqk: int, m: int, mode: int = 0, H: int = 2,
                W: int = 1) -> int:
    agg = tango_agg_flops(B, T, dqk, m) if mode == 0 else wango_agg_flops(B, T, dqk, m, H, W)
    return proj_flops(B, T, d, dqk, m) + agg + out_flops(B, T, d, m)


def logits_flops(B: int, T: int, d: int, vocab: int) -> int:
    """The tied-embedding logits x E^T of the language model (sec. 2.3)."""
    return 2 * B * T * d * vocab


def model_flops(B: int, T: int, d: int, dqk: int, m: int, vocab: int, n_apps: int, mode: int = 0,
                H: int = 2, W: int = 1) -> int:
    """n_apps block applications (eq. 11) and the logits; the embedding lookup and the
    RMSNorms are not counted."""
    return n_apps * block_flops(B, T, d, dqk, m, mode, H, W) + logits_flops(B, T, d, vocab)


def tango_bwd_flops(B: int, T: int, dqk: int, m: int) -> int:
    """Gradients of the TANGO aggregation per causal pair: the gate gradient
    sum_i alpha_ij dgbar_i and the weight gradient dgbar_i . g_j (m MACs each), the score
    and its two gradients into qhat and khat (dqk MACs each).  The recomputed forward is
    not counted (a training step may keep gbar and the denominators instead)."""
    return 2 * B * causal_pairs(T) * (2 * m + 3 * dqk)


def wango_bwd_flops(B: int, T: int, dqk: int, m: int, H: int, W: int) -> int:
    """Gradients of the WANGO aggregation at its linear cost: window pairs as in TANGO,
    and per token with an older prefix five d_h x m contractions against the running
    sums (the gate gradient through the reverse sum of phi(q~) dgbar^T and its update,
    the feature-map gradients S dgbar and R g, and the forward sum's update)."""
    d_h = dqk // H
    n_old = max(0, T - W)
    return 2 * B * (window_pairs(T, W) * (2 * m + 3 * dqk) + 5 * n_old * (d_h * m + dqk))


def agg_bwd_bytes(B: int, T: int, dqk: int, m: int, elem: int = 2) -> int:
    """q, k, g, v and dout read once; dq, dk, dg and dv written once."""
    return B * T * (4 * dqk + 5 * m) * elem


def decode_bytes(B: int, dqk: int, m: int, H: int, W: int, elem: int = 2, fold: int = 8) -> float:
    """One WANGO decode step, on average: the ring of W gate vectors read, the f32 state
    S read, S written once per `fold` steps (sources enter S in groups of `fold`), and
    this token's g, v read and u written (sec. 2.2 eq. 10 taken one token at a time); the
    q/k-sized terms are negligible and not counted."""
    d_h = dqk // H
    return B * (W * m * elem + d_h * m * 4 * (1 + 1 / fold) + 3 * m * elem)
