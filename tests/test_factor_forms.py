"""The two forms of the A/P epilogue's decay factor, emulated in fp32 on the CPU.

Below the diagonal an entry of A is beta_i e^{G_i - G_j} (k_i . k_j) / (|k_i| |k_j|). The
kernel evaluates its factor either as 2^{x_i - Gp_j} (one ex2 per entry) or, in chunks whose
total log2-decay is at least -100, as 2^{x_i} * 2^{-Gp_j} (row and column factors). These
checks pin the range argument behind that bound: at and beyond it the column factors stay
finite, the factored entries agree with the per-entry form to fp32 rounding, and masked
entries above the diagonal never turn into NaN. The error bounds come from the fp32
rounding of the exponents (about 2^-24 of |G| each, measured here at up to 6e-7 within the
bound and 1.3e-5 at a decay of 2^-2000), far below the fp16 rounding (2^-11) of the
operands built from A.
"""
import numpy as np

BOUND = -100.0          # the kernel's kFactoredMinLog2Decay
RK_MAX = 1.0 / np.sqrt(1e-6)  # 1/|k| is at most 1/sqrt(eps) with the norm epsilon


def _chunk(rng, total_log2):
    """Chunk-local inclusive log2-decays G (64 tokens, non-increasing, G[63] = total),
    betas, inverse key norms (some at the maximum) and raw dot products k_i . k_j."""
    steps = rng.random(64)
    g = -np.cumsum(steps / steps.sum() * -total_log2)
    beta = rng.random(64).astype(np.float32)
    rk = np.exp(rng.uniform(np.log(0.05), np.log(RK_MAX), 64))
    rk[:4] = RK_MAX
    kk = (rng.standard_normal((64, 64)) * 30).astype(np.float32)
    return g.astype(np.float32), beta, rk.astype(np.float32), kk


def _forms(g, beta, rk, kk):
    f32 = np.float32
    x = (g + np.log2(beta * rk)).astype(f32)          # row exponents
    gp = (g - np.log2(rk)).astype(f32)                # column exponents
    with np.errstate(over="ignore", invalid="ignore"):
        direct = kk * np.exp2((x[:, None] - gp[None, :]).astype(f32)).astype(f32)
        col = np.exp2(-gp).astype(f32)
        row = np.exp2(x).astype(f32)
        factored = (kk * row[:, None]).astype(f32) * col[None, :]
    lower = np.tril(np.ones((64, 64), dtype=bool), -1)
    with np.errstate(over="ignore", invalid="ignore"):  # above the diagonal: not compared
        truth = (beta.astype(np.float64)[:, None] * rk.astype(np.float64)[:, None]
                 * rk.astype(np.float64)[None, :] * kk.astype(np.float64)
                 * np.exp2(g.astype(np.float64)[:, None] - g.astype(np.float64)[None, :]))
    return direct, factored, col, lower, truth


def test_factored_form_is_finite_and_accurate_down_to_the_bound():
    rng = np.random.default_rng(0)
    for total in (-1.0, -30.0, -74.0, -99.0, BOUND):
        g, beta, rk, kk = _chunk(rng, total)
        direct, factored, col, lower, truth = _forms(g, beta, rk, kk)
        assert np.isfinite(col).all() and col.max() < 2.0 ** 110
        masked = np.where(lower, factored, 0.0)
        assert not np.isnan(factored).any()          # inf above the diagonal at most
        assert np.isfinite(masked).all()
        scale = np.abs(truth[lower]).max()
        err_f = np.abs(masked[lower] - truth[lower]).max() / scale
        err_d = np.abs(np.where(lower, direct, 0.0)[lower] - truth[lower]).max() / scale
        assert err_f < 2e-6 and err_d < 2e-6, (total, err_f, err_d)


def test_per_entry_form_covers_any_decay():
    """Past the bound the kernel keeps one ex2 per entry: its exponent is never above 0
    below the diagonal (before the row's beta and norms), so it stays finite however
    strong the decay."""
    rng = np.random.default_rng(1)
    for total in (-150.0, -400.0, -2000.0):
        g, beta, rk, kk = _chunk(rng, total)
        direct, _, _, lower, truth = _forms(g, beta, rk, kk)
        vals = np.where(lower, direct, 0.0)
        assert np.isfinite(vals).all()
        scale = max(np.abs(truth[lower]).max(), 1e-30)
        assert np.abs(vals[lower] - truth[lower]).max() / scale < 5e-5
