"""The 8-bit forward (fa_fwd_fp8) against the fp64 oracle run on the values
the E4M3 inputs stand for (the exact bytes times their per-tensor factors).

Tolerance, derived from the arithmetic: the 8-bit products are exact and are
summed in fp32, so S is accurate; what the kernel rounds is P, to E4M3 after
a 2^8 scaling (3 mantissa bits: at most 2^-4 of the value in the normal
range, at most 2^-18 absolute below it), and O, to bf16 (2^-8 of |O|).
Element by element:
    |O - O_ref| <= 2^-4 sum_k p_k |v_k| + 2^-18 sum_k |v_k| + 2^-8 |O_ref| + 1e-4
with p and v exact (the last term covers fp32 sums and exp2).  LSE does not
involve P's rounding and keeps the bf16 bound 1e-3."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h

pytestmark = pytest.mark.gpu


def run(x8, fac, scale, causal, window=0):
    q, k, v = (x8[n].to("cuda") for n in ("Q", "K", "V"))
    B, H, N, d = q.shape
    o, ob = h.guarded((B, H, N, d), torch.bfloat16)
    lse, lb = h.guarded((B, H, N), torch.float32)
    fa.fwd_fp8(q, k, v, scale, (fac["Q"], fac["K"], fac["V"]), causal, out=o,
               lse=lse, window=window)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    assert h.guards_intact(ob) and h.guards_intact(lb), "write outside O/LSE"
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    return h.np64(o), h.np64(lse)


def exact(x8, fac):
    return [inputs.e4m3_to_f64(x8[n], fac[n]) for n in ("Q", "K", "V")]


def bound(P, V, O_ref):
    """The per-element bound of the module docstring; P is [..., N, N]."""
    Va = np.abs(V)
    return (2.0 ** -4 * np.einsum("...rk,...kc->...rc", P, Va)
            + 2.0 ** -18 * Va.sum(axis=-2, keepdims=True)
            + 2.0 ** -8 * np.abs(O_ref) + 1e-4)


def check(o, lse, Q, K, V, scale, causal, window=0):
    O, L = oracle.fwd(Q, K, V, scale, causal, window=window)
    if window:
        # the oracle's probs entry point knows no window: rebuild P from LSE
        P = probs_from_lse(Q, K, scale, L, causal, window)
    else:
        P = oracle.probs(Q, K, scale, causal)
    err = np.abs(o - O)
    tol = bound(P, V, O)
    assert np.all(err <= tol), float(np.max(err - tol))
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16
    return float(err.max()), float(np.sqrt((err ** 2).mean()))


def probs_from_lse(Q, K, scale, L, causal, window):
    """p_rk = exp(scale q_r.k_k - LSE_r) on visible pairs (for the bound only;
    LSE from the oracle)."""
    N = Q.shape[-2]
    S = scale * np.einsum("...rd,...kd->...rk", Q, K)
    r = np.arange(N)[:, None]
    k = np.arange(N)[None, :]
    vis = np.ones((N, N), bool)
    if causal or window:
        vis &= k <= r
    if window:
        vis &= r - k < window
    return np.where(vis, np.exp(S - L[..., :, None]), 0.0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 127, 128, 129, 300, 513])
def test_small_ragged(N, causal):
    x8, fac = inputs.e4m3_inputs(2, 2, N, 128, seed=2000 + N)
    sc = 128 ** -0.5
    o, lse = run(x8, fac, sc, causal)
    check(o, lse, *exact(x8, fac), sc, causal)


@pytest.mark.parametrize("N,w", [(300, 16), (513, 200), (700, 129)])
def test_window(N, w):
    x8, fac = inputs.e4m3_inputs(1, 2, N, 128, seed=2100 + N + w)
    sc = 128 ** -0.5
    o, lse = run(x8, fac, sc, True, window=w)
    check(o, lse, *exact(x8, fac), sc, True, window=w)


def test_factors_enter_exactly():
    """Powers of two in the factors change no rounding: q and k factors only
    through their product, the v factor as an exact multiple of O."""
    x8, fac = inputs.e4m3_inputs(1, 2, 260, 128, seed=7)
    base = run(x8, {"Q": 1.0, "K": 1.0, "V": 1.0}, 0.05, True)
    moved = run(x8, {"Q": 4.0, "K": 0.25, "V": 1.0}, 0.05, True)
    assert np.array_equal(base[0], moved[0]) and np.array_equal(base[1], moved[1])
    twice = run(x8, {"Q": 1.0, "K": 1.0, "V": 2.0}, 0.05, True)
    assert np.array_equal(2 * base[0], twice[0]) and np.array_equal(base[1], twice[1])


@pytest.mark.parametrize("causal", [False, True])
def test_llama_shape_sampled_rows(causal):
    """4 x 32 heads, N = 4096, d = 128 at full size; sampled rows of every
    head against the oracle, with the bound built from those rows' P."""
    w = inputs.WORKLOADS["llama3_8b_fwd"]
    x8, fac = inputs.e4m3_inputs(w.B, w.H, w.N, w.d, seed=w.seed)
    o, lse = run(x8, fac, w.scale, causal)
    Q, K, V = exact(x8, fac)
    rows = inputs.sample_rows(w.B, w.H, w.N, per_head=6, seed=w.seed).numpy()
    O, L = oracle.fwd_rows(Q, K, V, w.scale, causal, rows)
    og = o.reshape(-1, w.d)[rows]
    lg = lse.reshape(-1)[rows]
    assert h.max_abs(lg, L) <= h.TOL_LSE_BF16
    Kf, Vf = K.reshape(-1, w.N, w.d), V.reshape(-1, w.N, w.d)
    Qf = Q.reshape(-1, w.d)
    for i, fr in enumerate(rows):
        bh, r = divmod(int(fr), w.N)
        s = w.scale * (Kf[bh] @ Qf[fr])
        p = np.exp(s - L[i])
        if causal:
            p[r + 1:] = 0.0
        Va = np.abs(Vf[bh])
        tol = 2.0 ** -4 * (p @ Va) + 2.0 ** -18 * Va.sum(0) + 2.0 ** -8 * np.abs(O[i]) + 1e-4
        err = np.abs(og[i] - O[i])
        assert np.all(err <= tol), (int(fr), float(np.max(err - tol)))


def test_accuracy_is_far_inside_the_bound():
    """The bound is a worst case; the typical error of the rounding of P is
    much smaller (independent roundings cancel in the sums)."""
    x8, fac = inputs.e4m3_inputs(1, 4, 1024, 128, seed=99)
    sc = 128 ** -0.5
    o, lse = run(x8, fac, sc, True)
    Q, K, V = exact(x8, fac)
    O, _ = oracle.fwd(Q, K, V, sc, True)
    rel_rms = np.linalg.norm(o - O) / np.linalg.norm(O)
    assert rel_rms <= 2e-2, rel_rms


def test_rejects_other_head_dims_and_bad_factors():
    q = torch.zeros((1, 1, 16, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError):
        fa.fwd_fp8(q, q, q, 1.0, (1.0, 1.0, 1.0))
    q = torch.zeros((1, 1, 16, 128), dtype=torch.uint8, device="cuda")
    for f in ((0.0, 1.0, 1.0), (1.0, -1.0, 1.0), (1.0, 1.0, float("nan"))):
        with pytest.raises(fa.FAError):
            fa.fwd_fp8(q, q, q, 1.0, f)
