"""Attention dropout on the CUDA path (fa_fwd_dropout, fa_bwd_dropout,
fa_dropout_mask) against the fp64 oracle with the same keep mask.

The keep decisions are integer work and are checked bit for bit: the mask
kernel's bytes against the oracle's Philox4x32-10 mask, and the decisions
inside the attention kernels through inputs that make every kept entry
visible in the output (Q = K = 0, and V or dO a shifted identity, so that
each output element is a single probability times the keep factor).  The
floating-point outputs are held to the library's tolerances, with the bf16
O bound multiplied by the keep factor 256/(256 - t): every term of O is
scaled by it, and so is every rounding error."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def keep_factor(p):
    t = oracle.dropout_threshold(p)
    return 256.0 / (256 - t)


def visible(N, causal, window):
    r = np.arange(N)[:, None]
    k = np.arange(N)[None, :]
    v = np.ones((N, N), bool)
    if causal or window:
        v &= k <= r
    if window:
        v &= r - k < window
    return v


# ------------------------------------------------------- the mask, bit-exact
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 5), (2, 3, 130), (1, 2, 257)])
@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_mask_matches_oracle_bit_for_bit(B, H, N, p):
    for seed in (0, 12345, 0xDEADBEEF_CAFEF00D):
        got = fa.dropout_mask(B, H, N, p, seed).cpu().numpy()
        ref = oracle.dropout_keep(B, H, N, p, seed)
        assert np.array_equal(got, ref.astype(np.uint8)), (p, seed)


def test_mask_many_heads():
    """Heads past the grid's z extent loop; the head index is part of the
    counter."""
    got = fa.dropout_mask(4, 100, 12, 0.3, 77).cpu().numpy()
    ref = oracle.dropout_keep(4, 100, 12, 0.3, 77)
    assert np.array_equal(got, ref.astype(np.uint8))


# ------------------------------- the keep decisions inside the attention kernels
def forward_keep_pattern(B, H, N, d, p, seed, causal, window, dtype):
    """With Q = K = 0 every visible key has probability 1/n_visible; with
    V[k, c] = [k == c0 + c], O[r, c] is that probability times M[r, c0 + c],
    so the nonzero pattern of O is the kernel's keep mask on visible pairs."""
    z = torch.zeros((B, H, N, d), dtype=DT[dtype], device="cuda")
    pat = np.zeros((B, H, N, N), bool)
    for c0 in range(0, N, d):
        n = min(d, N - c0)
        v = torch.zeros((B, H, N, d), dtype=DT[dtype], device="cuda")
        idx = torch.arange(n, device="cuda")
        v[:, :, c0 + idx, idx] = 1
        o, _ = fa.fwd(z, z, v, 1.0, causal, window=window, dropout_p=p, seed=seed)
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        pat[:, :, :, c0:c0 + n] = (o[..., :n] != 0).cpu().numpy()
    return pat


def backward_keep_pattern(B, H, N, d, p, seed, causal, window, dtype):
    """With Q = K = 0 and dO[r, c] = [r == r0 + c], dV[k, c] = M P[r0 + c, k]:
    the nonzero pattern of dV is the backward's regenerated keep mask."""
    z = torch.zeros((B, H, N, d), dtype=DT[dtype], device="cuda")
    v = torch.randn((B, H, N, d), generator=torch.Generator().manual_seed(5)).to(
        "cuda", DT[dtype])
    o, lse = fa.fwd(z, z, v, 1.0, causal, window=window, dropout_p=p, seed=seed)
    pat = np.zeros((B, H, N, N), bool)
    for r0 in range(0, N, d):
        n = min(d, N - r0)
        do = torch.zeros((B, H, N, d), dtype=DT[dtype], device="cuda")
        idx = torch.arange(n, device="cuda")
        do[:, :, r0 + idx, idx] = 1
        _, _, dv = fa.bwd(z, z, v, o, do, lse, 1.0, causal, window=window,
                          dropout_p=p, seed=seed)
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        pat[:, :, r0:r0 + n, :] = (dv[..., :n] != 0).transpose(2, 3).cpu().numpy()
    return pat


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,causal,window", [(128, False, 0), (300, False, 0),
                                             (300, True, 0), (260, True, 100)])
def test_forward_applies_the_oracle_mask(N, causal, window, d, dtype):
    B, H, p, seed = 1, 2, 0.5, 2024
    got = forward_keep_pattern(B, H, N, d, p, seed, causal, window, dtype)
    ref = oracle.dropout_keep(B, H, N, p, seed).astype(bool) & visible(N, causal, window)
    assert np.array_equal(got, ref), int((got != ref).sum())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N,causal,window", [(128, False, 0), (300, False, 0),
                                             (300, True, 0), (260, True, 100)])
def test_backward_regenerates_the_oracle_mask(N, causal, window, d, dtype):
    B, H, p, seed = 1, 2, 0.3, 99
    got = backward_keep_pattern(B, H, N, d, p, seed, causal, window, dtype)
    ref = oracle.dropout_keep(B, H, N, p, seed).astype(bool) & visible(N, causal, window)
    assert np.array_equal(got, ref), int((got != ref).sum())


# ------------------------------------------------- parity of the outputs
def run_fwd(x, scale, causal, window, p, seed):
    q, k, v = (x[n].to("cuda") for n in ("Q", "K", "V"))
    B, H, N, d = q.shape
    o, ob = h.guarded((B, H, N, d), q.dtype)
    lse, lb = h.guarded((B, H, N), torch.float32)
    fa.fwd(q, k, v, scale, causal, out=o, lse=lse, window=window, dropout_p=p,
           seed=seed)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    assert h.guards_intact(ob) and h.guards_intact(lb), "write outside O/LSE"
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    return h.np64(o), h.np64(lse)


def run_fwd_bwd(x, scale, causal, window, p, seed):
    q, k, v, do = (x[n].to("cuda") for n in ("Q", "K", "V", "dO"))
    B, H, N, d = q.shape
    o, lse = fa.fwd(q, k, v, scale, causal, window=window, dropout_p=p, seed=seed)
    outs = [h.guarded((B, H, N, d), q.dtype) for _ in range(3)]
    ws = fa.workspace(B, H, N, d)
    ws.fill_(0xFF)
    fa.bwd(q, k, v, o, do, lse, scale, causal, dq=outs[0][0], dk=outs[1][0],
           dv=outs[2][0], ws=ws, window=window, dropout_p=p, seed=seed)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    for t, b in outs:
        assert h.guards_intact(b), "write outside a gradient tensor"
        assert torch.isfinite(t.float()).all()
    return tuple(h.np64(t) for t, _ in outs)


def f64(x, names):
    return [inputs.to_f64(x[n]) for n in names]


def check_grads(got, ref):
    errs = [h.rel_l2(g, r) for g, r in zip(got, ref)]
    assert max(errs) <= h.TOL_GRAD_REL, dict(zip(("dQ", "dK", "dV"), errs))
    return errs


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,causal,window", [(7, False, 0), (130, True, 0),
                                             (300, False, 0), (300, True, 0),
                                             (513, True, 200)])
def test_bf16_forward_parity(N, causal, window, d, p):
    x = h.seeded(2, 2, N, d, seed=1200 + N + d, dtype="bf16")
    sc = d ** -0.5
    o, lse = run_fwd(x, sc, causal, window, p, 31 + N)
    O, L = oracle.fwd(*f64(x, ("Q", "K", "V")), sc, causal, window=window,
                      dropout_p=p, seed=31 + N)
    assert h.max_abs(o, O) <= h.TOL_O_BF16 * keep_factor(p)
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,causal,window", [(7, False, 0), (130, True, 0),
                                             (300, False, 0), (300, True, 0),
                                             (513, True, 200)])
def test_bf16_backward_parity(N, causal, window, d, p):
    x = h.seeded(1, 2, N, d, seed=1300 + N + d, dtype="bf16", with_dO=True)
    sc = d ** -0.5
    got = run_fwd_bwd(x, sc, causal, window, p, 77 + N)
    dQ, dK, dV, _ = oracle.bwd(*f64(x, ("Q", "K", "V", "dO")), sc, causal,
                               window=window, dropout_p=p, seed=77 + N)
    check_grads(got, (dQ, dK, dV))


@pytest.mark.parametrize("N,causal,window", [(33, False, 0), (200, True, 0),
                                             (200, True, 50)])
def test_f32_forward_backward_parity(N, causal, window):
    x = h.seeded(2, 1, N, 64, seed=1400 + N, dtype="f32", with_dO=True)
    p, seed, sc = 0.25, 4242, 0.125
    o, lse = run_fwd(x, sc, causal, window, p, seed)
    O, L = oracle.fwd(*f64(x, ("Q", "K", "V")), sc, causal, window=window,
                      dropout_p=p, seed=seed)
    assert h.max_abs(o, O) <= h.TOL_F32 * keep_factor(p)
    assert h.max_abs(lse, L) <= h.TOL_F32
    got = run_fwd_bwd(x, sc, causal, window, p, seed)
    dQ, dK, dV, _ = oracle.bwd(*f64(x, ("Q", "K", "V", "dO")), sc, causal,
                               window=window, dropout_p=p, seed=seed)
    errs = check_grads(got, (dQ, dK, dV))
    assert max(errs) < 1e-5


def test_training_workload_sampled_heads():
    """The training step's shape (8 x 16 heads, N = 2048, d = 128, causal) with
    dropout 0.1 at full size: sampled forward rows of every head, and the
    gradients of the first two heads in full (their counter words are 0 and
    1 both in the full batch and in the oracle's two-head copy)."""
    w = inputs.WORKLOADS["train_fwd_bwd"]
    x = inputs.workload_inputs(w)
    p, seed = 0.1, 0x5EED
    o, lse = run_fwd(x, w.scale, True, 0, p, seed)
    rows = inputs.sample_rows(w.B, w.H, w.N, per_head=8, seed=w.seed).numpy()
    Q, K, V = f64(x, ("Q", "K", "V"))
    O, L = oracle.fwd_rows(Q, K, V, w.scale, True, rows, dropout_p=p, seed=seed)
    assert h.max_abs(o.reshape(-1, w.d)[rows], O) <= h.TOL_O_BF16 * keep_factor(p)
    assert h.max_abs(lse.reshape(-1)[rows], L) <= h.TOL_LSE_BF16
    dq, dk, dv = run_fwd_bwd(x, w.scale, True, 0, p, seed)
    sub = {n: x[n][0:1, 0:2] for n in ("Q", "K", "V", "dO")}
    dQ, dK, dV, _ = oracle.bwd(*f64(sub, ("Q", "K", "V", "dO")), w.scale, True,
                               dropout_p=p, seed=seed)
    check_grads((dq[0:1, 0:2], dk[0:1, 0:2], dv[0:1, 0:2]), (dQ, dK, dV))


def test_long_context_sampled():
    """Causal N = 8192 with dropout 0.1, sampled rows of every head."""
    w = inputs.WORKLOADS["long_ctx_8k"]
    x = inputs.workload_inputs(w, with_dO=False)
    p, seed = 0.1, 8192
    o, lse = run_fwd(x, w.scale, True, 0, p, seed)
    rows = inputs.sample_rows(w.B, w.H, w.N, per_head=12, seed=w.seed).numpy()
    O, L = oracle.fwd_rows(*f64(x, ("Q", "K", "V")), w.scale, True, rows,
                           dropout_p=p, seed=seed)
    assert h.max_abs(o.reshape(-1, w.d)[rows], O) <= h.TOL_O_BF16 * keep_factor(p)
    assert h.max_abs(lse.reshape(-1)[rows], L) <= h.TOL_LSE_BF16


# ---------------------------------------------------------------- edge cases
def test_threshold_zero_is_the_plain_computation():
    """A dropout_p that rounds to t = 0 keeps everything: the same kernels
    and the same bits as without dropout."""
    x = h.seeded(1, 2, 300, 128, seed=5, dtype="bf16", with_dO=True)
    a = run_fwd(x, 0.1, True, 0, 0.001, 1)
    b = run_fwd(x, 0.1, True, 0, 0.0, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_same_seed_same_bits_other_seed_other_output():
    x = h.seeded(1, 2, 400, 64, seed=6, dtype="bf16", with_dO=True)
    a = run_fwd(x, 0.125, False, 0, 0.2, 10)
    b = run_fwd(x, 0.125, False, 0, 0.2, 10)
    c = run_fwd(x, 0.125, False, 0, 0.2, 11)
    assert np.array_equal(a[0], b[0])
    assert not np.array_equal(a[0], c[0])
    assert np.array_equal(a[1], c[1])  # LSE does not depend on the mask
    ga = run_fwd_bwd(x, 0.125, False, 0, 0.2, 10)
    gb = run_fwd_bwd(x, 0.125, False, 0, 0.2, 10)
    assert np.array_equal(ga[1], gb[1]) and np.array_equal(ga[2], gb[2])


def test_lse_is_the_undropped_one():
    x = h.seeded(2, 2, 333, 128, seed=8, dtype="bf16")
    _, l_drop = run_fwd(x, 0.09, True, 0, 0.6, 3)
    _, l_plain = run_fwd(x, 0.09, True, 0, 0.0, 0)
    assert h.max_abs(l_drop, l_plain) <= 1e-6


def test_rejected_probabilities():
    q = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    for p in (-0.1, 1.0, 0.999, float("nan"), float("inf")):
        with pytest.raises(fa.FAError):
            fa.fwd(q, q, q, 1.0, dropout_p=p, seed=1)
