"""Head dimension 256 against the fp64 oracle: the tensor-core bf16 forward
(one query block per work item, S double-buffered in TMEM), the tensor-core
bf16 backward (one half of d per work item, 64-query blocks, V in TMEM), and
the fp32 path, with the library's tolerances (bf16 O <= 1e-2, LSE <= 1e-3,
gradients relative L2 <= 1e-2, fp32 <= 1e-5)."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h

pytestmark = pytest.mark.gpu


def run_fwd(x, scale, causal, window=0):
    q, k, v = (x[n].to("cuda") for n in ("Q", "K", "V"))
    B, H, N, d = q.shape
    o, ob = h.guarded((B, H, N, d), q.dtype)
    lse, lb = h.guarded((B, H, N), torch.float32)
    fa.fwd(q, k, v, scale, causal, out=o, lse=lse, window=window)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    assert h.guards_intact(ob) and h.guards_intact(lb), "write outside O/LSE"
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    return h.np64(o), h.np64(lse)


def run_fwd_bwd(x, scale, causal, window=0):
    q, k, v, do = (x[n].to("cuda") for n in ("Q", "K", "V", "dO"))
    B, H, N, d = q.shape
    o, lse = fa.fwd(q, k, v, scale, causal, window=window)
    outs = [h.guarded((B, H, N, d), q.dtype) for _ in range(3)]
    ws = fa.workspace(B, H, N, d)
    ws.fill_(0xFF)
    fa.bwd(q, k, v, o, do, lse, scale, causal, dq=outs[0][0], dk=outs[1][0],
           dv=outs[2][0], ws=ws, window=window)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    for t, b in outs:
        assert h.guards_intact(b), "write outside a gradient tensor"
        assert torch.isfinite(t.float()).all()
    return tuple(h.np64(t) for t, _ in outs)


def f64(x, names):
    return [inputs.to_f64(x[n]) for n in names]


def check_grads(got, ref, tol=h.TOL_GRAD_REL):
    errs = [h.rel_l2(g, r) for g, r in zip(got, ref)]
    assert max(errs) <= tol, dict(zip(("dQ", "dK", "dV"), errs))
    return errs


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 127, 128, 129, 255, 300, 513])
def test_bf16_forward_small_ragged(N, causal):
    x = h.seeded(2, 2, N, 256, seed=3000 + N)
    sc = 256 ** -0.5
    o, lse = run_fwd(x, sc, causal)
    O, L = oracle.fwd(*f64(x, ("Q", "K", "V")), sc, causal)
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("N,w", [(300, 16), (513, 200), (700, 129), (1000, 1)])
def test_bf16_forward_window(N, w):
    x = h.seeded(1, 2, N, 256, seed=3100 + N + w)
    if w < 16:  # a window of a few keys copies rows of V (see the window tests)
        x["V"] = (x["V"].float() * 0.25).to(torch.bfloat16)
    sc = 256 ** -0.5
    o, lse = run_fwd(x, sc, True, window=w)
    O, L = oracle.fwd(*f64(x, ("Q", "K", "V")), sc, True, window=w)
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("N,w", [(300, 16), (520, 100)])
def test_window_row_whose_first_visible_key_is_in_a_later_block(N, w):
    """As the d <= 128 test of the same name: rows that see nothing in the
    first key block of their window, with all scaled scores near -128, so
    that rebasing from the placeholder reference would overflow."""
    x, sc = h.late_first_key_inputs(N, 256, seed=3700 + N + w)
    o, lse = run_fwd(x, sc, True, window=w)
    O, L = oracle.fwd(*f64(x, ("Q", "K", "V")), sc, window=w)
    assert L.max() < -40.0
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


def test_later_block_holds_the_max():
    """The largest scores of every row sit in the last key block ("FlashAttention
    from scratch" test recipe, as at d = 128), so every row rescales there and
    both column halves of a row must agree on the maximum.  The 1e-2 bound on
    O assumes |O| < 2 (bf16 output rounding); the recipe keeps it there."""
    x = h.seeded(1, 2, 640, 256, seed=3200)
    k = x["K"].float()
    k[:, :, -100:] *= 3.0
    x["K"] = k.to(torch.bfloat16)
    # at d = 256 the raised keys dominate more than at d = 128: V / 4 keeps
    # |O| below 2 (the window tests' treatment of peaked rows)
    x["V"] = (x["V"].float() * 0.25).to(torch.bfloat16)
    sc = 256 ** -0.5
    o, lse = run_fwd(x, sc, False)
    O, L = oracle.fwd(*f64(x, ("Q", "K", "V")), sc, False)
    assert np.abs(O).max() < 2.0
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_forward_full_size_sampled(causal):
    w = inputs.WORKLOADS["d256_fwd"]
    x = inputs.workload_inputs(w, with_dO=False)
    o, lse = run_fwd(x, w.scale, causal)
    rows = inputs.sample_rows(w.B, w.H, w.N, per_head=24, seed=w.seed).numpy()
    O, L = oracle.fwd_rows(*f64(x, ("Q", "K", "V")), w.scale, causal, rows)
    assert h.max_abs(o.reshape(-1, w.d)[rows], O) <= h.TOL_O_BF16
    assert h.max_abs(lse.reshape(-1)[rows], L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 63, 64, 65, 127, 128, 129, 255, 300, 513])
def test_bf16_backward_small(N, causal):
    x = h.seeded(1, 2, N, 256, seed=3300 + N, with_dO=True)
    sc = 256 ** -0.5
    got = run_fwd_bwd(x, sc, causal)
    dQ, dK, dV, _ = oracle.bwd(*f64(x, ("Q", "K", "V", "dO")), sc, causal)
    check_grads(got, (dQ, dK, dV))


@pytest.mark.parametrize("N,w", [(500, 150), (300, 1), (300, 64), (513, 129), (700, 300)])
def test_bf16_backward_window(N, w):
    x = h.seeded(1, 2, N, 256, seed=3400 + N + w, with_dO=True)
    sc = 256 ** -0.5
    got = run_fwd_bwd(x, sc, True, window=w)
    dQ, dK, dV, _ = oracle.bwd(*f64(x, ("Q", "K", "V", "dO")), sc, True, window=w)
    check_grads(got, (dQ, dK, dV))


def test_bf16_backward_multi_head_batch():
    """Several heads and batches (items of different heads and both halves
    of d interleaved on the CTAs), ragged N."""
    x = h.seeded(2, 3, 390, 256, seed=3450, with_dO=True)
    sc = 256 ** -0.5
    got = run_fwd_bwd(x, sc, True)
    dQ, dK, dV, _ = oracle.bwd(*f64(x, ("Q", "K", "V", "dO")), sc, True)
    check_grads(got, (dQ, dK, dV))


def test_bf16_backward_dk_dv_repeat_bit_identically():
    """dK and dV accumulate on chip without atomics: any difference between
    two runs is a race.  (dQ is summed with atomics, so only its values are
    compared, within the gradient tolerance.)"""
    x = h.seeded(2, 8, 1000, 256, seed=3460, with_dO=True)
    a = run_fwd_bwd(x, 0.0625, True)
    b = run_fwd_bwd(x, 0.0625, True)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert h.rel_l2(a[0], b[0]) < 1e-3


def test_training_shape_sampled_heads():
    """4 x 16 heads, N = 2048, d = 256, causal: two heads in full."""
    w = inputs.WORKLOADS["d256_train"]
    x = inputs.workload_inputs(w)
    dq, dk, dv = run_fwd_bwd(x, w.scale, True)
    g = np.random.default_rng(w.seed)
    for bh in sorted(g.choice(w.B * w.H, size=2, replace=False).tolist()):
        b, hh = divmod(bh, w.H)
        sub = {n: x[n][b:b + 1, hh:hh + 1] for n in ("Q", "K", "V", "dO")}
        dQ, dK, dV, _ = oracle.bwd(*f64(sub, ("Q", "K", "V", "dO")), w.scale, True)
        check_grads((dq[b:b + 1, hh:hh + 1], dk[b:b + 1, hh:hh + 1],
                     dv[b:b + 1, hh:hh + 1]), (dQ, dK, dV))


@pytest.mark.parametrize("causal", [False, True])
def test_f32(causal):
    x = h.seeded(1, 2, 200, 256, seed=3500, dtype="f32", with_dO=True)
    sc = 256 ** -0.5
    o, lse = run_fwd(x, sc, causal)
    Q, K, V, dO = f64(x, ("Q", "K", "V", "dO"))
    O, L = oracle.fwd(Q, K, V, sc, causal)
    assert h.max_abs(o, O) <= h.TOL_F32 and h.max_abs(lse, L) <= h.TOL_F32
    got = run_fwd_bwd(x, sc, causal)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, causal)
    errs = check_grads(got, (dQ, dK, dV))
    assert max(errs) < 1e-5


@pytest.mark.parametrize("N,causal,window", [(300, False, 0), (513, True, 0), (700, True, 200)])
def test_dropout(N, causal, window):
    """Dropout at d = 256: the keep decisions of the forward and of the
    backward (both tensor-core kernels, Philox per 4 x 4 patch) are the
    oracle's; bf16 O bound times the keep factor."""
    x = h.seeded(1, 2, N, 256, seed=3700 + N, with_dO=True)
    sc, p, seed = 256 ** -0.5, 0.2, 99 + N
    q, k, v, do = (x[n].to("cuda") for n in ("Q", "K", "V", "dO"))
    o, lse = fa.fwd(q, k, v, sc, causal, window=window, dropout_p=p, seed=seed)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, sc, causal, window=window, dropout_p=p,
                        seed=seed)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    Q, K, V, dO = f64(x, ("Q", "K", "V", "dO"))
    O, L = oracle.fwd(Q, K, V, sc, causal, window=window, dropout_p=p, seed=seed)
    keep_factor = 256.0 / (256 - oracle.dropout_threshold(p))
    assert h.max_abs(h.np64(o), O) <= h.TOL_O_BF16 * keep_factor
    assert h.max_abs(h.np64(lse), L) <= h.TOL_LSE_BF16
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, causal, window=window, dropout_p=p,
                               seed=seed)
    check_grads((h.np64(dq), h.np64(dk), h.np64(dv)), (dQ, dK, dV))


def test_dropout_forward_applies_the_oracle_mask():
    """Q = K = 0 and V a shifted identity expose the d = 256 forward's keep
    decisions bit for bit (as in the d <= 128 mask tests)."""
    B, H, N, d, p, seed = 1, 2, 384, 256, 0.5, 7
    z = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    got = np.zeros((B, H, N, N), bool)
    for c0 in range(0, N, d):
        n = min(d, N - c0)
        v.zero_()
        idx = torch.arange(n, device="cuda")
        v[:, :, c0 + idx, idx] = 1
        o, _ = fa.fwd(z, z, v, 1.0, False, dropout_p=p, seed=seed)
        torch.cuda.synchronize()
        got[:, :, :, c0:c0 + n] = (o[..., :n] != 0).cpu().numpy()
    ref = oracle.dropout_keep(B, H, N, p, seed).astype(bool)
    assert np.array_equal(got, ref), int((got != ref).sum())


def test_repeated_runs_are_bit_identical():
    """The forward has no atomics: any difference between runs is a race (a
    wait that let a read overtake the tensor core).  Many items per CTA, many
    key blocks per row."""
    x = h.seeded(2, 16, 1024, 256, seed=3600)
    q, k, v = (x[n].to("cuda") for n in ("Q", "K", "V"))
    ref = None
    for _ in range(4):
        o, lse = fa.fwd(q, k, v, 0.0625, False)
        torch.cuda.synchronize()
        cur = (o.clone(), lse.clone())
        if ref is None:
            ref = cur
        else:
            assert torch.equal(ref[0], cur[0]) and torch.equal(ref[1], cur[1])
    O, L = oracle.fwd_rows(*f64(x, ("Q", "K", "V")), 0.0625, False,
                           inputs.sample_rows(2, 16, 1024, per_head=32, seed=1).numpy())
    rows = inputs.sample_rows(2, 16, 1024, per_head=32, seed=1).numpy()
    assert h.max_abs(h.np64(ref[0]).reshape(-1, 256)[rows], O) <= h.TOL_O_BF16
