"""Backward parity of the CUDA path (through the C ABI) against the fp64
oracle's closed-form gradients on the same seeded inputs: dQ, dK and dV of the
scalar <dO, O>, relative L2 error <= 1e-2, for small ragged shapes in full and
for the training workload (8 x 16 heads, N = 2048, d = 128, causal) on
sampled heads."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h

pytestmark = pytest.mark.gpu


def run_fwd_bwd(x, scale, causal, window=0):
    q, k, v, do = (x[n].to("cuda") for n in ("Q", "K", "V", "dO"))
    B, H, N, d = q.shape
    o, lse = fa.fwd(q, k, v, scale, causal, window=window)
    dq, dqb = h.guarded((B, H, N, d), q.dtype)
    dk, dkb = h.guarded((B, H, N, d), q.dtype)
    dv, dvb = h.guarded((B, H, N, d), q.dtype)
    ws = fa.workspace(B, H, N, d)
    ws.fill_(0xFF)  # the workspace's entry contents must not matter
    fa.bwd(q, k, v, o, do, lse, scale, causal, dq=dq, dk=dk, dv=dv, ws=ws,
           window=window)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    for t, b in ((dq, dqb), (dk, dkb), (dv, dvb)):
        assert h.guards_intact(b), "write outside a gradient tensor"
        assert torch.isfinite(t.float()).all(), "unwritten or non-finite gradient"
    return h.np64(dq), h.np64(dk), h.np64(dv)


def oracle_grads(x, scale, causal, window=0):
    Q, K, V, dO = (inputs.to_f64(x[n]) for n in ("Q", "K", "V", "dO"))
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, scale, causal, window=window)
    return dQ, dK, dV


def check(got, ref, tol):
    errs = [h.rel_l2(g, r) for g, r in zip(got, ref)]
    assert max(errs) <= tol, dict(zip(("dQ", "dK", "dV"), errs))
    return errs


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 127, 128, 129, 255, 300, 513])
def test_bf16_small_ragged(N, d, causal):
    x = h.seeded(1, 2, N, d, seed=400 + N + d, dtype="bf16", with_dO=True)
    sc = d ** -0.5
    got = run_fwd_bwd(x, sc, causal)
    check(got, oracle_grads(x, sc, causal), h.TOL_GRAD_REL)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [33, 200])
def test_f32_small(N, d, causal):
    x = h.seeded(2, 1, N, d, seed=500 + N + d, dtype="f32", with_dO=True)
    sc = d ** -0.5
    got = run_fwd_bwd(x, sc, causal)
    errs = check(got, oracle_grads(x, sc, causal), h.TOL_GRAD_REL)
    assert max(errs) < 1e-5  # fp32 arithmetic throughout


def test_bf16_multi_head_batch_ragged():
    x = h.seeded(3, 3, 700, 128, seed=611, dtype="bf16", with_dO=True)
    got = run_fwd_bwd(x, 0.09, True)
    check(got, oracle_grads(x, 0.09, True), h.TOL_GRAD_REL)


def test_training_workload_sampled_heads():
    """The training step's shape at full size; the oracle checks four heads
    (chosen by seed) in full."""
    w = inputs.WORKLOADS["train_fwd_bwd"]
    x = inputs.workload_inputs(w)
    dq, dk, dv = run_fwd_bwd(x, w.scale, True)
    g = np.random.default_rng(w.seed)
    heads = sorted(g.choice(w.B * w.H, size=4, replace=False).tolist())
    for bh in heads:
        b, hh = divmod(bh, w.H)
        sub = {n: x[n][b:b + 1, hh:hh + 1] for n in ("Q", "K", "V", "dO")}
        ref = oracle_grads(sub, w.scale, True)
        got = (dq[b:b + 1, hh:hh + 1], dk[b:b + 1, hh:hh + 1], dv[b:b + 1, hh:hh + 1])
        check(got, ref, h.TOL_GRAD_REL)


# --- causal sliding window ("LLM Architecture Refresh [3]", section 5) ---

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,w", [(7, 2), (128, 1), (129, 64), (300, 5), (300, 129),
                                 (513, 256), (700, 384)])
def test_bf16_window_small_ragged(N, w, d):
    x = h.seeded(1, 2, N, d, seed=700 + N + w + d, dtype="bf16", with_dO=True)
    sc = d ** -0.5
    got = run_fwd_bwd(x, sc, True, window=w)
    check(got, oracle_grads(x, sc, True, window=w), h.TOL_GRAD_REL)


@pytest.mark.parametrize("N,w", [(33, 4), (200, 129)])
def test_f32_window_small(N, w):
    x = h.seeded(2, 1, N, 64, seed=800 + N + w, dtype="f32", with_dO=True)
    got = run_fwd_bwd(x, 0.125, True, window=w)
    errs = check(got, oracle_grads(x, 0.125, True, window=w), h.TOL_GRAD_REL)
    assert max(errs) < 1e-5


def test_window_multi_head_batch():
    x = h.seeded(2, 3, 1500, 128, seed=901, dtype="bf16", with_dO=True)
    got = run_fwd_bwd(x, 0.09, True, window=300)
    check(got, oracle_grads(x, 0.09, True, window=300), h.TOL_GRAD_REL)


def test_backward_is_repeatable():
    """Atomics reorder the fp32 dQ sums, so repeated calls agree to rounding,
    and dK, dV (no atomics) agree exactly."""
    x = h.seeded(1, 4, 520, 128, seed=7, dtype="bf16", with_dO=True)
    a = run_fwd_bwd(x, 0.1, True)
    b = run_fwd_bwd(x, 0.1, True)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert h.rel_l2(a[0], b[0]) < 1e-3
