"""The largest tensors the library accepts: B*H*N*d just under 2^31
elements (4095 heads of 4096 x 128, 4 GiB per bf16 tensor), so that every
offset past 2^31 bytes and near 2^31 elements is exercised.  The oracle
checks rows of the first, a middle and the last head (the last head's last
row ends one element short of 2^31 - 2^19) and the last head's gradients."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h

pytestmark = pytest.mark.gpu


def test_maximum_size_forward_and_backward():
    B, H, N, d = 1, 4095, 4096, 128
    assert B * H * N * d < 2 ** 31 <= B * (H + 1) * N * d
    sc = d ** -0.5
    x = inputs.seeded_inputs_cuda(B, H, N, d, seed=4242, with_dO=True)
    o, lse = fa.fwd(x["Q"], x["K"], x["V"], sc, True)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    rows = np.array([0, 1, 127, 128, 2047, 4000, N - 2, N - 1])
    for hh in (0, H // 2, H - 1):
        Q, K, V = (inputs.to_f64(x[n][:, hh:hh + 1]) for n in ("Q", "K", "V"))
        O, L = oracle.fwd_rows(Q, K, V, sc, True, rows)
        assert h.max_abs(h.np64(o[0, hh])[rows], O) <= h.TOL_O_BF16, hh
        assert h.max_abs(h.np64(lse[0, hh])[rows], L) <= h.TOL_LSE_BF16, hh
    dq, dk, dv = fa.bwd(x["Q"], x["K"], x["V"], o, x["dO"], lse, sc, True)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    hh = H - 1
    Q, K, V, dO = (inputs.to_f64(x[n][:, hh:hh + 1]) for n in ("Q", "K", "V", "dO"))
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, True)
    for got, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        assert h.rel_l2(h.np64(got[:, hh:hh + 1]), ref) <= h.TOL_GRAD_REL
    del x, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def test_maximum_size_head_dim_256_forward_and_backward():
    """The same bound at head dimension 256: 8191 heads of 1024 x 256 (one
    2^18 short of 2^31 elements), through the d = 256 forward and the
    tensor-core backward (its items walk each key block twice, once per half
    of d, and add dQ with reds from registers)."""
    B, H, N, d = 1, 8191, 1024, 256
    assert B * H * N * d < 2 ** 31 <= B * (H + 1) * N * d
    sc = d ** -0.5
    x = inputs.seeded_inputs_cuda(B, H, N, d, seed=4343, with_dO=True)
    o, lse = fa.fwd(x["Q"], x["K"], x["V"], sc, True)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    rows = np.array([0, 1, 63, 64, 127, 128, 700, N - 2, N - 1])
    for hh in (0, H // 2, H - 1):
        Q, K, V = (inputs.to_f64(x[n][:, hh:hh + 1]) for n in ("Q", "K", "V"))
        O, L = oracle.fwd_rows(Q, K, V, sc, True, rows)
        assert h.max_abs(h.np64(o[0, hh])[rows], O) <= h.TOL_O_BF16, hh
        assert h.max_abs(h.np64(lse[0, hh])[rows], L) <= h.TOL_LSE_BF16, hh
    dq, dk, dv = fa.bwd(x["Q"], x["K"], x["V"], o, x["dO"], lse, sc, True)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    for hh in (0, H - 1):
        Q, K, V, dO = (inputs.to_f64(x[n][:, hh:hh + 1]) for n in ("Q", "K", "V", "dO"))
        dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, True)
        for got, ref in ((dq, dQ), (dk, dK), (dv, dV)):
            assert h.rel_l2(h.np64(got[:, hh:hh + 1]), ref) <= h.TOL_GRAD_REL, hh
    del x, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def test_maximum_size_head_dim_64_forward_and_backward():
    """The same bound at head dimension 64: 8191 heads of 4096 x 64, through
    the d = 64 forward (S issued ahead of P V, one issuing thread per query
    block) and the tensor-core backward."""
    B, H, N, d = 1, 8191, 4096, 64
    assert B * H * N * d < 2 ** 31 <= B * (H + 1) * N * d
    sc = d ** -0.5
    x = inputs.seeded_inputs_cuda(B, H, N, d, seed=4444, with_dO=True)
    for causal in (False, True):
        o, lse = fa.fwd(x["Q"], x["K"], x["V"], sc, causal)
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        rows = np.array([0, 1, 127, 128, 255, 256, 2047, 4000, N - 2, N - 1])
        for hh in (0, H // 2, H - 1):
            Q, K, V = (inputs.to_f64(x[n][:, hh:hh + 1]) for n in ("Q", "K", "V"))
            O, L = oracle.fwd_rows(Q, K, V, sc, causal, rows)
            assert h.max_abs(h.np64(o[0, hh])[rows], O) <= h.TOL_O_BF16, (causal, hh)
            assert h.max_abs(h.np64(lse[0, hh])[rows], L) <= h.TOL_LSE_BF16, (causal, hh)
    dq, dk, dv = fa.bwd(x["Q"], x["K"], x["V"], o, x["dO"], lse, sc, True)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    hh = H - 1
    Q, K, V, dO = (inputs.to_f64(x[n][:, hh:hh + 1]) for n in ("Q", "K", "V", "dO"))
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, True)
    for got, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        assert h.rel_l2(h.np64(got[:, hh:hh + 1]), ref) <= h.TOL_GRAD_REL
    del x, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
