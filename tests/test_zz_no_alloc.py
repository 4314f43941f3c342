"""fa_bwd_noalloc, the backward for callers that cannot allocate device
memory (a plugin that receives only its input and output buffers, a loop
that must not pay cudaMalloc's synchronisation, a fixed memory budget): it
runs on a scratch array the library reserves once per GPU instead of a
caller workspace.  Called through the C ABI with raw pointers, its output
must match fa_bwd's (which uses a caller workspace) within the gradient
tolerance, on two calls in a row (the scratch keeps the previous call's
contents, which must not leak into the next), and the fp64 oracle's
gradients as well; sizes beyond the scratch must be refused before anything
runs.  The cases cover the bf16 tensor-core backward, the fp32 path and head
dimension 256, which use the scratch differently.  This file is collected
last so that a stop-at-first-failure run has already run every other test."""
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h

pytestmark = pytest.mark.gpu


def _noalloc(q, k, v, o, do, lse, dq, dk, dv, scale, causal):
    B, H, N, d = q.shape
    dt = fa.FA_F32 if q.dtype == torch.float32 else fa.FA_BF16
    return fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                             dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale),
                             causal, dt, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,H,N,d,causal,dtype", [
    (2, 4, 700, 128, True, "bf16"),
    (1, 8, 1000, 64, False, "bf16"),
    (1, 3, 300, 256, True, "bf16"),
    (2, 1, 200, 128, True, "f32"),
])
def test_noalloc_matches_workspace_backward_twice(B, H, N, d, causal, dtype):
    x = h.seeded(B, H, N, d, seed=900 + N, dtype=dtype, with_dO=True)
    q, k, v, do = (x[n].cuda() for n in ("Q", "K", "V", "dO"))
    sc = d ** -0.5
    o, lse = fa.fwd(q, k, v, sc, causal)
    ref = [h.np64(t) for t in fa.bwd(q, k, v, o, do, lse, sc, causal)]
    Q, K, V, dO = (inputs.to_f64(x[n]) for n in ("Q", "K", "V", "dO"))
    exact = oracle.bwd(Q, K, V, dO, sc, causal)[:3]
    tol = h.TOL_GRAD_REL if dtype == "bf16" else h.TOL_F32
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    for _ in range(2):
        dq, dqb = h.guarded((B, H, N, d), tdt)
        dk, dkb = h.guarded((B, H, N, d), tdt)
        dv, dvb = h.guarded((B, H, N, d), tdt)
        assert _noalloc(q, k, v, o, do, lse, dq, dk, dv, sc, causal) == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        for t, b, r, e in ((dq, dqb, ref[0], exact[0]), (dk, dkb, ref[1], exact[1]),
                           (dv, dvb, ref[2], exact[2])):
            assert h.guards_intact(b)
            assert torch.isfinite(t.float()).all()
            got = h.np64(t)
            assert h.rel_l2(got, r) <= tol      # the workspace backward
            assert h.rel_l2(got, e) <= tol      # the oracle


def test_noalloc_refuses_sizes_beyond_its_scratch():
    B, H, N, d = 1, 32, 4096, 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) > (64 << 20)
    p = 1 << 20  # never dereferenced: the size check comes first
    st = fa.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0.1, 1,
                           fa.FA_BF16, None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_workspace_size(1, 32, 2048, 128) <= (64 << 20)
