"""The forward and the backward captured into a CUDA graph (causal, sliding
window, dropout; d = 64, 128, 256): the backward's three launches (D and the
zeroed accumulator, the backward kernel, the dQ conversion) are chained as
programmatic dependent launches, and a graph keeps those edges.  Replays must
give the eager results: O, LSE, dK and dV bit for bit (no
launch-order-dependent arithmetic), dQ (fp32 reduce-adds whose order varies
between launches) within rounding, and, without dropout, the fp64 oracle's
gradients."""
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,window,dropout_p", [
    (64, 0, 0.0), (128, 0, 0.0), (256, 0, 0.0),  # causal
    (128, 300, 0.0), (256, 300, 0.0),             # sliding window of 300 keys
    (128, 0, 0.1), (256, 0, 0.1),                 # causal with dropout
])
def test_fwd_bwd_graph_replay_matches_eager(d, window, dropout_p):
    B, H, N, causal = 1, 4, 700, True
    sc = d ** -0.5
    seed = 77
    x = h.seeded(B, H, N, d, seed=900 + d + window, dtype="bf16", with_dO=True)
    q, k, v, do = (x[n].to("cuda") for n in ("Q", "K", "V", "dO"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.workspace(B, H, N, d)

    def step():
        fa.fwd(q, k, v, sc, causal, out=o, lse=lse, window=window, dropout_p=dropout_p,
               seed=seed)
        fa.bwd(q, k, v, o, do, lse, sc, causal, dq=dq, dk=dk, dv=dv, ws=ws, window=window,
               dropout_p=dropout_p, seed=seed)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # eager run (and warm-up) off the default stream
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    eager = [t.clone() for t in (o, lse, dq, dk, dv)]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for rep in range(2):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))  # every output must be rewritten by the replay
        g.replay()
        torch.cuda.synchronize()
        assert fa.last_device_status() == fa.FA_OK
        for name, got, ref in (("O", o, eager[0]), ("LSE", lse, eager[1]),
                               ("dK", dk, eager[3]), ("dV", dv, eager[4])):
            assert torch.equal(got, ref), f"replay {rep}: {name} differs from the eager run"
        assert torch.isfinite(dq.float()).all()
        assert h.rel_l2(h.np64(dq), h.np64(eager[2])) <= 1e-3

    if dropout_p:  # the dropout paths' own parity tests compare them with the oracle
        return
    Q, K, V, dO = (inputs.to_f64(x[n]) for n in ("Q", "K", "V", "dO"))
    dQr, dKr, dVr, _ = oracle.bwd(Q, K, V, dO, sc, causal, window=window)
    for got, ref in ((dq, dQr), (dk, dKr), (dv, dVr)):
        assert h.rel_l2(h.np64(got), ref) <= h.TOL_GRAD_REL
