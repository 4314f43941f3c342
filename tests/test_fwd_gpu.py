"""Forward parity of the CUDA path (through the C ABI) against the fp64 oracle
on the same seeded inputs: small ragged shapes element by element, the named
workloads at full size on sampled rows, and the edge cases."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_sm_gb300 as fa
import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests import helpers as h
from tests.conftest import load_golden

pytestmark = pytest.mark.gpu


def run_fwd(x, scale, causal, window=0):
    """Calls fa_fwd (fa_fwd_window when window > 0) with NaN-prefilled,
    guard-banded O and LSE."""
    q, k, v = (x[n].to("cuda") for n in ("Q", "K", "V"))
    B, H, N, d = q.shape
    o, ob = h.guarded((B, H, N, d), q.dtype)
    lse, lb = h.guarded((B, H, N), torch.float32)
    fa.fwd(q, k, v, scale, causal, out=o, lse=lse, window=window)
    torch.cuda.synchronize()
    assert fa.last_device_status() == fa.FA_OK
    assert h.guards_intact(ob) and h.guards_intact(lb), "write outside O/LSE"
    assert torch.isfinite(o.float()).all(), "unwritten or non-finite O"
    assert torch.isfinite(lse).all(), "unwritten or non-finite LSE"
    return h.np64(o), h.np64(lse)


def test_f32_single_head_workload():
    w = inputs.WORKLOADS["single_head_f32"]
    x = inputs.workload_inputs(w)
    o, lse = run_fwd(x, w.scale, False)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), w.scale, False)
    assert h.max_abs(o, O) <= h.TOL_F32
    assert h.max_abs(lse, L) <= h.TOL_F32


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_worked_3x2_example(dtype):
    """The 3x2 example of "Flash Attention, From First Principles" (scale 1),
    zero-padded to d = 64 so that the scores are unchanged."""
    g = load_golden("fp_3x2_example.json")
    Q = torch.zeros((1, 1, 3, 64))
    K = torch.zeros((1, 1, 3, 64))
    V = torch.zeros((1, 1, 3, 64))
    Q[0, 0, :, :2] = torch.tensor(g["Q"], dtype=torch.float32)
    K[0, 0, :, :2] = torch.tensor(g["K"], dtype=torch.float32)
    V[0, 0, :, :2] = torch.tensor(g["V"], dtype=torch.float32)
    cast = torch.float32 if dtype == "f32" else torch.bfloat16
    x = {"Q": Q.to(cast), "K": K.to(cast), "V": V.to(cast)}
    o, lse = run_fwd(x, 1.0, False)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), 1.0)
    tol_o = h.TOL_F32 if dtype == "f32" else h.TOL_O_BF16
    tol_l = h.TOL_F32 if dtype == "f32" else h.TOL_LSE_BF16
    assert h.max_abs(o, O) <= tol_o
    assert h.max_abs(lse, L) <= tol_l
    assert np.max(np.abs(o[0, 0, :, :2] - np.array(g["O"]))) <= 5e-4 + tol_o


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 127, 128, 129, 255, 256, 300, 513])
def test_bf16_small_ragged(N, d, causal):
    x = h.seeded(2, 2, N, d, seed=100 + N + d, dtype="bf16")
    sc = d ** -0.5
    o, lse = run_fwd(x, sc, causal)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), sc, causal)
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [64, 200, 320])
def test_f32_small_ragged(N, causal):
    x = h.seeded(1, 3, N, 128, seed=300 + N, dtype="f32")
    o, lse = run_fwd(x, 0.125, causal)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), 0.125, causal)
    assert h.max_abs(o, O) <= h.TOL_F32
    assert h.max_abs(lse, L) <= h.TOL_F32


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_later_block_holds_the_max(d):
    """"FlashAttention from scratch" test recipe: the largest score of every
    row sits in the last key block, so every row rescales."""
    N = 640
    x = h.seeded(1, 2, N, d, seed=77, dtype="bf16")
    K = x["K"].float()
    K[:, :, -100:, :] *= 3.0
    x["K"] = K.to(torch.bfloat16)
    o, lse = run_fwd(x, d ** -0.5, False)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), d ** -0.5)
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_reference_moves_every_block(d, causal):
    """Keys of block b scaled by 1, 3, 6, 9, 12: at each later block a third
    to three quarters of the rows see their maximum rise past the exponent
    reference by more than its slack, so every warp rescales O at every block
    ("LLM Architecture Refresh [3]", section 4, the running-max correction).
    At d = 64 the rescale waits for the previous P V in flight.  V / 4 keeps
    the nearly one-hot rows' |O| below 2, where the 1e-2 bound holds."""
    N = 640
    x = h.seeded(1, 2, N, d, seed=79 + d, dtype="bf16")
    K = x["K"].float()
    for b, f in enumerate((1.0, 3.0, 6.0, 9.0, 12.0)):
        K[:, :, 128 * b:128 * (b + 1), :] *= f
    x["K"] = K.to(torch.bfloat16)
    x["V"] = (x["V"].float() * 0.25).to(torch.bfloat16)
    o, lse = run_fwd(x, d ** -0.5, causal)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), d ** -0.5, causal)
    assert np.abs(O).max() < 2.0
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_d64_one_long_head(causal):
    """d = 64 with one head of 8192 rows: 64 single-block items for 304
    workers, so most workers idle and, under the mask, the items range from
    1 to 64 key blocks.  Rows sampled across the sequence against the
    oracle."""
    N, d = 8192, 64
    x = h.seeded(1, 1, N, d, seed=5150, dtype="bf16")
    o, lse = run_fwd(x, d ** -0.5, causal)
    rows = np.array([0, 1, 127, 128, 1000, 4095, 4096, 6001, N - 129, N - 128, N - 1])
    Q, K, V = (inputs.to_f64(x[n]) for n in ("Q", "K", "V"))
    O, L = oracle.fwd_rows(Q, K, V, d ** -0.5, causal, rows)
    A, _ = oracle.fwd_rows(Q, K, np.abs(V), d ** -0.5, causal, rows)
    # the first causal rows see one or two keys: O is then a row of V, |O|
    # up to ~4, where bf16 rounding alone exceeds 1e-2 (see the bound below)
    err = np.abs(o.reshape(-1, d)[rows] - O)
    assert np.all(err <= np.maximum(h.TOL_O_BF16, rounding_bound(O, A)))
    assert h.max_abs(lse.reshape(-1)[rows], L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_d64_many_short_heads(causal):
    """d = 64 with 4 x 64 heads of 130 rows: two query blocks per head (the
    second of 2 rows), 512 single-block items over the workers, several
    waves of tiny items.  Every row against the oracle."""
    B, H, N, d = 4, 64, 130, 64
    x = h.seeded(B, H, N, d, seed=5151, dtype="bf16")
    o, lse = run_fwd(x, d ** -0.5, causal)
    Q, K, V = (inputs.to_f64(x[n]) for n in ("Q", "K", "V"))
    O, L, bound = bf16_output_bound(Q, K, V, d ** -0.5, causal)
    # (the first causal rows of each head copy a row of V; see above)
    assert np.all(np.abs(o - O) <= np.maximum(h.TOL_O_BF16, bound))
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


def test_bf16_large_logits_stay_finite():
    """Logits with a range near 58 ("LLM Architecture Refresh [3]",
    section 3): no overflow, no NaN.  Such rows are nearly one-hot, so O
    copies rows of V; V / 4 keeps |O| below 2, where the 1e-2 bound holds
    (bf16 output rounding alone exceeds it for |O| >= 4)."""
    N, d = 512, 64
    x = h.seeded(1, 2, N, d, seed=78, dtype="bf16")
    x["V"] = (x["V"].float() * 0.25).to(torch.bfloat16)
    o, lse = run_fwd(x, 1.0, True)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), 1.0, True)
    assert np.abs(O).max() < 2.0
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


def _sampled_parity(w, causal, per_head=48, window=0):
    x = inputs.workload_inputs(w, with_dO=False)
    o, lse = run_fwd(x, w.scale, causal, window)
    rows = inputs.sample_rows(w.B, w.H, w.N, per_head=per_head, seed=w.seed).numpy()
    Q, K, V = (inputs.to_f64(x[n]) for n in ("Q", "K", "V"))
    O, L = oracle.fwd_rows(Q, K, V, w.scale, causal, rows, window=window)
    og = o.reshape(-1, w.d)[rows]
    lg = lse.reshape(-1)[rows]
    return h.max_abs(og, O), h.max_abs(lg, L)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name", ["gpt2_medium_fwd", "llama3_8b_fwd"])
def test_workload_full_size_sampled(name, causal):
    eo, el = _sampled_parity(inputs.WORKLOADS[name], causal)
    assert eo <= h.TOL_O_BF16 and el <= h.TOL_LSE_BF16, (eo, el)


@pytest.mark.parametrize("name", ["long_ctx_8k", "long_ctx_16k", "long_ctx_32k"])
def test_long_context_sampled(name):
    eo, el = _sampled_parity(inputs.WORKLOADS[name], True, per_head=24)
    assert eo <= h.TOL_O_BF16 and el <= h.TOL_LSE_BF16, (eo, el)


# --- causal sliding window ("LLM Architecture Refresh [3]", section 5) ---

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,w", [(7, 1), (128, 1), (128, 64), (129, 128), (129, 129),
                                 (300, 16), (300, 129), (300, 256), (513, 200),
                                 (513, 384), (1000, 127)])
def test_bf16_window_small_ragged(N, w, d):
    x = h.seeded(2, 2, N, d, seed=500 + N + w + d, dtype="bf16")
    sc = d ** -0.5
    o, lse = run_fwd(x, sc, True, window=w)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), sc, window=w)
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("N,w", [(7, 2), (7, 3), (300, 5), (129, 4)])
def test_bf16_tiny_window(N, w):
    """Windows of a few keys: O is then close to single value rows, so V is
    scaled by 1/4 to keep |O| < 1, where the bf16 output's own rounding stays
    well inside the 1e-2 bound (with |O| near 4 a half ulp alone is 0.008)."""
    x = h.seeded(1, 2, N, 128, seed=550 + N + w, dtype="bf16")
    x["V"] = (x["V"].float() * 0.25).to(torch.bfloat16)
    o, lse = run_fwd(x, 0.0884, True, window=w)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), 0.0884, window=w)
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


@pytest.mark.parametrize("N,w", [(64, 1), (200, 17), (320, 129)])
def test_f32_window_small(N, w):
    x = h.seeded(1, 3, N, 128, seed=600 + N + w, dtype="f32")
    o, lse = run_fwd(x, 0.125, True, window=w)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), 0.125, window=w)
    assert h.max_abs(o, O) <= h.TOL_F32
    assert h.max_abs(lse, L) <= h.TOL_F32


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,w", [(300, 16), (640, 40), (520, 100)])
def test_window_row_whose_first_visible_key_is_in_a_later_block(N, w, d):
    """Under the window a row of query block q may see nothing in the first
    key block the block visits (rows 128q + w .. of block q see no key of
    block kv_lo(q)), so its first visible scores arrive in the next block
    while the running reference is still the placeholder.  With all scaled
    scores near -128 (times log2(e) below -128), rebasing from that
    placeholder would overflow; O and LSE must match the oracle."""
    x, sc = h.late_first_key_inputs(N, d, seed=700 + N + w + d)
    o, lse = run_fwd(x, sc, True, window=w)
    O, L = oracle.fwd(*(inputs.to_f64(x[n]) for n in ("Q", "K", "V")), sc, window=w)
    assert L.max() < -40.0
    assert h.max_abs(o, O) <= h.TOL_O_BF16
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


def bf16_half_ulp(x):
    """Half a unit in the last place of bf16 (8 significant bits) at |x|."""
    m, e = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))  # |x| = m 2^e, m in [0.5, 1)
    return np.where(m > 0, np.ldexp(1.0, e - 9), 0.0)


def bf16_output_bound(Q, K, V, scale, causal):
    """Element-wise error bound of the bf16 forward, from its arithmetic:
    P is rounded to bf16 before the P V product (relative error <= 2^-8 per
    weight, and the largest weight is not exactly 1 since the exponent
    reference may trail the row maximum), while l sums the unrounded values;
    then O is rounded to bf16 (half an ulp).  With p the exact probabilities,
      |O - O_ref| <= (2^-8 + 2e-4) sum_k p_k |v_k|
                     + half_ulp(|O_ref| + 2^-8 sum_k p_k |v_k|) + 1e-5,
    the 2e-4 and 1e-5 covering the fp32 score and product sums and exp2.
    sum_k p_k |v_k| is the oracle's forward with |V| as the values."""
    O, L = oracle.fwd(Q, K, V, scale, causal)
    A, _ = oracle.fwd(Q, K, np.abs(V), scale, causal)
    return O, L, rounding_bound(O, A)


def rounding_bound(O, A):
    """The bound of bf16_output_bound from the oracle's O and
    A = sum_k p_k |v_k|."""
    return (2.0 ** -8 + 2e-4) * A + bf16_half_ulp(np.abs(O) + 2.0 ** -8 * A) + 1e-5


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_peaked_rows_within_the_rounding_bound(d, causal):
    """Nearly one-hot rows (scale 1 on N(0,1) inputs: score spread about
    sqrt(d)) with |V| in [2, 8), so that O copies value rows of that size:
    the rows where the forward's rescale slack can matter.  Every element is
    held to the bound its arithmetic gives (bf16_output_bound), and most of
    them have |O| >= 2."""
    N = 700
    x = h.seeded(1, 2, N, d, seed=880 + d + causal, dtype="bf16")
    v = x["V"].float()
    x["V"] = (torch.sign(v) * (2.0 + 5.9 * torch.rand(v.shape, generator=torch.Generator().manual_seed(881))))
    x["V"] = x["V"].to(torch.bfloat16)
    o, lse = run_fwd(x, 1.0, causal)
    Q, K, V = (inputs.to_f64(x[n]) for n in ("Q", "K", "V"))
    O, L, bound = bf16_output_bound(Q, K, V, 1.0, causal)
    assert np.mean(np.abs(O) >= 2.0) > 0.5
    err = np.abs(o - O)
    assert np.all(err <= bound), float(np.max(err - bound))
    assert h.max_abs(lse, L) <= h.TOL_LSE_BF16


def test_window_covering_the_sequence_is_the_causal_forward():
    x = h.seeded(2, 3, 700, 128, seed=9, dtype="bf16")
    oc, lc = run_fwd(x, 0.09, True)
    for w in (700, 701, 100000):
        ow, lw = run_fwd(x, 0.09, True, window=w)
        assert np.array_equal(ow, oc) and np.array_equal(lw, lc)


@pytest.mark.parametrize("w", [64, 256, 3000])
def test_window_long_context_sampled(w):
    eo, el = _sampled_parity(inputs.WORKLOADS["long_ctx_8k"], True, per_head=24, window=w)
    assert eo <= h.TOL_O_BF16 and el <= h.TOL_LSE_BF16, (eo, el)


def test_repeated_calls_are_identical():
    x = h.seeded(2, 4, 777, 128, seed=5, dtype="bf16")
    a = run_fwd(x, 0.1, True)
    b = run_fwd(x, 0.1, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bounded_wait_times_out_and_reports():
    """Failure detection without a fault: a wait on a barrier that nothing
    completes gives up after 0.2 s, and the host reads FA_ERR_TIMEOUT."""
    assert fa.fa_selftest_wait_timeout(200000, None) == fa.FA_OK
    assert fa.last_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.last_device_status() == fa.FA_OK  # cleared by the read
    x = h.seeded(1, 1, 256, 64, seed=6, dtype="bf16")
    run_fwd(x, 0.125, False)  # the context is still usable
