"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Nothing here compares the oracle with itself or with the CUDA path.  Each test
ties one oracle function to a printed worked example (tests/golden/, each file
naming its page and section), a closed form, an invariant or a brute-force
finite difference, chosen so that a dropped term, a wrong sign or index, or a
transposed operand fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_sm_gb300 import inputs
from tests.conftest import load_golden


def printed(dec):
    """Tolerance of a value printed with ``dec`` decimals."""
    return 0.5 * 10.0 ** (-dec) + 1e-12


def as4(a):
    a = np.asarray(a, dtype=np.float64)
    return a.reshape((1, 1) + a.shape)


def rand4(B, H, N, d, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((B, H, N, d))


# --- the 3x2 example ("Flash Attention, From First Principles", Stops 1-3) ---

def test_scores_3x2_example_exact():
    g = load_golden("fp_3x2_example.json")
    S = oracle.scores(as4(g["Q"]), as4(g["K"]), g["scale"])[0, 0]
    # S is printed exactly; S_12 = 0 but S_21 = 2 catches a transposed product
    np.testing.assert_array_equal(S, np.array(g["S"], dtype=np.float64))


def test_probs_3x2_example_printed():
    g = load_golden("fp_3x2_example.json")
    P = oracle.probs(as4(g["Q"]), as4(g["K"]), g["scale"])[0, 0]
    assert np.max(np.abs(P - np.array(g["P"]))) <= printed(g["P_printed_decimals"])
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_fwd_3x2_example_printed():
    g = load_golden("fp_3x2_example.json")
    O, LSE = oracle.fwd(as4(g["Q"]), as4(g["K"]), as4(g["V"]), g["scale"])
    assert np.max(np.abs(O[0, 0] - np.array(g["O"]))) <= printed(g["O_printed_decimals"])
    # LSE of each row equals log of the row's sum of exponentials of the
    # printed integer scores, which are exact
    S = np.array(g["S"], dtype=np.float64)
    expect = np.log(np.exp(S).sum(axis=1))
    np.testing.assert_allclose(LSE[0, 0], expect, rtol=0, atol=1e-14)


# --- the streamed row and the backward receipt (same page) ---

def _row_as_attention(scores, d=2):
    """Queries and keys whose scaled scores are exactly ``scores`` in every
    row: q = (1, 0, ...), k_j = (s_j, 0, ...), scale 1."""
    n = len(scores)
    Q = np.zeros((1, 1, n, d))
    Q[..., 0] = 1.0
    K = np.zeros((1, 1, n, d))
    K[0, 0, :, 0] = np.array(scores, dtype=np.float64)
    return Q, K


def test_streamed_row_film_and_resurrection():
    g = load_golden("fp_streamed_row.json")
    Q, K = _row_as_attention(g["scores"])
    V = as4(g["V"])
    O, LSE = oracle.fwd(Q, K, V, 1.0)
    dec = g["printed_decimals"]
    # every query row of this construction has the same scores; take row 0
    assert np.max(np.abs(O[0, 0, 0] - np.array(g["o"]))) <= printed(dec["o"])
    P = oracle.probs(Q, K, 1.0)[0, 0, 0]
    assert np.max(np.abs(P - np.array(g["weights"]))) <= printed(dec["weights"])
    # the saved statistics: LSE = m + ln r with the printed m and r
    m, r = g["final_m"], g["final_r"]
    assert abs(LSE[0, 0, 0] - (m + math.log(r))) <= printed(dec["final_r"]) / r
    # backward recompute of the middle weight from LSE alone
    assert abs(math.exp(g["scores"][1] - LSE[0, 0, 0]) - g["P_2"]) <= printed(dec["P_2"])
    # and the streamed (tiled, one key at a time) oracle lands on the same row
    O1, _, _, trace = oracle.fwd_tiled(Q, K, V, 1.0, False, 1, 1,
                                       trace_bh=0, trace_row=0)
    assert trace[-1, 0] == m
    assert abs(trace[-1, 1] - r) <= printed(dec["final_r"])
    np.testing.assert_allclose(O1, O, rtol=0, atol=1e-15)


def test_softmax_examples_and_shift_invariance():
    g = load_golden("fp_softmax_examples.json")
    tol = printed(g["printed_decimals"])
    for case in g["cases"]:
        Q, K = _row_as_attention(case["row"])
        P = oracle.probs(Q, K, 1.0)[0, 0, 0]
        assert np.max(np.abs(P - np.array(case["softmax"]))) <= tol
    a, b = g["shift_pair"]
    Pa = oracle.probs(*_row_as_attention(a), 1.0)[0, 0, 0]
    Pb = oracle.probs(*_row_as_attention(b), 1.0)[0, 0, 0]
    np.testing.assert_allclose(Pa, Pb, rtol=0, atol=1e-15)


# --- the 4x4 worked example ("FlashAttention from scratch", Worked example) ---

def test_tiled_trace_4x4_example():
    g = load_golden("fas_4x4_example.json")
    Q, K, V = as4(g["Q"]), as4(g["K"]), as4(g["V"])
    qi = g["query_index"]
    S = oracle.scores(Q, K, g["scale"])[0, 0]
    np.testing.assert_array_equal(S[qi], np.array(g["query_scores"], float))
    O, _, _, trace = oracle.fwd_tiled(Q, K, V, g["scale"], False, 4,
                                      g["block_k"], trace_bh=0, trace_row=qi)
    dec = g["printed_decimals"]
    assert trace.shape[0] == len(g["after_block"])
    for t, step in enumerate(g["after_block"]):
        assert trace[t, 0] == step["m"]
        assert abs(trace[t, 1] - step["l"]) <= printed(dec["l"])
        assert np.max(np.abs(trace[t, 2:] - np.array(step["o"]))) <= printed(dec["o"])
    assert np.max(np.abs(O[0, 0, qi] - np.array(g["final_O"]))) <= printed(dec["final_O"])
    # the plain (untiled) definition gives the same row
    Ou, _ = oracle.fwd(Q, K, V, g["scale"])
    assert np.max(np.abs(Ou[0, 0, qi] - np.array(g["final_O"]))) <= printed(dec["final_O"])


def test_negative_control_without_rescale_is_caught():
    """The mistake the worked example warns about, planted in the oracle: the
    result must be the page's wrong answer and must fail the true pin."""
    g = load_golden("fas_4x4_example.json")
    Q, K, V = as4(g["Q"]), as4(g["K"]), as4(g["V"])
    qi = g["query_index"]
    O, _, _, _ = oracle.fwd_tiled(Q, K, V, g["scale"], False, 4, g["block_k"],
                                  flags=oracle.PLANT_NO_RESCALE)
    dec = g["printed_decimals"]
    assert np.max(np.abs(O[0, 0, qi] - np.array(g["no_rescale_O"]))) <= printed(dec["no_rescale_O"])
    assert np.max(np.abs(O[0, 0, qi] - np.array(g["final_O"]))) > 0.1


# --- the online normaliser ("LLM Architecture Refresh [3]", section 2) ---

def test_online_normalizer_rebase_walkthrough():
    g = load_golden("lar_rebase_walkthrough.json")
    m, l = oracle.online_normalizer(g["logits"], g["block"])
    tol = printed(g["printed_decimals"])
    np.testing.assert_array_equal(m, np.array(g["m_after_block"]))
    assert np.max(np.abs(l - np.array(g["l_after_block"]))) <= tol
    # the streamed sum equals the one-shot sum exp(x - max)
    x = np.array(g["logits"])
    assert abs(l[-1] - np.exp(x - x.max()).sum()) < 1e-15


def test_online_normalizer_hostile_row_matches_one_shot():
    """Logits x8 (a range near 58, as in section 3's hostile input): every
    block size gives the one-shot normaliser to fp64 rounding."""
    x = np.random.default_rng(3).standard_normal(2048) * 8.0
    ref = np.exp(x - x.max()).sum()
    for block in (64, 128, 512, 2048):
        m, l = oracle.online_normalizer(x, block)
        assert m[-1] == x.max()
        assert abs(l[-1] - ref) / ref < 1e-13


# --- tiled == untiled ("FlashAttention from scratch", worked example end;
#     "LLM Architecture Refresh [3]", section 5) ---

@pytest.mark.parametrize("block", [8, 3])
def test_tiled_equals_untiled_64x16(block):
    Q, K, V = (rand4(1, 1, 64, 16, s) for s in (11, 12, 13))
    Ou, Lu = oracle.fwd(Q, K, V, 1.0)
    Ot, Lt, _, _ = oracle.fwd_tiled(Q, K, V, 1.0, False, block, block)
    assert np.max(np.abs(Ot - Ou)) < 1e-14
    assert np.max(np.abs(Lt - Lu)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_tile_shape_does_not_move_the_result(causal):
    Q, K, V = (rand4(2, 2, 200, 16, s) for s in (21, 22, 23))
    sc = 0.25
    Ou, Lu = oracle.fwd(Q, K, V, sc, causal)
    for bq, bk in ((64, 64), (128, 128), (37, 100), (200, 7)):
        Ot, Lt, _, _ = oracle.fwd_tiled(Q, K, V, sc, causal, bq, bk)
        assert np.max(np.abs(Ot - Ou)) < 1e-13
        assert np.max(np.abs(Lt - Lu)) < 1e-13


def test_later_block_holds_the_largest_score():
    """The test recipe of "FlashAttention from scratch" (How do you test your
    implementation?): the row max sits in the last key block, so the rebase
    must fire."""
    Q = np.zeros((1, 1, 8, 2)); Q[..., 0] = 1.0
    K = np.zeros((1, 1, 8, 2)); K[0, 0, :, 0] = np.arange(8) * 0.5
    V = rand4(1, 1, 8, 2, 5)
    Ou, _ = oracle.fwd(Q, K, V, 1.0)
    Ot, _, _, tr = oracle.fwd_tiled(Q, K, V, 1.0, False, 8, 3, trace_bh=0,
                                    trace_row=0)
    assert list(tr[:, 0]) == [1.0, 2.5, 3.5]
    np.testing.assert_allclose(Ot, Ou, rtol=0, atol=1e-15)
    Ob, _, _, _ = oracle.fwd_tiled(Q, K, V, 1.0, False, 8, 3,
                                   flags=oracle.PLANT_NO_RESCALE)
    assert np.max(np.abs(Ob - Ou)) > 1e-2


# --- causal skip and FLOP counts ("LLM Architecture Refresh [3]", 7-8) ---

def test_causal_skip_table():
    g = load_golden("lar_causal_skip.json")
    for row in g["rows"]:
        flops, comp, skip = oracle.tile_census(1, g["seq"], 64, row["block"],
                                               row["block"], True)
        assert (comp, skip) == (row["computed"], row["skipped"])
        assert round(100 * skip / (comp + skip)) == row["percent_skipped"]


@pytest.mark.parametrize("B", [1, 2, 3, 8, 16, 63, 64, 128, 256])
def test_skipped_fraction_closed_form(B):
    _, comp, skip = oracle.tile_census(1, 128 * B, 128, 128, 128, True)
    assert comp + skip == B * B
    assert skip * 2 * B == (B - 1) * B * B   # skip / B^2 == (B-1)/(2B)


def test_flop_table():
    g = load_golden("lar_flops.json")
    tol = printed(g["gflops_printed_decimals"])
    for row in g["rows"]:
        for causal, key in ((False, "noncausal_gflops"), (True, "causal_gflops")):
            flops, _, _ = oracle.tile_census(g["heads"], row["seq"], g["d"],
                                             g["block"], g["block"], causal)
            assert abs(flops / 1e9 - row[key]) <= tol
        # non-causal tiled FLOPs equal the untiled 4 N^2 d per head exactly
        f_nc, _, _ = oracle.tile_census(g["heads"], row["seq"], g["d"],
                                        g["block"], g["block"], False)
        assert f_nc == 4 * row["seq"] ** 2 * g["d"] * g["heads"]


def test_census_matches_tiled_loop_counters():
    Q, K, V = (rand4(1, 2, 77, 4, s) for s in (1, 2, 3))
    for causal in (False, True):
        for bq, bk in ((16, 16), (10, 32), (77, 5)):
            _, _, ctr, _ = oracle.fwd_tiled(Q, K, V, 0.5, causal, bq, bk)
            assert ctr == oracle.tile_census(2, 77, 4, bq, bk, causal)


# --- closed forms and special cases ---

def test_single_key_returns_value_row():
    Q, K, V = (rand4(2, 3, 1, 8, s) for s in (7, 8, 9))
    O, LSE = oracle.fwd(Q, K, V, 0.3)
    np.testing.assert_array_equal(O, V)
    s = 0.3 * np.einsum("bhnd,bhnd->bhn", Q, K)
    np.testing.assert_allclose(LSE, s, rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_give_running_mean(causal):
    N, d = 9, 4
    Q = rand4(1, 1, N, d, 1)
    K = np.tile(rand4(1, 1, 1, d, 2), (1, 1, N, 1))
    V = rand4(1, 1, N, d, 3)
    O, LSE = oracle.fwd(Q, K, V, 0.5, causal)
    for r in range(N):
        cnt = r + 1 if causal else N
        np.testing.assert_allclose(O[0, 0, r], V[0, 0, :cnt].mean(axis=0), atol=1e-14)
        s = 0.5 * Q[0, 0, r] @ K[0, 0, 0]
        assert abs(LSE[0, 0, r] - (s + math.log(cnt))) < 1e-13


def test_causal_first_row_is_first_value():
    Q, K, V = (rand4(1, 2, 6, 3, s) for s in (4, 5, 6))
    O, _ = oracle.fwd(Q, K, V, 1.0, True)
    np.testing.assert_array_equal(O[:, :, 0], V[:, :, 0])


def test_large_logits_stay_finite_and_rows_sum_to_one():
    """Section 3's hostile input: logits with a range near 58."""
    Q, K, V = (rand4(1, 1, 512, 64, s) for s in (31, 32, 33))
    sc = 1.0  # <q, k> over d = 64 has std 8, so the row range is ~58
    P = oracle.probs(Q, K, sc)
    assert np.ptp(oracle.scores(Q, K, sc)[0, 0], axis=1).max() > 40
    assert np.all(np.isfinite(P))
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, rtol=0, atol=1e-13)
    O, LSE = oracle.fwd(Q, K, V, sc)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(LSE))


def test_fwd_rows_equals_full_forward_at_those_rows():
    Q, K, V = (rand4(2, 2, 50, 8, s) for s in (41, 42, 43))
    O, LSE = oracle.fwd(Q, K, V, 0.4, True)
    rows = np.array([0, 7, 49, 50, 99, 150, 199])
    Or, Lr = oracle.fwd_rows(Q, K, V, 0.4, True, rows)
    np.testing.assert_array_equal(Or, O.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(Lr, LSE.reshape(-1)[rows])


# --- backward: finite differences and identities ---

def _loss(Q, K, V, dO, sc, causal):
    O, _ = oracle.fwd(Q, K, V, sc, causal)
    return float(np.sum(O * dO))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 1), (3, 2), (6, 4), (5, 3)])
def test_gradients_match_central_differences(causal, N, d):
    Q, K, V, dO = (rand4(1, 2, N, d, s) for s in (51, 52, 53, 54))
    sc = 0.7
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, sc, causal)
    h = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            fp = _loss(Q, K, V, dO, sc, causal)
            X[idx] = old - h
            fm = _loss(Q, K, V, dO, sc, causal)
            X[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(num - G)) < 1e-7


def test_D_equals_rowwise_dot_of_dO_and_O():
    Q, K, V, dO = (rand4(2, 2, 40, 8, s) for s in (61, 62, 63, 64))
    for causal in (False, True):
        O, _ = oracle.fwd(Q, K, V, 0.35, causal)
        _, _, _, D = oracle.bwd(Q, K, V, dO, 0.35, causal)
        np.testing.assert_allclose(D, np.sum(dO * O, axis=-1), rtol=0, atol=1e-13)


def test_equal_keys_backward_closed_forms():
    """With every key equal, P is uniform: dQ = 0 (each dS row sums to zero)
    and dV_k = mean over rows of dO (non-causal)."""
    N, d = 7, 3
    Q = rand4(1, 1, N, d, 71)
    K = np.tile(rand4(1, 1, 1, d, 72), (1, 1, N, 1))
    V, dO = rand4(1, 1, N, d, 73), rand4(1, 1, N, d, 74)
    dQ, dK, dV, _ = oracle.bwd(Q, K, V, dO, 0.9, False)
    np.testing.assert_allclose(dQ, 0.0, atol=1e-14)
    np.testing.assert_allclose(dV[0, 0], np.tile(dO[0, 0].mean(axis=0), (N, 1)), atol=1e-14)


# --- the causal sliding window ("LLM Architecture Refresh [3]", section 5:
# each query attends only to the last w keys, itself included) ---

def test_window_covering_every_key_is_causal():
    Q, K, V = (rand4(2, 2, 23, 5, s) for s in (81, 82, 83))
    Oc, Lc = oracle.fwd(Q, K, V, 0.4, True)
    for w in (23, 24, 1000):
        Ow, Lw = oracle.fwd(Q, K, V, 0.4, window=w)
        # the same terms in the same order: identical
        assert np.array_equal(Ow, Oc) and np.array_equal(Lw, Lc)


def test_window_of_one_returns_own_value_row():
    Q, K, V = (rand4(1, 3, 11, 4, s) for s in (84, 85, 86))
    sc = 0.6
    O, LSE = oracle.fwd(Q, K, V, sc, window=1)
    np.testing.assert_allclose(O, V, rtol=0, atol=1e-15)
    np.testing.assert_allclose(LSE, sc * np.sum(Q * K, axis=-1), rtol=0, atol=1e-13)


@pytest.mark.parametrize("w", [2, 3, 7])
def test_window_with_constant_scores_averages_the_last_w_values(w):
    """Q = 0 makes every visible score 0: row r is the plain mean of
    v_max(0, r-w+1) .. v_r and LSE_r = ln(min(r+1, w))."""
    N, d = 13, 3
    Q = np.zeros((1, 1, N, d))
    K, V = rand4(1, 1, N, d, 87), rand4(1, 1, N, d, 88)
    O, LSE = oracle.fwd(Q, K, V, 1.0, window=w)
    for r in range(N):
        lo = max(0, r - w + 1)
        np.testing.assert_allclose(O[0, 0, r], V[0, 0, lo:r + 1].mean(axis=0), atol=1e-14)
        assert abs(LSE[0, 0, r] - math.log(r + 1 - lo)) < 1e-14


@pytest.mark.parametrize("N,w,bq,bk", [(37, 11, 8, 5), (64, 16, 16, 16), (50, 1, 7, 9), (40, 33, 8, 8)])
def test_window_tiled_equals_untiled_and_skips_old_tiles(N, w, bq, bk):
    Q, K, V = (rand4(1, 2, N, 6, s) for s in (89, 90, 91))
    O, L = oracle.fwd(Q, K, V, 0.45, window=w)
    Ot, Lt, (flops, computed, skipped) = oracle.fwd_tiled_window(Q, K, V, 0.45, w, bq, bk)
    np.testing.assert_allclose(Ot, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(Lt, L, rtol=0, atol=1e-13)
    # brute-force tile census: a tile is needed iff some (query, key) pair in
    # it is visible, i.e. key <= query and key >= query - w + 1
    need = 0
    for i in range(0, N, bq):
        for j in range(0, N, bk):
            qs, ks = range(i, min(N, i + bq)), range(j, min(N, j + bk))
            if any(k <= q and k >= q - w + 1 for q in qs for k in ks):
                need += 1
    tiles = -(-N // bq) * -(-N // bk) * 2
    assert computed == 2 * need and computed + skipped == tiles


@pytest.mark.parametrize("N,d,w", [(7, 3, 3), (5, 2, 1), (6, 4, 5)])
def test_window_gradients_match_central_differences(N, d, w):
    Q, K, V, dO = (rand4(1, 2, N, d, s) for s in (92, 93, 94, 95))
    sc = 0.8
    dQ, dK, dV, D = oracle.bwd(Q, K, V, dO, sc, window=w)
    O, _ = oracle.fwd(Q, K, V, sc, window=w)
    np.testing.assert_allclose(D, np.sum(dO * O, axis=-1), rtol=0, atol=1e-13)
    h = 1e-6

    def loss():
        Ow, _ = oracle.fwd(Q, K, V, sc, window=w)
        return float(np.sum(Ow * dO))

    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            fp = loss()
            X[idx] = old - h
            fm = loss()
            X[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(num - G)) < 1e-7


def test_window_rows_equal_full_window_forward():
    Q, K, V = (rand4(2, 2, 30, 4, s) for s in (96, 97, 98))
    O, L = oracle.fwd(Q, K, V, 0.5, window=6)
    rows = [0, 5, 29, 30 + 7, 60 + 29, 90 + 12]
    Or, Lr = oracle.fwd_rows(Q, K, V, 0.5, True, rows, window=6)
    np.testing.assert_allclose(Or, O.reshape(-1, 4)[rows], rtol=0, atol=0)
    np.testing.assert_allclose(Lr, L.reshape(-1)[rows], rtol=0, atol=0)


# --- dropout (the reading of "algorithm 2's extra lines", "Flash Attention,
# From First Principles", what is left out): P o M with M = keep * 256/(256-t),
# keep from Philox4x32-10 over 4x4 (query, key) patches ---

def test_philox_matches_published_known_answers():
    g = load_golden("philox4x32_10_kat.json")
    for case in g["cases"]:
        ctr = [int(x, 16) for x in case["counter"]]
        key = [int(x, 16) for x in case["key"]]
        assert oracle.philox4x32_10(ctr, key) == tuple(int(x, 16) for x in case["out"])


def test_dropout_patch_layout_and_locality():
    """keep(r, k) is byte k%4 of word r%4 of the call at counter
    (k/4, r/4, head, 0); it depends on nothing but (head, r, k, seed)."""
    seed, p = 0x1234_5678_9ABC_DEF0, 0.3
    t = oracle.dropout_threshold(p)
    keep = oracle.dropout_keep(2, 3, 40, p, seed)
    g = np.random.default_rng(5)
    for _ in range(50):
        bh, r, k = int(g.integers(6)), int(g.integers(40)), int(g.integers(40))
        out = oracle.philox4x32_10((k // 4, r // 4, bh, 0), (seed & 0xFFFFFFFF, seed >> 32))
        byte = (out[r % 4] >> (8 * (k % 4))) & 0xFF
        assert keep.reshape(6, 40, 40)[bh, r, k] == (byte >= t)
    big = oracle.dropout_keep(2, 3, 100, p, seed)
    assert np.array_equal(big[:, :, :40, :40], keep)
    other = oracle.dropout_keep(2, 3, 40, p, seed + 1)
    assert not np.array_equal(other, keep)


@pytest.mark.parametrize("p", [0.1, 0.25, 0.5, 0.9])
def test_dropout_keep_rate(p):
    keep = oracle.dropout_keep(2, 4, 512, p, 77)
    q = 1 - oracle.dropout_threshold(p) / 256
    n = keep.size
    assert abs(keep.mean() - q) < 5 * math.sqrt(q * (1 - q) / n)


def test_dropout_threshold_zero_is_no_dropout():
    Q, K, V = (rand4(1, 2, 19, 4, s) for s in (101, 102, 103))
    O0, L0 = oracle.fwd(Q, K, V, 0.5, True)
    O1, L1 = oracle.fwd(Q, K, V, 0.5, True, dropout_p=0.001, seed=3)  # t = 0
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_dropout_keeps_lse_and_is_unbiased():
    Q, K, V = (rand4(1, 1, 6, 2, s) for s in (104, 105, 106))
    O, L = oracle.fwd(Q, K, V, 0.7, False)
    acc = np.zeros_like(O)
    n = 3000
    for seed in range(n):
        Od, Ld = oracle.fwd(Q, K, V, 0.7, False, dropout_p=0.5, seed=seed)
        assert np.array_equal(Ld, L)  # the normaliser is the undropped row's
        acc += Od
    assert np.max(np.abs(acc / n - O)) < 0.06


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3)])
def test_dropout_gradients_match_central_differences(causal, window):
    N, d = 6, 3
    Q, K, V, dO = (rand4(1, 2, N, d, s) for s in (107, 108, 109, 110))
    sc, p, seed = 0.8, 0.4, 99
    dQ, dK, dV, D = oracle.bwd(Q, K, V, dO, sc, causal, window=window, dropout_p=p, seed=seed)
    O, _ = oracle.fwd(Q, K, V, sc, causal, window=window, dropout_p=p, seed=seed)
    np.testing.assert_allclose(D, np.sum(dO * O, axis=-1), rtol=0, atol=1e-13)
    h = 1e-6

    def loss():
        Od, _ = oracle.fwd(Q, K, V, sc, causal, window=window, dropout_p=p, seed=seed)
        return float(np.sum(Od * dO))

    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            fp = loss()
            X[idx] = old - h
            fm = loss()
            X[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(num - G)) < 1e-7


def test_dropout_rows_equal_full_forward():
    Q, K, V = (rand4(2, 2, 30, 4, s) for s in (111, 112, 113))
    O, L = oracle.fwd(Q, K, V, 0.5, True, dropout_p=0.2, seed=11)
    rows = [0, 5, 29, 37, 89, 102]
    Or, Lr = oracle.fwd_rows(Q, K, V, 0.5, True, rows, dropout_p=0.2, seed=11)
    np.testing.assert_allclose(Or, O.reshape(-1, 4)[rows], rtol=0, atol=0)
    np.testing.assert_allclose(Lr, L.reshape(-1)[rows], rtol=0, atol=0)


# --- the seeded generator is exact in the oracle's arithmetic ---

def test_bf16_inputs_widen_exactly():
    t = inputs.seeded_inputs(1, 2, 33, 16, seed=5, dtype="bf16")
    for name in ("Q", "K", "V"):
        x = inputs.to_f64(t[name])
        back = torch.from_numpy(x).to(torch.bfloat16)
        assert torch.equal(back, t[name])


def test_seeded_inputs_are_reproducible_and_ordered():
    a = inputs.seeded_inputs(1, 1, 8, 4, seed=9, dtype="f32", with_dO=True)
    b = inputs.seeded_inputs(1, 1, 8, 4, seed=9, dtype="f32", with_dO=False)
    for n in ("Q", "K", "V"):
        assert torch.equal(a[n], b[n])
    assert not torch.equal(a["Q"], a["K"])
