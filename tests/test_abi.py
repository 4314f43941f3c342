"""The C ABI without a GPU: the library loads, exports every symbol that
include/fa.h declares, rejects bad arguments before launching anything, and
its host-side scheduler census agrees with the pages' causal tile count."""
import ctypes
import os
import re

import pytest

import exact_tiled_attention_sm_gb300 as fa
import oracle
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from exact_tiled_attention_sm_gb300 import _build
    _build.build()
    return fa.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    decl = declared_symbols()
    assert len(decl) >= 8
    assert sorted(fa.EXPORTS) == decl
    for name in decl:
        assert hasattr(L, name), name


def test_status_strings(L):
    assert fa.fa_status_string(fa.FA_OK) == "ok"
    assert fa.fa_status_string(fa.FA_ERR_TIMEOUT) == "device wait timed out"
    assert fa.fa_version() >= 100


def _fwd(**kw):
    a = dict(Q=16, K=16, V=16, O=16, LSE=16, B=1, H=1, N=16, d=64, scale=0.1,
             causal=0, dt=fa.FA_BF16, stream=None)
    a.update(kw)
    return fa.fa_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"],
                     a["N"], a["d"], a["scale"], a["causal"], a["dt"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(Q=None), fa.FA_ERR_INVALID_ARG),
    (dict(LSE=None), fa.FA_ERR_INVALID_ARG),
    (dict(K=24), fa.FA_ERR_INVALID_ARG),          # not 16-byte aligned
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(dt=7), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 20, H=1 << 10, N=1 << 10), fa.FA_ERR_INVALID_ARG),  # overflow
])
def test_fwd_rejects_bad_arguments(L, kw, expect):
    assert _fwd(**kw) == expect


def test_bwd_rejects_bad_arguments(L):
    n = fa.fa_bwd_workspace_size(1, 1, 16, 64)
    assert n >= 16 * 4 + 16 * 64 * 4
    args = [256] * 9 + [1, 1, 16, 64, 0.1, 0, fa.FA_BF16]
    # short workspace, null workspace, misaligned workspace
    assert fa.fa_bwd(*args, 256, n - 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd(*args, None, n, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd(*args, 272, n, None) == fa.FA_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = None  # dQ
    assert fa.fa_bwd(*bad, 256, n, None) == fa.FA_ERR_INVALID_ARG
    bad = list(args)
    bad[12] = 32   # d
    assert fa.fa_bwd(*bad, 256, n, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_workspace_size(1, 1, 16, 48) == 0
    assert fa.fa_bwd_workspace_size(0, 1, 16, 64) == 0


def test_workspace_size_is_linear_in_N(L):
    """The backward's scratch is O(N) per head and the forward's is zero:
    nothing grows like N^2 ("LLM Architecture Refresh [3]", section 6)."""
    sizes = [fa.fa_bwd_workspace_size(1, 32, n, 128) for n in (8192, 16384, 32768)]
    assert sizes[1] == 2 * sizes[0] and sizes[2] == 2 * sizes[1]
    assert sizes[2] == 32 * 32768 * (128 + 1) * 4


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 1000, 2048, 4096, 8192, 16384, 32768])
def test_schedule_census_matches_tile_walk(L, N, causal):
    comp, skip, items = fa.fa_fwd_schedule_census(N, causal)
    _, oc, os_ = oracle.tile_census(1, N, 128, 128, 128, causal)
    assert (comp, skip) == (oc, os_)
    nq = -(-N // 128)
    assert items == -(-nq // 2)


@pytest.mark.parametrize("N", [8192, 16384, 32768])
def test_schedule_skips_closed_form_fraction(L, N):
    """(B-1)/(2B) of the 128x128 tiles are skipped for B blocks a side
    ("LLM Architecture Refresh [3]", section 7)."""
    comp, skip, _ = fa.fa_fwd_schedule_census(N, True)
    Bk = N // 128
    assert comp + skip == Bk * Bk
    assert skip * 2 * Bk == (Bk - 1) * Bk * Bk


@pytest.mark.parametrize("N,w", [(1, 1), (100, 7), (128, 1), (129, 128), (300, 129),
                                 (1000, 256), (2048, 64), (4096, 1000), (513, 513),
                                 (600, 5000)])
def test_window_schedule_census_matches_tiled_walk(L, N, w):
    """The sliding window's key-block ranges visit exactly the tiles the
    oracle's windowed tile loop computes ("LLM Architecture Refresh [3]",
    sections 5 and 7)."""
    import numpy as np
    comp, skip, items = fa.fa_fwd_schedule_census_window(N, 1, w)
    z = np.zeros((1, 1, N, 1))
    _, _, (_, oc, os_) = oracle.fwd_tiled_window(z, z, z, 1.0, w, 128, 128)
    assert (comp, skip) == (oc, os_)
    assert items == -(-(-(-N // 128)) // 2)


def test_window_entry_points_reject_bad_windows(L):
    a = [16, 16, 16, 16, 16, 1, 1, 16, 64, 0.1]
    for w in (0, -1, -300):
        assert fa.fa_fwd_window(*a, w, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    n = fa.fa_bwd_workspace_size(1, 1, 16, 64)
    b = [256] * 9 + [1, 1, 16, 64, 0.1]
    for w in (0, -2):
        assert fa.fa_bwd_window(*b, w, fa.FA_BF16, 256, n, None) == fa.FA_ERR_INVALID_ARG
    with pytest.raises(fa.FAError):
        fa.fa_fwd_schedule_census_window(16, 1, -1)


def test_dropout_threshold_matches_the_oracle(L):
    """t = round(256 p) with ties to even, on both sides; values exact in fp32
    so that both sides round the same number."""
    import numpy as np
    ps = [0.0, 0.1, 0.25, 0.5, 0.9, 1 / 512, 3 / 512, 5 / 512, 509 / 512,
          510.9 / 512, 0.3333]
    for p in ps:
        p32 = float(np.float32(p))
        assert fa.fa_dropout_threshold(p32) == oracle.dropout_threshold(p32), p
    for p in (-1e-9, -0.5, 511 / 512, 1.0, 2.0, float("nan"), float("inf")):
        assert fa.fa_dropout_threshold(p) == -1, p


def test_dropout_entry_points_reject_bad_arguments(L):
    a = [16, 16, 16, 16, 16, 1, 1, 16, 64, 0.1]
    n = fa.fa_bwd_workspace_size(1, 1, 16, 64)
    b = [256] * 9 + [1, 1, 16, 64, 0.1]
    for causal, window, p in ((0, 0, -0.1), (0, 0, 1.0), (1, -1, 0.1),
                              (0, 0, float("nan"))):
        assert fa.fa_fwd_dropout(*a, causal, window, p, 1, fa.FA_BF16,
                                 None) == fa.FA_ERR_INVALID_ARG
        assert fa.fa_bwd_dropout(*b, causal, window, p, 1, fa.FA_BF16, 256, n,
                                 None) == fa.FA_ERR_INVALID_ARG
    for args in ((None, 1, 1, 16, 0.1, 0), (16, 0, 1, 16, 0.1, 0),
                 (16, 1, 1, 0, 0.1, 0), (16, 1, 1, 300000, 0.1, 0),
                 (16, 1, 1, 16, 1.5, 0)):
        assert fa.fa_dropout_mask(*args, None) == fa.FA_ERR_INVALID_ARG


def test_fp8_entry_point_rejects_bad_arguments(L):
    a = [16, 16, 16, 16, 16, 1, 1, 16]
    for d, f, w, expect in ((64, (1.0, 1.0, 1.0), 0, fa.FA_ERR_UNSUPPORTED),
                            (128, (0.0, 1.0, 1.0), 0, fa.FA_ERR_INVALID_ARG),
                            (128, (1.0, float("inf"), 1.0), 0, fa.FA_ERR_INVALID_ARG),
                            (128, (1.0, 1.0, -2.0), 0, fa.FA_ERR_INVALID_ARG),
                            (128, (1.0, 1.0, 1.0), -1, fa.FA_ERR_INVALID_ARG),
                            (128, (1e30, 1e30, 1.0), 0, fa.FA_ERR_INVALID_ARG)):
        assert fa.fa_fwd_fp8(*a, d, 0.1, 0, w, *f, None) == expect


def test_library_has_no_oracle_symbols(L):
    """The product library and the oracle share nothing."""
    assert not hasattr(L, "oracle_fwd")
    path = fa.LIB_PATH
    data = open(path, "rb").read()
    assert b"oracle_" not in data


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300)])
@pytest.mark.parametrize("BH,N,sms", [(128, 1024, 152), (128, 1024, 148), (1, 256, 152),
                                      (3, 1000, 152), (5, 129, 152), (64, 4096, 152),
                                      (4095, 4096, 152), (7, 2048, 2), (1, 1, 152)])
def test_forward_work_list_covers_every_query_block_once(L, BH, N, sms, causal, window, d):
    """The forward launch's work list, walked on the host exactly as the CTAs
    take it (waves, snake order, head groups; at d = 128 pairs of query
    blocks, without a mask the pairs of a last wave that fills at most half
    the grid split into single blocks; at d = 64 single blocks for two
    workers per CTA): every (head, 128-row query block) is held by exactly one
    item."""
    counts, grid, items = fa.fa_fwd_schedule_cover(BH, N, causal, window, sms, d)
    assert 1 <= grid <= sms
    assert all(c == 1 for row in counts for c in row)
    nq = (N + 127) // 128
    if d == 64:
        assert items == BH * nq
    else:
        assert BH * ((nq + 1) // 2) <= items <= BH * nq


def test_forward_work_list_splits_the_last_partial_wave(L):
    """128 heads of 1024 rows at d = 128 without a mask on 152 SMs: 512
    two-block items make 3 waves and 56 items, so those 56 become 112
    single-block items and the grid stays at 152."""
    counts, grid, items = fa.fa_fwd_schedule_cover(128, 1024, False, 0, 152, 128)
    assert grid == 152 and all(c == 1 for row in counts for c in row)
    assert items == 3 * 152 + 2 * 56
    # under the causal mask the items differ in cost and none is split
    _, _, items_c = fa.fa_fwd_schedule_cover(128, 1024, True, 0, 152, 128)
    assert items_c == 512
    # at d = 64 every item is one query block, for 2 x 152 workers
    counts, grid, items = fa.fa_fwd_schedule_cover(128, 1024, False, 0, 152, 64)
    assert grid == 152 and items == 1024
    assert all(c == 1 for row in counts for c in row)
