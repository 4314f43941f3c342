"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never loads it and it never
loads the CUDA library: the two share no code.  Inputs are numpy float64
arrays in [B, H, N, d] order; bf16 or fp32 tensors are converted exactly
(every bf16 and fp32 value is a float64 value) before they reach it.

Each wrapper below names the passage of the pages it restates; the C source
(oracle.c) holds the arithmetic.  What pins each function to the pages, other
than itself, is in tests/test_oracle_pins.py.
"""
import ctypes
import os

import numpy as np

from . import build as _build

PLANT_NO_RESCALE = 1  # negative control only: the rebase of l and o is dropped

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_longlong)
        i, d_, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_longlong
        L.oracle_scores.argtypes = [dp, dp, dp, i, i, i, i, d_, i]
        L.oracle_probs.argtypes = [dp, dp, dp, i, i, i, i, d_, i]
        L.oracle_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_, i, i]
        L.oracle_fwd_rows.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_, i,
                                      lp, i64, i]
        L.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i,
                                 d_, i, i]
        L.oracle_fwd_tiled.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_, i,
                                       i, i, i, lp, i64, i, dp]
        L.oracle_online_normalizer.argtypes = [dp, i, i, dp, dp]
        L.oracle_tile_census.argtypes = [i64, i, i, i, i, i, lp]
        L.oracle_fwd_w.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_, i, i]
        L.oracle_fwd_rows_w.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_, i,
                                        i, lp, i64, i]
        L.oracle_bwd_w.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i,
                                   d_, i, i]
        L.oracle_fwd_tiled_w.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_,
                                         i, i, i, lp]
        u32p, u64 = ctypes.POINTER(ctypes.c_uint32), ctypes.c_uint64
        L.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.oracle_philox4x32_10.restype = None
        L.oracle_dropout_keep.argtypes = [i, i, i, i, u64,
                                          ctypes.POINTER(ctypes.c_uint8)]
        L.oracle_fwd_x.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_, i, i, i,
                                   u64, i]
        L.oracle_fwd_rows_x.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d_, i,
                                        i, i, u64, lp, i64, i]
        L.oracle_bwd_x.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i,
                                   d_, i, i, i, u64, i]
        for name in ("oracle_scores", "oracle_probs", "oracle_fwd",
                     "oracle_fwd_rows", "oracle_bwd", "oracle_fwd_tiled",
                     "oracle_online_normalizer", "oracle_tile_census",
                     "oracle_fwd_w", "oracle_fwd_rows_w", "oracle_bwd_w",
                     "oracle_fwd_tiled_w", "oracle_dropout_keep",
                     "oracle_fwd_x", "oracle_fwd_rows_x", "oracle_bwd_x"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape4(Q):
    if Q.ndim != 4:
        raise ValueError("expected [B, H, N, d]")
    return Q.shape


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: oracle rejected its arguments (rc={rc})")


def scores(Q, K, scale, causal=False):
    """Full scaled score matrix S = scale*QK^T (-inf above the diagonal when
    causal) for small inputs.  "Flash Attention, From First Principles",
    Stop 1."""
    Q, K = _f64(Q), _f64(K)
    B, H, N, d = _shape4(Q)
    S = np.empty((B, H, N, N))
    _check(lib().oracle_scores(_ptr(Q), _ptr(K), _ptr(S), B, H, N, d,
                               float(scale), int(causal)), "scores")
    return S


def probs(Q, K, scale, causal=False):
    """Row softmax of the scores with the max subtracted ("Flash Attention,
    From First Principles", Stop 2.5 and Stop 3)."""
    Q, K = _f64(Q), _f64(K)
    B, H, N, d = _shape4(Q)
    P = np.empty((B, H, N, N))
    _check(lib().oracle_probs(_ptr(Q), _ptr(K), _ptr(P), B, H, N, d,
                              float(scale), int(causal)), "probs")
    return P


def dropout_threshold(p):
    """t = round(256 p): the byte threshold of the dropout probability p."""
    t = int(round(256.0 * float(p)))
    if not 0 <= t <= 255:
        raise ValueError("dropout probability must lie in [0, 1)")
    return t


def philox4x32_10(ctr, key):
    """The counter-based generator Philox4x32-10 (Salmon et al., SC'11)."""
    c = (ctypes.c_uint32 * 4)(*ctr)
    k = (ctypes.c_uint32 * 2)(*key)
    out = (ctypes.c_uint32 * 4)()
    lib().oracle_philox4x32_10(c, k, out)
    return tuple(out)


def dropout_keep(B, H, N, p, seed):
    """keep[b, h, r, k] in {0, 1} of the dropout reading (see oracle.c)."""
    keep = np.empty((B, H, N, N), dtype=np.uint8)
    _check(lib().oracle_dropout_keep(B, H, N, dropout_threshold(p), int(seed),
                                     keep.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))),
           "dropout_keep")
    return keep


def fwd(Q, K, V, scale, causal=False, nthreads=0, window=0, dropout_p=0.0,
        seed=0):
    """O = softmax(scale*QK^T)V and LSE = m + ln l, row by row ("FlashAttention
    from scratch", follow-up on the backward pass, for L = m + log l).
    window > 0: the causal sliding window of the "LLM Architecture Refresh
    [3]" section 5 contrast, query r sees keys r - window + 1 .. r."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = _shape4(Q)
    O = np.empty((B, H, N, d))
    LSE = np.empty((B, H, N))
    if dropout_p:
        _check(lib().oracle_fwd_x(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                                  B, H, N, d, float(scale), int(causal),
                                  int(window), dropout_threshold(dropout_p),
                                  int(seed), int(nthreads)), "fwd_x")
        return O, LSE
    if window > 0:
        _check(lib().oracle_fwd_w(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                                  B, H, N, d, float(scale), int(window),
                                  int(nthreads)), "fwd_w")
        return O, LSE
    _check(lib().oracle_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                            B, H, N, d, float(scale), int(causal),
                            int(nthreads)), "fwd")
    return O, LSE


def fwd_rows(Q, K, V, scale, causal, rows, nthreads=0, window=0, dropout_p=0.0,
             seed=0):
    """The forward definition evaluated only at the flat rows
    (b*H + h)*N + r listed in ``rows``; returns O[len(rows), d], LSE[len].
    window > 0 selects the causal sliding window (see fwd)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = _shape4(Q)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    O = np.empty((rows.size, d))
    LSE = np.empty((rows.size,))
    _check(lib().oracle_fwd_rows_x(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, N, d,
        float(scale), int(causal), int(window), dropout_threshold(dropout_p),
        int(seed), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        rows.size, int(nthreads)), "fwd_rows")
    return O, LSE


def bwd(Q, K, V, dO, scale, causal=False, nthreads=0, window=0, dropout_p=0.0,
        seed=0):
    """dQ, dK, dV of the scalar <dO, O>, plus D_r = sum_k p_rk dP_rk ("Flash
    Attention, From First Principles", "The ghost at the door"; "FlashAttention
    from scratch", follow-up on the backward pass).  window > 0 selects the
    causal sliding window (see fwd)."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, d = _shape4(Q)
    dQ = np.empty((B, H, N, d))
    dK = np.empty((B, H, N, d))
    dV = np.empty((B, H, N, d))
    D = np.empty((B, H, N))
    if dropout_p:
        _check(lib().oracle_bwd_x(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ),
                                  _ptr(dK), _ptr(dV), _ptr(D), B, H, N, d,
                                  float(scale), int(causal), int(window),
                                  dropout_threshold(dropout_p), int(seed),
                                  int(nthreads)), "bwd_x")
        return dQ, dK, dV, D
    if window > 0:
        _check(lib().oracle_bwd_w(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ),
                                  _ptr(dK), _ptr(dV), _ptr(D), B, H, N, d,
                                  float(scale), int(window), int(nthreads)),
               "bwd_w")
        return dQ, dK, dV, D
    _check(lib().oracle_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ),
                            _ptr(dK), _ptr(dV), _ptr(D), B, H, N, d,
                            float(scale), int(causal), int(nthreads)), "bwd")
    return dQ, dK, dV, D


def fwd_tiled(Q, K, V, scale, causal, block_q, block_k, flags=0,
              trace_bh=-1, trace_row=-1):
    """The query-outer, key-block-inner online-softmax loop ("LLM Architecture
    Refresh [3]", section 4 and section 7).  Returns (O, LSE, counters, trace)
    with counters = (matmul FLOPs, tiles computed, tiles skipped) and trace a
    [blocks, 2 + d] array of (m, l, o) of one row after each key block."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = _shape4(Q)
    O = np.empty((B, H, N, d))
    LSE = np.empty((B, H, N))
    counters = np.zeros(3, dtype=np.int64)
    nblk = -(-N // block_k)
    trace = np.full((nblk, 2 + d), np.nan)
    _check(lib().oracle_fwd_tiled(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, N, d,
        float(scale), int(causal), int(block_q), int(block_k), int(flags),
        counters.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        int(trace_bh), int(trace_row), _ptr(trace)), "fwd_tiled")
    used = ~np.isnan(trace[:, 0])
    return O, LSE, tuple(int(c) for c in counters), trace[used]


def fwd_tiled_window(Q, K, V, scale, window, block_q, block_k):
    """fwd_tiled for the causal sliding window: key blocks entirely older than
    a query block's window are skipped as well as future ones.  Returns
    (O, LSE, counters)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = _shape4(Q)
    O = np.empty((B, H, N, d))
    LSE = np.empty((B, H, N))
    counters = np.zeros(3, dtype=np.int64)
    _check(lib().oracle_fwd_tiled_w(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, N, d,
        float(scale), int(window), int(block_q), int(block_k),
        counters.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong))),
        "fwd_tiled_w")
    return O, LSE, tuple(int(c) for c in counters)


def online_normalizer(x, block):
    """Running (m, l) after each block of a streamed row ("LLM Architecture
    Refresh [3]", section 2)."""
    x = _f64(x).ravel()
    nblk = -(-x.size // block)
    m = np.empty(nblk)
    l = np.empty(nblk)
    _check(lib().oracle_online_normalizer(_ptr(x), x.size, int(block),
                                          _ptr(m), _ptr(l)), "normalizer")
    return m, l


def tile_census(heads, N, d, block_q, block_k, causal):
    """(matmul FLOPs, tiles computed, tiles skipped) of the tiled loop without
    doing its arithmetic ("LLM Architecture Refresh [3]", sections 7-8)."""
    out = np.zeros(3, dtype=np.int64)
    _check(lib().oracle_tile_census(
        int(heads), int(N), int(d), int(block_q), int(block_k), int(causal),
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong))), "census")
    return tuple(int(c) for c in out)


def cores():
    return os.cpu_count() or 1
