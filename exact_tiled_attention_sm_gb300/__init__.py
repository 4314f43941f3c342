"""Python binding of libfa.so, the exact tiled attention library for sm_103a.

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  The
raw entry points mirror include/fa.h (``fa_fwd``, ``fa_bwd``, ...); ``fwd``
and ``bwd`` are tensor conveniences that allocate outputs with torch and call
them.  There is no fallback: if libfa.so is missing or was built for another
machine, every call raises.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_BF16, FA_F32 = 0, 1

# Every symbol include/fa.h declares.
EXPORTS = ("fa_fwd", "fa_bwd_workspace_size", "fa_bwd", "fa_fwd_window",
           "fa_bwd_window", "fa_fwd_dropout", "fa_bwd_dropout", "fa_fwd_fp8",
           "fa_dropout_threshold", "fa_dropout_mask", "fa_bwd_noalloc",
           "fa_last_device_status",
           "fa_status_string", "fa_selftest_wait_timeout",
           "fa_fwd_schedule_census", "fa_fwd_schedule_census_window",
           "fa_fwd_schedule_cover", "fa_version")

_lib = None


class FAError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def use_library(path):
    """Makes every later call go to the library at ``path`` instead of
    libfa.so; only before the first call.  bench.py --balance uses it to load
    the trace build (libfa_trace.so: the same kernels, recording per-CTA
    start and end times)."""
    global LIB_PATH
    if _lib is not None:
        raise RuntimeError("the library is already loaded")
    LIB_PATH = path


def lib():
    """Loads libfa.so (raising if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        L.fa_fwd.restype = i
        L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        L.fa_bwd_workspace_size.restype = ctypes.c_size_t
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f,
                             i, i, vp, ctypes.c_size_t, vp]
        L.fa_bwd.restype = i
        L.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        L.fa_fwd_window.restype = i
        L.fa_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i,
                                    i, f, i, i, vp, ctypes.c_size_t, vp]
        L.fa_bwd_window.restype = i
        u64 = ctypes.c_ulonglong
        L.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i,
                                     f, u64, i, vp]
        L.fa_fwd_dropout.restype = i
        L.fa_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i,
                                     i, i, f, i, i, f, u64, i, vp,
                                     ctypes.c_size_t, vp]
        L.fa_bwd_dropout.restype = i
        L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, f, f,
                                 f, vp]
        L.fa_fwd_fp8.restype = i
        L.fa_dropout_threshold.argtypes = [f]
        L.fa_dropout_threshold.restype = i
        L.fa_dropout_mask.argtypes = [vp, i, i, i, f, u64, vp]
        L.fa_dropout_mask.restype = i
        L.fa_fwd_schedule_census_window.argtypes = [
            i, i, i, ctypes.POINTER(ctypes.c_longlong)]
        L.fa_fwd_schedule_census_window.restype = i
        L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i,
                                     i, i, f, i, i, vp]
        L.fa_bwd_noalloc.restype = i
        L.fa_last_device_status.argtypes = [vp]
        L.fa_last_device_status.restype = i
        L.fa_status_string.argtypes = [i]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        L.fa_selftest_wait_timeout.restype = i
        L.fa_fwd_schedule_census.argtypes = [i, i, ctypes.POINTER(ctypes.c_longlong)]
        L.fa_fwd_schedule_census.restype = i
        L.fa_fwd_schedule_cover.argtypes = [i, i, i, i, i, i, ctypes.POINTER(i),
                                            ctypes.POINTER(i), ctypes.POINTER(i)]
        L.fa_fwd_schedule_cover.restype = i
        L.fa_version.argtypes = []
        L.fa_version.restype = i
        _lib = L
    return _lib


# ---------------------------------------------------------------- raw C ABI
def fa_fwd(Q, K, V, O, LSE, B, H, N, d, scale, causal, dt, stream):
    return lib().fa_fwd(Q, K, V, O, LSE, B, H, N, d, scale, int(causal), dt, stream)


def fa_bwd_workspace_size(B, H, N, d):
    return lib().fa_bwd_workspace_size(B, H, N, d)


def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, dt,
           workspace, workspace_bytes, stream):
    return lib().fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale,
                        int(causal), dt, workspace, workspace_bytes, stream)


def fa_fwd_window(Q, K, V, O, LSE, B, H, N, d, scale, window, dt, stream):
    return lib().fa_fwd_window(Q, K, V, O, LSE, B, H, N, d, scale, int(window),
                               dt, stream)


def fa_bwd_window(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, window,
                  dt, workspace, workspace_bytes, stream):
    return lib().fa_bwd_window(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d,
                               scale, int(window), dt, workspace,
                               workspace_bytes, stream)


def fa_fwd_dropout(Q, K, V, O, LSE, B, H, N, d, scale, causal, window,
                   dropout_p, seed, dt, stream):
    return lib().fa_fwd_dropout(Q, K, V, O, LSE, B, H, N, d, scale,
                                int(causal), int(window), float(dropout_p),
                                int(seed), dt, stream)


def fa_bwd_dropout(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal,
                   window, dropout_p, seed, dt, workspace, workspace_bytes,
                   stream):
    return lib().fa_bwd_dropout(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d,
                                scale, int(causal), int(window),
                                float(dropout_p), int(seed), dt, workspace,
                                workspace_bytes, stream)


def fa_fwd_fp8(Q, K, V, O, LSE, B, H, N, d, scale, causal, window, q_descale,
               k_descale, v_descale, stream):
    return lib().fa_fwd_fp8(Q, K, V, O, LSE, B, H, N, d, scale, int(causal),
                            int(window), float(q_descale), float(k_descale),
                            float(v_descale), stream)


def fa_dropout_threshold(dropout_p):
    return lib().fa_dropout_threshold(float(dropout_p))


def fa_dropout_mask(keep, B, H, N, dropout_p, seed, stream):
    return lib().fa_dropout_mask(keep, B, H, N, float(dropout_p), int(seed),
                                 stream)


def fa_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal,
                   dt, stream):
    """fa_bwd with the library's own scratch array instead of a workspace, for
    callers that cannot allocate device memory (see include/fa.h)."""
    return lib().fa_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d,
                                scale, int(causal), dt, stream)


def fa_last_device_status(stream=None):
    return lib().fa_last_device_status(stream)


def fa_status_string(s):
    return lib().fa_status_string(s).decode()


def fa_selftest_wait_timeout(limit_us, stream=None):
    return lib().fa_selftest_wait_timeout(limit_us, stream)


def fa_fwd_schedule_census(N, causal):
    out = (ctypes.c_longlong * 3)()
    st = lib().fa_fwd_schedule_census(N, int(causal), out)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_schedule_census")
    return tuple(out)


def fa_fwd_schedule_census_window(N, causal, window):
    out = (ctypes.c_longlong * 3)()
    st = lib().fa_fwd_schedule_census_window(N, int(causal), int(window), out)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_schedule_census_window")
    return tuple(out)


def fa_fwd_schedule_cover(BH, N, causal, window, num_sms, d=128):
    """(counts per (head, query block) as a BH x ceil(N/128) list of lists,
    grid, items) of the forward launch's work list."""
    nq = (N + 127) // 128
    counts = (ctypes.c_int * (BH * nq))()
    grid, items = ctypes.c_int(0), ctypes.c_int(0)
    st = lib().fa_fwd_schedule_cover(BH, N, int(causal), int(window), int(d), num_sms,
                                     counts, ctypes.byref(grid), ctypes.byref(items))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_schedule_cover")
    return [list(counts[b * nq:(b + 1) * nq]) for b in range(BH)], grid.value, items.value


def fa_version():
    return lib().fa_version()


def status_string(s):
    try:
        return fa_status_string(s)
    except Exception:  # library not loadable: still name the code
        return {0: "ok", 1: "invalid argument", 2: "unsupported",
                3: "CUDA error", 4: "device wait timed out"}.get(s, "unknown")


# ---------------------------------------------------------- tensor helpers
def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check_tensor(t, shape, name):
    if not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous CUDA tensor of shape {shape}")


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def fwd(q, k, v, scale, causal=False, out=None, lse=None, stream=None,
        window=0, dropout_p=0.0, seed=0):
    """O, LSE = attention forward of [B, H, N, d] CUDA tensors (bf16 or fp32).
    window > 0: causal sliding window of that many keys (fa_fwd_window);
    dropout_p > 0: attention dropout with the keep mask of ``seed``
    (fa_fwd_dropout)."""
    import torch
    B, H, N, d = q.shape
    dt = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, (B, H, N, d), n)
        if t.dtype != q.dtype:
            raise TypeError("q, k and v must share one dtype")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_tensor(out, (B, H, N, d), "out")
    _check_tensor(lse, (B, H, N), "lse")
    if dropout_p:
        st = fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                            out.data_ptr(), lse.data_ptr(), B, H, N, d,
                            float(scale), causal, window, dropout_p, seed, dt,
                            _stream_ptr(stream))
    elif window:
        st = fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           out.data_ptr(), lse.data_ptr(), B, H, N, d,
                           float(scale), window, dt, _stream_ptr(stream))
    else:
        st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                    lse.data_ptr(), B, H, N, d, float(scale), causal, dt,
                    _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_dropout" if dropout_p else
                      "fa_fwd_window" if window else "fa_fwd")
    return out, lse


def fwd_fp8(q8, k8, v8, scale, descales, causal=False, out=None, lse=None,
            stream=None, window=0):
    """O (bf16), LSE = attention forward of E4M3 [B, H, N, 128] CUDA tensors
    (torch.float8_e4m3fn or their raw uint8 bytes) standing for
    descales[0] * q8, descales[1] * k8, descales[2] * v8 (fa_fwd_fp8)."""
    import torch
    B, H, N, d = q8.shape
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _check_tensor(t, (B, H, N, d), n)
        if t.element_size() != 1:
            raise TypeError(f"{n} must hold one byte per element (E4M3)")
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    _check_tensor(out, (B, H, N, d), "out")
    _check_tensor(lse, (B, H, N), "lse")
    if out.dtype != torch.bfloat16:
        raise TypeError("out must be bf16")
    qd, kd, vd = descales
    st = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(),
                    lse.data_ptr(), B, H, N, d, float(scale), causal, window,
                    qd, kd, vd, _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return out, lse


def workspace(B, H, N, d, device=None):
    """A device buffer large enough for fa_bwd on this shape."""
    import torch
    n = fa_bwd_workspace_size(B, H, N, d)
    if n == 0:
        raise FAError(FA_ERR_INVALID_ARG, "fa_bwd_workspace_size")
    return torch.empty((n,), dtype=torch.uint8, device=device or "cuda")


def bwd(q, k, v, o, do, lse, scale, causal=False, dq=None, dk=None, dv=None,
        ws=None, stream=None, window=0, dropout_p=0.0, seed=0):
    """dQ, dK, dV of attention for upstream gradient ``do``.  window > 0:
    causal sliding window of that many keys (fa_bwd_window); dropout_p > 0:
    the forward's dropout, regenerated from ``seed`` (fa_bwd_dropout)."""
    import torch
    B, H, N, d = q.shape
    dt = _dtype_code(q)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check_tensor(t, (B, H, N, d), n)
    _check_tensor(lse, (B, H, N), "lse")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = workspace(B, H, N, d, q.device) if ws is None else ws
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
            dv.data_ptr(), B, H, N, d, float(scale))
    if dropout_p:
        st = fa_bwd_dropout(*args, causal, window, dropout_p, seed, dt,
                            ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    elif window:
        st = fa_bwd_window(*args, window, dt, ws.data_ptr(), ws.numel(),
                           _stream_ptr(stream))
    else:
        st = fa_bwd(*args, causal, dt, ws.data_ptr(), ws.numel(),
                    _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_bwd_dropout" if dropout_p else
                      "fa_bwd_window" if window else "fa_bwd")
    return dq, dk, dv


def dropout_mask(B, H, N, dropout_p, seed, device=None, stream=None):
    """The keep mask of fa_fwd_dropout as a [B, H, N, N] uint8 CUDA tensor
    (1 kept, 0 dropped), written by fa_dropout_mask."""
    import torch
    keep = torch.empty((B, H, N, N), dtype=torch.uint8, device=device or "cuda")
    st = fa_dropout_mask(keep.data_ptr(), B, H, N, dropout_p, seed,
                         _stream_ptr(stream))
    if st != FA_OK:
        raise FAError(st, "fa_dropout_mask")
    return keep


def last_device_status(stream=None):
    return fa_last_device_status(_stream_ptr(stream) if stream is not None else None)
