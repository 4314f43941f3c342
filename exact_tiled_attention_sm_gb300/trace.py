"""Per-CTA timing of the persistent kernels, from the trace build of the
library (libfa_trace.so: the product sources compiled with FA_CTA_TRACE, see
csrc/fa_trace.cuh), and the balance summary `bench.py --balance` prints.
Marshalling and arithmetic on recorded times only; the attention itself runs
in the trace build's kernels exactly as in libfa.so."""
import ctypes

READERS = {"fwd": "fa_cta_trace_fwd", "bwd": "fa_cta_trace_bwd", "bwd64": "fa_cta_trace_bwd64",
           "fwd256": "fa_cta_trace_fwd256", "bwd256": "fa_cta_trace_bwd256"}
MAX_CTAS = 1024  # kTraceMaxCtas in csrc/fa_trace.cuh


def read(lib, kernel):
    """(start, end) in ns of every CTA of the last traced launch of `kernel`
    ("fwd", "bwd", "bwd64", "fwd256" or "bwd256"), then cleared on the
    device."""
    buf = (ctypes.c_ulonglong * (2 * MAX_CTAS))()
    fn = getattr(lib, READERS[kernel])
    fn.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]
    fn.restype = ctypes.c_int
    if fn(buf, MAX_CTAS) != 0:
        raise RuntimeError(f"{READERS[kernel]} failed")
    return [(buf[2 * c], buf[2 * c + 1]) for c in range(MAX_CTAS) if buf[2 * c]]


def summarize(marks):
    """Balance of one launch from its CTAs' (start, end) marks: the launch's
    span (first start to last end), each CTA's busy time (its end minus its
    start), and when the CTAs finished relative to the first start."""
    t0 = min(s for s, _ in marks)
    ends = sorted(e - t0 for _, e in marks)
    busy = [e - s for s, e in marks]
    span = ends[-1]
    mean_busy = sum(busy) / len(busy)
    return {
        "ctas": len(marks),
        "span_us": round(span / 1e3, 2),
        "busy_mean_us": round(mean_busy / 1e3, 2),
        "busy_max_us": round(max(busy) / 1e3, 2),
        "busy_max_over_mean": round(max(busy) / mean_busy, 4),
        "first_finish_us": round(ends[0] / 1e3, 2),
        "median_finish_us": round(ends[len(ends) // 2] / 1e3, 2),
        "last_finish_us": round(ends[-1] / 1e3, 2),
        "tail_us": round((ends[-1] - ends[0]) / 1e3, 2),
        "tail_frac_of_span": round((ends[-1] - ends[0]) / span, 4),
        "idle_frac": round(1.0 - sum(busy) / (len(busy) * span), 4),
    }
