"""Shared helpers for the GPU parity tests: run the CUDA path and the fp64 oracle
on the same seeded inputs and compare element by element.

Tolerance (stated for bf16 outputs, applied to every path): max |dO| <= 1e-2,
mean |dO| <= 1e-3, max |dLSE| <= 1e-3, against the fp64 oracle evaluated on
exactly the values the GPU received.
"""
import numpy as np

TOL_MAX_O = 1e-2
TOL_MEAN_O = 1e-3
TOL_MAX_LSE = 1e-3


def errors(o_gpu, o_ref, lse_gpu=None, lse_ref=None):
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    d = np.abs(o_gpu - o_ref)
    out = {"max_o": float(d.max()) if d.size else 0.0,
           "mean_o": float(d.mean()) if d.size else 0.0,
           "worst_o_index": tuple(int(i) for i in np.unravel_index(int(d.argmax()), d.shape))
           if d.size else ()}
    if lse_gpu is not None:
        lg = np.asarray(lse_gpu, np.float64)
        lr = np.asarray(lse_ref, np.float64)
        both_inf = np.isneginf(lg) & np.isneginf(lr)
        with np.errstate(invalid="ignore"):
            dl = np.where(both_inf, 0.0, np.abs(lg - lr))
        out["max_lse"] = float(dl.max()) if dl.size else 0.0
    return out


def assert_close(e, what=""):
    assert np.isfinite(e["max_o"]), (what, e)
    assert e["max_o"] <= TOL_MAX_O, (what, e)
    assert e["mean_o"] <= TOL_MEAN_O, (what, e)
    if "max_lse" in e:
        assert e["max_lse"] <= TOL_MAX_LSE, (what, e)


# |dO| histogram bin edges for the full-output reports
HIST_EDGES = (0.0, 1e-4, 3e-4, 1e-3, 3e-3, 1e-2, np.inf)

# reports of the full-output comparisons, printed at the end of the run (conftest)
REPORTS = []


def full_report(name, o_gpu, o_ref, lse_gpu, lse_ref, row_axes):
    """Error figures over every output element of a workload: max and mean |dO|, the
    worst row (its index along `row_axes` of O), max |dLSE| and a histogram of |dO|.
    The report is kept for the end-of-run summary and returned."""
    e = errors(o_gpu, o_ref, lse_gpu, lse_ref)
    d = np.abs(np.asarray(o_gpu, np.float64) - np.asarray(o_ref, np.float64))
    hist, _ = np.histogram(d, bins=np.array(HIST_EDGES))
    rep = {"workload": name, "elements": int(d.size), "max_o": e["max_o"],
           "mean_o": e["mean_o"], "max_lse": e["max_lse"],
           "worst_row": [int(e["worst_o_index"][a]) for a in row_axes],
           "hist_edges": [float(x) for x in HIST_EDGES[1:-1]],
           "hist_counts": [int(c) for c in hist]}
    REPORTS.append(rep)
    return e, rep

