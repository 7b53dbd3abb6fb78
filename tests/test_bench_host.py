"""The benchmark's host-side arithmetic, on the CPU: the roofline's nominal
bytes (both logit tensors read once over the valid positions) of each target
workload, and the classification of GPU/oracle disagreements in the parity
counts that the benchmark reports."""
import importlib.util
import os

import numpy as np

import oracle
from speculative_decoding_verify_03_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def test_nominal_bytes_of_the_target_workloads():
    """sum_b (2 gamma_b + 1) V s: the per-call byte counts of the workloads'
    shapes (B x (2 gamma + 1) x V x element size)."""
    b = _bench()
    assert b.nominal_bytes(W.WORKLOADS[1], None) == 64 * 9 * 50304 * 4 == 115_900_416
    assert b.nominal_bytes(W.WORKLOADS[2], None) == 256 * 17 * 128256 * 2 == 1_116_340_224
    assert b.nominal_bytes(W.WORKLOADS[3], None) == 4096 * 9 * 1024 * 4 == 150_994_944
    gam = np.array([1, 8, 3], np.int32)
    w4 = W.WORKLOADS[4]
    assert b.nominal_bytes(w4, gam) == (3 + 17 + 7) * 152064 * 2
    # greedy reads the target only: (gamma + 1) rows
    from dataclasses import replace
    assert b.nominal_bytes(replace(W.WORKLOADS[0], temperature=0.0), None) == 5 * 50304 * 4


def test_parity_counts_classify_disagreements():
    b = _bench()
    n = 6
    diag = np.zeros(n, oracle.DIAG_DTYPE)
    diag["accept_margin"] = [1.0, 5e-7, 1.0, 1.0, 1.0, 1.0]
    diag["cdf_margin"] = [1.0, 1.0, 2e-7, 1.0, 1.0, 1.0]
    diag["topp_margin"] = np.inf
    diag["n_tests"] = [2, 1, 3, 1, 1, 0]
    diag["n_draws"] = 1
    o = {"accepted_len": np.array([1, 0, 2, 0, 0, 0]), "next_token": np.array([5, 6, 7, 8, 9, 1]),
         "diag": diag}
    acc = np.array([1, 1, 2, 0, 0, 0])   # row 1 differs (near an acceptance boundary)
    nxt = np.array([5, 6, 9, 8, 3, 1])   # row 2 differs (near a CDF boundary); row 4 is hard
    c = b.parity_counts(o, acc, nxt)
    assert c == {"rows": 6, "draws": 14, "near_boundary": 2, "disagree": 3, "hard": 1,
                 "disagree_frac": 3 / 14}


def test_launch_counts_per_call():
    """Kernels one call launches, by the kernel the dispatcher selects: the
    strip path a counter clear and the kernel; the row path with a
    workspace a counter clear, the row kernel and the second kernel for
    deferred rows; the warp-per-row and cluster kernels one."""
    b = _bench()
    assert b.calls_launches("strip_kernel") == 2
    assert b.calls_launches("row_cta_kernel") == 3
    assert b.calls_launches("row_kernel") == 1
    assert b.calls_launches("verify_kernel") == 1
