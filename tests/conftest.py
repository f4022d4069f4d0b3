"""pytest configuration: registers the ``gpu`` marker, puts the repo root on
sys.path, and reports the GPU parity margins at the end of the session."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """One line per attention parity check: the largest |out err| (below 8
    and at 8 or more), the share of the bound it used, and the largest
    |lse err|.  Shown even under -q; also written as JSON to the file that
    KV4_PARITY_LOG names."""
    gc = sys.modules.get("gpu_common")
    records = getattr(gc, "PARITY_RECORDS", None) if gc is not None else None
    if not records:
        return
    tr = terminalreporter
    tr.section("attention parity vs the oracle (bound: 2e-2, + half a bf16 ulp at |out| >= 8; "
               "lse 1e-3)")
    for r in records:
        tr.write_line(f"  {r['case'][:48]:48s} out<8 {r['max_out_err_below_8']:.4f}  "
                      f"out>=8 {r['max_out_err_at_8_and_above']:.4f}  "
                      f"share {r['max_share_of_out_bound']:.3f}  lse {r['max_lse_err']:.2e}")
    worst = max(r["max_share_of_out_bound"] for r in records)
    worst_lse = max(r["share_of_lse_bound"] for r in records)
    tr.write_line(f"{len(records)} parity checks; largest share of the out bound {worst:.3f}, "
                  f"of the lse bound {worst_lse:.3f}")
    path = os.environ.get("KV4_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump(records, f, indent=1)
