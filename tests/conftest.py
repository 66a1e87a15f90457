import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libftmoe")


def pytest_terminal_summary(terminalreporter):
    """Counts of every output comparison of the session: elements outside the stated
    tolerance, those carried by the re-quantization allowance, and measured errors against
    the bounds the tests hold them to."""
    log = sys.modules.get("_ftmoe_check_log")
    if log is None or not (log.checks or log.measures):
        return
    tr = terminalreporter
    tr.section("output checks (stated tolerance 2e-2 |ref| + 1e-3 max|ref|)")
    tot_n = tot_out = tot_carried = 0
    for c in log.checks:
        tot_n += c["n"]
        tot_out += c["outside_tolerance"]
        tot_carried += c["carried_by_allowance"]
        tr.write_line(f"{c['test']} | {c['what']}: {c['n']} elements, {c['outside_tolerance']} outside the "
                      f"tolerance, {c['carried_by_allowance']} carried by the re-quantization allowance "
                      f"(max |err|/tol {c['max_err_over_tol_carried']:.3f}), {c['failing']} failing")
    tr.write_line(f"total: {tot_n} elements in {len(log.checks)} checks, {tot_out} outside the stated "
                  f"tolerance, {tot_carried} carried by the allowance")
    for m in log.measures:
        tr.write_line(f"{m['test']} | {m['what']}: measured {m['value']:.4g}, bound {m['bound']:.4g}")
