import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


def pytest_terminal_summary(terminalreporter):
    """How many compared heads each tolerance exemption took, per workload
    (policy: an oracle mass within 1e-5 of T; top-k: an oracle top-k gap
    within 1e-5 relative)."""
    mod = sys.modules.get("parity_util")
    reports = getattr(mod, "REPORTS", None) if mod else None
    if not reports:
        return
    terminalreporter.write_sep("-", "parity exemptions per workload")
    for name, rep in reports:
        if rep["checked"]:
            terminalreporter.write_line(
                f"{name}: {rep['checked']} heads compared, {rep['decode_checked']} decoded, "
                f"policy-exempt {rep['policy_exempt']}, top-k-exempt {rep['topk_exempt']}")
