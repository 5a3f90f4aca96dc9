import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """Near-tie rows per test: how many rows each parity comparison found within 1e-6 of a
    race or top-p tie, and how many of those differed from the oracle's choice and were
    accepted on validity against the definition instead."""
    parity = sys.modules.get("parity")
    log = getattr(parity, "NEAR_LOG", None)
    if not log:
        return
    per = {}
    for test, _label, rows, near, acc in log:
        t = per.setdefault(test, [0, 0, 0, 0])
        t[0] += 1
        t[1] += rows
        t[2] += near
        t[3] += acc
    tr = terminalreporter
    tr.section("near-tie rows (compared / near a tie / accepted on validity)")
    for test, (calls, rows, near, acc) in sorted(per.items()):
        tr.write_line(f"{test}: {calls} comparisons, {rows} rows, {near} near, {acc} accepted")
    tot = [sum(v[i] for v in per.values()) for i in range(4)]
    tr.write_line(f"total: {tot[0]} comparisons, {tot[1]} rows, {tot[2]} near, {tot[3]} accepted")
    # with KPS_NEAR_LOG set, every comparison is also written there, one JSON object a line
    path = os.environ.get("KPS_NEAR_LOG")
    if path:
        import json
        with open(path, "a") as f:
            for test, label, rows, near, acc in log:
                f.write(json.dumps({"test": test, "label": label, "rows": rows, "near": near, "accepted": acc}) + "\n")
