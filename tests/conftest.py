import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Print every GPU-vs-oracle comparison of the run: rows and elements compared, error
    maxima, and the count of O elements under the one-BF16-ulp rule for |O| >= 4 (with how
    many of them were more than 1.5e-2 off)."""
    log = []  # the helper module may be imported under two names
    for name in ("tests.gpu_util", "gpu_util"):
        log += getattr(sys.modules.get(name), "PARITY_LOG", [])
    if not log:
        return
    tr = terminalreporter
    tr.section("parity against the oracle")
    tr.write_line(f"{'test':<78} {'rows':>10} {'o_max':>9} {'o_mean':>9} {'lse_max':>9} {'|O|>=4':>7} {'>1.5e-2':>7}")
    for name, st in log:
        tr.write_line(f"{name[-78:]:<78} {st['n_rows']:>10} {st['o_max']:>9.2e} {st['o_mean']:>9.2e} "
                      f"{st['lse_max']:>9.2e} {st['n_ulp_rule']:>7} {st['n_over_literal']:>7}")
