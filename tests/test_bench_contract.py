"""bench.py's host-side pieces run without a GPU: the module imports, the
source hash the recorded ncu traffic is keyed on is computable, and the
recorded entry names a kernel the step launches."""
import importlib.util
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_bench_imports_and_hashes():
    b = _bench()
    h = b.src_hash("grads")
    assert re.fullmatch(r"[0-9a-f]{16}", h)
    for name, rec in b.NCU_TRAFFIC.items():
        assert name in b.KERNEL_NAMES.values()
        assert re.fullmatch(r"[0-9a-f]{16}", rec["sha"]) and rec["bytes_per_launch"] > 0
    assert b.LAUNCHES_PER_STEP == len(b.PHASES)
