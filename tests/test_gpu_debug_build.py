"""The bounds-checked build (libcsa2_debug.so, compiled with CSA2_DEBUG):
it builds, loads in place of libcsa2.so when CSA2_DEBUG=1, raises no
bounds error on valid decode / Reindex / prefill cases whose results match
the oracle, and still reports an index past a sequence (tests/_debug_run.py,
run in a child process so that this process keeps the normal library)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_runs_clean():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "csa2_build", os.path.join(ROOT, "fp4_kv_cache_index_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    assert b.build(debug=True).endswith("libcsa2_debug.so")
    env = dict(os.environ, CSA2_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_debug_run.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "all cases clean" in r.stdout
