"""The library's debug build: index checks in the kernels and guard bytes around every workspace
buffer, the stand-ins for a memory checker.  The build is made here (build.py --debug) and the
cases of tests/_debug_cases.py run against it in a child process (the binding loads one build
per process): small parity cases through every kernel path with no damaged guard and no failed
check, and a planted overflow that the check finds."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_debug_build_cases():
    import importlib.util
    spec = importlib.util.spec_from_file_location("dg_build_script",
                                                  os.path.join(ROOT, "uniform_state_discrete_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(debug=True)
    env = dict(os.environ, DG_LIBRARY="debug")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_debug_cases.py")], env=env,
                         capture_output=True, text=True, timeout=900)
    print(out.stdout[-4000:])
    assert out.returncode == 0, out.stderr[-4000:]
    assert "debug cases ok" in out.stdout
