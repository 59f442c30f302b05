"""Without the built library every entry point fails loudly (ImportError);
nothing falls back to a CPU path (CPU only)."""
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "selective_state_space_113_b300"

PROBE = r"""
import selective_state_space_113_b300 as ssm
from selective_state_space_113_b300 import workloads            # usable without the library
for name in ("ssm_scan_fwd", "ssm_scan_bwd", "ssm_ssd_fwd", "ssm_step", "scan"):
    try:
        f = getattr(ssm, name)
        if name == "scan":
            f(None, None, None, None, None, None)
    except ImportError as e:
        assert "not built" in str(e), e
        print("refused", name)
    else:
        raise SystemExit(f"{name} did not fail without the library")
"""


def test_entry_points_fail_without_the_library(tmp_path):
    dst = tmp_path / PKG
    shutil.copytree(os.path.join(ROOT, PKG), dst,
                    ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc"))
    assert not any(p.suffix == ".so" for p in dst.iterdir())
    r = subprocess.run([sys.executable, "-c", PROBE], cwd=tmp_path, capture_output=True,
                       text=True, timeout=300, env=dict(os.environ, PYTHONPATH=str(tmp_path)))
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("refused") == 5
