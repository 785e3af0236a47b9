"""Decode steps driven from plain C with host buffers (tests/c_abi/e2e_step.c):
the C ABI used the way a serving loop written in C uses it, with the
library's host time per call measured apart from any Python binding."""

import json
import subprocess

import pytest

from paged_kv_decode_08_gb300 import build


def test_c_driver_compiles_and_links():
    pytest.importorskip("torch")
    try:
        exe = build.build_c_e2e(force=True)
    except RuntimeError as e:
        if "no C compiler" in str(e):
            pytest.skip(str(e))
        raise
    assert exe.endswith("e2e_step")


@pytest.mark.gpu
def test_c_driver_runs_decode_steps_from_host_buffers(cuda_device):
    exe = build.build_c_e2e()
    r = subprocess.run([exe, "50", "5"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["splits"] == 1
    assert 0 < d["host_us_per_call_median"] < 1000
    assert d["e2e_us_per_step"] > 0 and d["wall_us_per_step_median"] > 0
