"""Host rules checked on the CPU (compiled with nvcc, run on the host, no GPU): the kernel's
shared-memory layout over every launch shape, the launcher's shape rule over the calls a GB300
context accepts, and the rule that keeps draw counters in call order across calls with and
without own outputs."""
import concurrent.futures
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


PROGRAMS = ("layout_check", "shape_check", "order_check")


def _compile(nvcc, out_dir, name):
    exe = str(out_dir / name)
    r = subprocess.run([nvcc, "-O1", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                        "-I", os.path.join(ROOT, "include"), "-o", exe, os.path.join(ROOT, "tests", name + ".cu")],
                       capture_output=True, text=True, timeout=900)
    return exe, r.returncode, r.stderr[-2000:]


@pytest.fixture(scope="module")
def programs(tmp_path_factory):
    """The three host programs, compiled side by side (each takes the library's whole source)."""
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    out_dir = tmp_path_factory.mktemp("host_rules")
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(PROGRAMS)) as ex:
        built = list(ex.map(lambda n: _compile(nvcc, out_dir, n), PROGRAMS))
    return dict(zip(PROGRAMS, built))


def _build_and_run(programs, name):
    exe, rc, err = programs[name]
    assert rc == 0, err
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
    assert " 0 bad" in r.stdout
    return r.stdout


def test_every_layout_is_aligned_and_fits(programs):
    _build_and_run(programs, "layout_check")


def test_every_accepted_call_gets_a_shape_that_fits(programs):
    """Every automatic shape fits; a forced split that cannot fit is refused with STRATA_ERANGE.
    (A bf16 row of 524,288 ids with a mask and a 4,096-id window under the concurrency hint is a
    shape whose one-block split does not fit: the rule splits such a row further.)"""
    out = _build_and_run(programs, "shape_check")
    assert "shapes" in out


def test_counters_stay_in_call_order_across_launch_kinds(programs):
    """Random streams of sampling and logprobs launches (PDL or not, early loads or not, own outputs
    or not) through the library's flag rule and an event model of programmatic dependent launch:
    every sampling call takes its counters after the one before it, and calls with own outputs
    still take theirs early when nothing before them takes counters late."""
    out = _build_and_run(programs, "order_check")
    assert "took counters early" in out
