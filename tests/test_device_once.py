"""Per-device set-up bookkeeping (csrc/device_once.h) on the CPU: the kernel
launchers raise each kernel's shared-memory limit once per device, because a
function attribute applies only to the device that was current when it was
set.  The header has no CUDA types, so it is compiled here with g++ alone."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_sm_flashattention_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "device_once.h"

static fa::DeviceOnceFlags flags;
static int calls[fa::kMaxFlagDevices];
static int fail_next = 0;

static int setup_on(int dev) {
  return fa::once_per_device(flags, dev, [dev] {
    ++calls[dev];
    if (fail_next) { fail_next = 0; return -7; }
    return 0;
  });
}

int main() {
  int rc = 0;
  // first launch on device 0 sets up, later ones do not
  rc |= setup_on(0); rc |= setup_on(0); rc |= setup_on(0);
  // a second device needs its own set-up
  rc |= setup_on(1); rc |= setup_on(1);
  // a failed set-up reports its code, leaves the flag clear and is retried
  fail_next = 1;
  const int failed = setup_on(5);
  rc |= setup_on(5); rc |= setup_on(5);
  // device indices outside the table are refused without running set-up
  const int out_lo = setup_on(-1), out_hi = setup_on(fa::kMaxFlagDevices);
  std::printf("%d %d %d %d %d %d %d %d\n", rc, calls[0], calls[1], calls[5], failed, out_lo, out_hi, calls[2]);
  return 0;
}
"""


def test_once_per_device(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "once.cc"
    exe = tmp_path / "once"
    src.write_text(PROGRAM)
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    rc, c0, c1, c5, failed, out_lo, out_hi, c2 = map(int, out)
    assert rc == 0
    assert (c0, c1, c2) == (1, 1, 0)
    assert failed == -7 and c5 == 2
    assert out_lo == -1 and out_hi == -1
