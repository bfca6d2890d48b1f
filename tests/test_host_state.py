"""Host-side state of the library: per-device memos only, safe across threads.

The launchers keep no process-wide value that holds for one device alone
(an attribute set once, an SM count read once): anything memoised is keyed
by the device ordinal and held in atomics, so a process that drives several
GPUs, or calls from several threads, gets each device's own value.  The memo
itself is tested here on the host (plain C++, fake device ordinals, racing
threads); a scan of the sources checks that no other static state exists.
"""
import os
import re
import shutil
import subprocess

import pytest

from conftest import ROOT

CSRC = os.path.join(ROOT, "paged_kv_decode_store_gb300", "csrc")

MEMO_TEST = r"""
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>
#include "device_cache.h"

static pkvd::PerDeviceMemo<int> memo;
static pkvd::PerDeviceMemo<unsigned long long> wide;

int main() {
  // unknown devices read 0; out-of-range ordinals are ignored
  if (memo.get(0) != 0 || memo.get(-1) != 0 || memo.get(pkvd::kMaxDevicesCached) != 0) return 1;
  memo.put(-1, 5);
  memo.put(pkvd::kMaxDevicesCached, 5);
  if (memo.get(-1) != 0 || memo.get(pkvd::kMaxDevicesCached) != 0) return 2;
  // 16 threads race on every device's first lookup; each stores that
  // device's own value (device d -> 1000 + d), as a real query would
  std::vector<std::thread> ts;
  for (int t = 0; t < 16; ++t)
    ts.emplace_back([t] {
      for (int round = 0; round < 2000; ++round)
        for (int d = 0; d < pkvd::kMaxDevicesCached; ++d) {
          const int dev = (d + t) % pkvd::kMaxDevicesCached;
          const int v = memo.get(dev);
          if (v != 0 && v != 1000 + dev) std::abort();
          memo.put(dev, 1000 + dev);
          const unsigned long long w = (1ull << 40) | (unsigned long long)dev;
          const unsigned long long r = wide.get(dev);
          if (r != 0 && r != w) std::abort();      // a torn 64-bit word would show here
          wide.put(dev, w);
        }
    });
  for (auto& th : ts) th.join();
  for (int d = 0; d < pkvd::kMaxDevicesCached; ++d)
    if (memo.get(d) != 1000 + d || wide.get(d) != ((1ull << 40) | (unsigned long long)d)) return 3;
  std::puts("ok");
  return 0;
}
"""


def test_per_device_memo_under_racing_threads(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("needs g++")
    src = tmp_path / "memo.cpp"
    src.write_text(MEMO_TEST)
    exe = tmp_path / "memo"
    subprocess.run([cxx, "-std=c++17", "-O2", "-pthread", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)


# a declaration with static storage inside a function or class body:
# indented `static <type> <name>[...] (= | ; | {)`
STATIC_DECL = re.compile(r"^\s+static\s+[A-Za-z_][\w:<>, ]*\s+[A-Za-z_]\w*(\[[^\]]*\])*\s*(=|;|\{)")


def test_no_function_local_static_state():
    offenders = []
    for f in sorted(os.listdir(CSRC)):
        if not f.endswith((".cu", ".cuh", ".h", ".cpp")):
            continue
        for n, line in enumerate(open(os.path.join(CSRC, f)), 1):
            code = line.split("//")[0]
            if not STATIC_DECL.match(code) or "constexpr" in code:
                continue
            if "PerDeviceMemo<" in code or "std::atomic<" in code:
                continue                      # per-device, atomic memos are the allowed form
            offenders.append(f"{f}:{n}: {line.strip()}")
    assert not offenders, "\n".join(offenders)


def test_scan_catches_the_forms_it_forbids():
    """The pattern above matches the kinds of state it exists to keep out."""
    for bad in ["  static size_t configured = 0;", "  static int cache[64] = {0};",
                "    static bool tried = false;", "  static EncodeTiled fn = nullptr;"]:
        assert STATIC_DECL.match(bad), bad
    for ok in ["  static constexpr int kX = 3;", "  __device__ static float to_f(float x) { return x; }",
               "static int helper(int a) {", "  return static_cast<int>(x);"]:
        assert not (STATIC_DECL.match(ok) and "constexpr" not in ok), ok
