"""The kernels' division by a launch-invariant divisor (FastDiv in
csrc/pd_internal.h: multiply-high, add, shift, after Granlund and Montgomery,
"Division by invariant integers using multiplication", section 4) gives the
plain integer quotient, and the split geometry the kernels compute with it
equals split_chunk_tokens, the function the host ABI, the merge pass and the
policy tests use.  Host code only: compiled with the system C++ compiler."""

import os
import shutil
import subprocess

import pytest

from paged_kv_decode_splitk_gb300 import pd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_decode_splitk_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include "pd_internal.h"

using namespace pd;

static uint64_t state = 0x9e3779b97f4a7c15ull;
static uint32_t next_u32() {  // xorshift64*
    state ^= state >> 12; state ^= state << 25; state ^= state >> 27;
    return static_cast<uint32_t>((state * 0x2545f4914f6cdd1dull) >> 32);
}

static long long bad = 0, checked = 0;
static void check(int n, int d) {
    const FastDiv f = make_fastdiv(d);
    ++checked;
    if (fast_div(n, f) != n / d) {
        if (bad < 5) std::printf("mismatch %d / %d: %d vs %d\n", n, d, fast_div(n, f), n / d);
        ++bad;
    }
}

int main() {
    const int kMax = 0x7fffffff;
    // every divisor up to 4096 against the quotient boundaries k*d - 1, k*d
    // and the ends of the range
    for (int d = 1; d <= 4096; ++d) {
        for (long long k = 0; k * d <= kMax && k <= 4096; ++k) {
            const long long n = k * d;
            if (n - 1 >= 0) check(static_cast<int>(n - 1), d);
            check(static_cast<int>(n), d);
        }
        const long long top = (static_cast<long long>(kMax) / d) * d;
        check(static_cast<int>(top), d);
        if (top - 1 >= 0) check(static_cast<int>(top - 1), d);
        check(kMax, d);
        for (int i = 0; i < 64; ++i) check(static_cast<int>(next_u32() & 0x7fffffffu), d);
    }
    // powers of two and their neighbours, large primes, random divisors
    int special[] = {8191, 65521, 65536, 65537, 131071, 524287, 1048573, 16777213,
                     2147483629, 2147483647, 1073741824, 1073741823, 1073741825};
    for (int d : special)
        for (int i = 0; i < 20000; ++i) check(static_cast<int>(next_u32() & 0x7fffffffu), d);
    for (int j = 0; j < 2000; ++j) {
        const int d = static_cast<int>(next_u32() & 0x7fffffffu) | 1;
        for (int i = 0; i < 200; ++i) check(static_cast<int>(next_u32() & 0x7fffffffu), d);
        check(kMax, d);
        check(d - 1, d);
        check(d, d);
    }
    // the split geometry: every context length up to 70000 for the split
    // counts and block sizes the kernels take, and random long contexts
    long long gbad = 0, gchecked = 0;
    const int bss[] = {16, 32, 48, 64, 128, 256, 272};
    for (int n = 1; n <= 64; ++n)
        for (int bs : bss) {
            const FastDiv fn = make_fastdiv(n), fb = make_fastdiv(bs);
            for (int L = 0; L <= 70000; L += (L < 4096 ? 1 : 7)) {
                ++gchecked;
                if (split_chunk_tokens_fd(L, fn, fb, 256) != split_chunk_tokens(L, n, bs, 256)) ++gbad;
            }
            for (int i = 0; i < 2000; ++i) {
                const int L = static_cast<int>(next_u32() % 500000000u);
                ++gchecked;
                if (split_chunk_tokens_fd(L, fn, fb, 256) != split_chunk_tokens(L, n, bs, 256)) ++gbad;
            }
        }
    std::printf("div %lld %lld geom %lld %lld\n", checked, bad, gchecked, gbad);
    return 0;
}
"""


def _cuda_include() -> str | None:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return os.path.join(cand, "include")
    nvcc = shutil.which("nvcc")
    if nvcc:
        inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
        if os.path.exists(os.path.join(inc, "cuda_runtime.h")):
            return inc
    return None


def test_fast_division_equals_integer_division():
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("no C++ compiler or CUDA headers")
    d = os.path.join(os.path.dirname(pd.LIB_PATH), "fastdiv_test")
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "fastdiv.cc")
    exe = os.path.join(d, "fastdiv")
    with open(src, "w") as f:
        f.write(PROGRAM)
    subprocess.run([cxx, "-O2", "-std=c++17", f"-I{CSRC}", f"-I{inc}", src, "-o", exe], check=True,
                   capture_output=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    last = out.strip().splitlines()[-1].split()
    assert last[0] == "div" and last[3] == "geom", out
    checked, bad, gchecked, gbad = int(last[1]), int(last[2]), int(last[4]), int(last[5])
    assert checked > 10_000_000 and gchecked > 1_000_000, out
    assert bad == 0, out
    assert gbad == 0, out
