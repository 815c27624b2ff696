"""The C boundary from C: include/pd.h compiles as strict C99 on its own, and
a C program linked against libpd.so gets from the host entry points (policy,
parsing, workspace size, pack gate, split chunks, build constants) what the
oracle's own statement of the rules gives.  No kernel is launched, so no GPU
is needed."""

import os
import shutil
import subprocess

import pytest

from oracle import policy as P
from paged_kv_decode_splitk_gb300 import pd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "pd.h"

int main(void) {
    int ms = 0, pw = 0, phd = 0, mkv = 0, pol = -1, pin = -1, s, h, n;
    const char *words[] = {"auto", "legacy", "off", "7", " 40 ", "bogus"};
    if (pd_build_info(&ms, &pw, &phd, &mkv) != PD_OK) return 1;
    printf("build %d %d %d %d\n", ms, pw, phd, mkv);
    for (s = 0; s < 6; ++s) {
        int rc = pd_parse_policy(words[s], &pol, &pin);
        printf("parse %d %d %d\n", rc, rc == PD_OK ? pol : -9, rc == PD_OK ? pin : -9);
    }
    for (s = 0; s < 3; ++s)
        for (h = 1; h <= 64; h *= 2)
            printf("splits %d %d %d\n", pd_num_splits(s, 5, 148, h, 12, 32), s, h);
    printf("ws %zu\n", pd_workspace_bytes(256, 32, 128, 10));
    printf("pack %d %d %d\n", pd_gqa_pack_shape_ok(16, 2, 256), pd_gqa_pack_shape_ok(16, 2, 128),
           pd_gqa_pack_shape_ok(24, 2, 256));
    for (n = 1; n <= 16; n *= 2) printf("chunk %d %d\n", n, pd_split_chunk_tokens(32768, n, 16));
    printf("last '%s'\n", pd_last_error() ? "ok" : "null");
    return 0;
}
"""


def _scratch() -> str:
    # beside the built library (an ignored build folder of the repository)
    d = os.path.join(os.path.dirname(pd.LIB_PATH), "c_abi_test")
    os.makedirs(d, exist_ok=True)
    return d


@pytest.fixture(scope="module")
def built():
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = pd.LIB_PATH
    pd.lib()  # the library exists and loads
    d = _scratch()
    src = os.path.join(d, "use_pd.c")
    with open(src, "w") as f:
        f.write(PROGRAM)
    exe = os.path.join(d, "use_pd")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           src, "-o", exe, lib, f"-Wl,-rpath,{os.path.dirname(lib)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_compiles_alone_as_strict_c99():
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = os.path.join(_scratch(), "only_header.c")
    with open(src, "w") as f:
        f.write('#include "pd.h"\nint main(void) { return PD_OK; }\n')
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), src], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_agrees_with_the_oracle_rules(built):
    out = subprocess.run([built], capture_output=True, text=True, check=True).stdout.splitlines()
    lines = [l.split() for l in out]
    build = [l for l in lines if l[0] == "build"][0]
    assert [int(x) for x in build[1:]] == [P.MAX_DECODE_SPLITS, P.DECODE_GQA_PACK_WIDTH,
                                           P.DECODE_GQA_PACK_HEAD_DIM, P.MIN_KV_PER_SPLIT]
    names = {pd.PD_POLICY_LEGACY: P.POLICY_LEGACY, pd.PD_POLICY_AUTO: P.POLICY_AUTO,
             pd.PD_POLICY_PINNED: P.POLICY_PINNED}
    words = ["auto", "legacy", "off", "7", " 40 ", "bogus"]
    for w, l in zip(words, [l for l in lines if l[0] == "parse"]):
        rc, pol, pin = (int(x) for x in l[1:])
        try:
            want = P.parse_policy(w)
        except ValueError:
            want = None
        if want is None:
            assert rc == pd.PD_ERR_INVALID, w
        else:
            assert rc == pd.PD_OK and (names[pol], pin) == want, (w, pol, pin, want)
    for l in [l for l in lines if l[0] == "splits"]:
        n, s, h = (int(x) for x in l[1:])
        assert n == P.num_splits(names[s], 5, 148, h, 12, 32), (s, h, n)
    ws = int([l for l in lines if l[0] == "ws"][0][1])
    assert ws == P.workspace_f32_values(256, 32, 128, 10) * 4
    pack = [int(x) for x in [l for l in lines if l[0] == "pack"][0][1:]]
    assert pack == [int(P.gqa_pack_shape_ok(16, 2, 256)), int(P.gqa_pack_shape_ok(16, 2, 128)),
                    int(P.gqa_pack_shape_ok(24, 2, 256))]
    for l in [l for l in lines if l[0] == "chunk"]:
        n, c = int(l[1]), int(l[2])
        assert c == P.split_chunk_tokens(32768, n, 16), (n, c)
