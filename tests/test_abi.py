"""CPU tests of the C ABI: the library loads, exports what include/pd.h
declares, and its host logic (policy, parsing, workspace sizing, argument
validation) agrees with the oracle's independent statement of the rules.
No call here launches a kernel."""

import ctypes
import os
import re
import subprocess
import sys

import pytest

from oracle import policy as P
from paged_kv_decode_splitk_gb300 import pd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    return pd.lib()


def test_library_exports_every_declared_symbol(L):
    syms = pd.header_symbols()
    assert len(syms) >= 28
    for s in syms:
        assert hasattr(L, s), s
    # ... and the binding wraps each of them under the same name
    for s in syms:
        assert s in pd._SIGS, s


def test_only_declared_symbols_are_exported():
    out = subprocess.run(["nm", "-D", "--defined-only", pd.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(pd.header_symbols())


def _header_defines():
    text = open(os.path.join(ROOT, "include", "pd.h")).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(PD_[A-Z0-9_]+)\s+\(?(-?\d+)\)?", text)}


def test_build_info_matches_header_kernels_and_oracle():
    """The kernels' compile-time pack width / head dim (their PD_GQA / PD_HDIM) equal the
    header's constants, which equal the oracle's (DECODE_GQA_PACK_WIDTH test idea)."""
    info = pd.pd_build_info()
    d = _header_defines()
    assert info["max_splits"] == d["PD_MAX_DECODE_SPLITS"] == P.MAX_DECODE_SPLITS
    assert info["pack_width"] == d["PD_GQA_PACK_WIDTH"] == P.DECODE_GQA_PACK_WIDTH
    assert info["pack_head_dim"] == d["PD_GQA_PACK_HEAD_DIM"] == P.DECODE_GQA_PACK_HEAD_DIM
    assert info["min_kv_per_split"] == d["PD_MIN_KV_PER_SPLIT"] == P.MIN_KV_PER_SPLIT
    assert d["PD_SPLITK_TARGET_WAVES"] == P.SPLITK_TARGET_WAVES


def test_kernel_source_defines_the_pack_width_the_host_dispatches_on():
    src = open(os.path.join(ROOT, "paged_kv_decode_splitk_gb300", "csrc", "pd_unit.cuh")).read()
    assert int(re.search(r"#define PD_GQA (\d+)", src).group(1)) == _header_defines()["PD_GQA_PACK_WIDTH"]
    assert int(re.search(r"#define PD_HDIM (\d+)", src).group(1)) == _header_defines()["PD_GQA_PACK_HEAD_DIM"]


def test_status_codes_match_binding():
    d = _header_defines()
    for name in ("PD_OK", "PD_NOT_APPLICABLE", "PD_ERR_INVALID", "PD_ERR_CAPACITY", "PD_ERR_WORKSPACE",
                 "PD_ERR_CUDA", "PD_ERR_ALLOC", "PD_ERR_UNSUPPORTED", "PD_DEV_BAD_BLOCK_ID",
                 "PD_DEV_BAD_CONTEXT_LEN", "PD_DEV_BAD_TILE_COUNT", "PD_DEV_WAIT_TIMEOUT"):
        assert getattr(pd, name) == d[name], name


@pytest.mark.parametrize("sm", [48, 132, 148, 152])
def test_policy_agrees_with_oracle(sm):
    for hq in list(range(1, 65)) + [96, 128]:
        for seqs in (1, 2, 3, 7, 17, 64, 256):
            for maxd in (0, 1, 64):
                for pol in ("legacy", "auto", "pinned"):
                    for pin in ((0,) if pol != "pinned" else (0, 1, 5, 16, 40)):
                        want = P.num_splits(pol, pin, sm, hq, seqs, maxd)
                        got = pd.pd_num_splits(pol, pin, sm, hq, seqs, maxd)
                        assert got == want, (pol, pin, sm, hq, seqs, maxd)
        assert pd.pd_auto_splits(sm, hq) == P.auto_splits(sm, hq)
        assert pd.pd_legacy_splits(sm, hq, 3) == P.legacy_splits(sm, hq, 3)


def test_policy_rejects_bad_arguments():
    with pytest.raises(pd.PdError):
        pd.pd_auto_splits(0, 8)
    with pytest.raises(pd.PdError):
        pd.pd_num_splits(7, 0, 148, 8, 1, 0)
    with pytest.raises(pd.PdError):
        pd.pd_legacy_splits(148, 0, 1)


PARSE_CASES = ["legacy", " AUTO ", "0", "off", "False", "no", "3", "16", "17", " 007 ",
               "99999999999999999999", "", " ", "-3", "+3", "3.0", "auto2", "yes", "0x10", "\tLegacy\n"]


@pytest.mark.parametrize("text", PARSE_CASES)
def test_parse_policy_agrees_with_oracle(text):
    names = {"legacy": pd.PD_POLICY_LEGACY, "auto": pd.PD_POLICY_AUTO, "pinned": pd.PD_POLICY_PINNED}
    try:
        want = P.parse_policy(text)
    except ValueError:
        with pytest.raises(pd.PdError):
            pd.pd_parse_policy(text)
        return
    assert pd.pd_parse_policy(text) == (names[want[0]], want[1])


@pytest.mark.parametrize("text", ["1", "on", " TRUE", "yes", "0", "off", "false", "No ", "maybe", ""])
def test_parse_gqa_pack_agrees_with_oracle(text):
    try:
        want = P.parse_gqa_pack(text)
    except ValueError:
        with pytest.raises(pd.PdError):
            pd.pd_parse_gqa_pack(text)
        return
    assert pd.pd_parse_gqa_pack(text) == want


def test_resolve_policy():
    assert pd.pd_resolve_policy("auto", None) == (pd.PD_POLICY_AUTO, 0)
    assert pd.pd_resolve_policy("auto", "4") == (pd.PD_POLICY_PINNED, 4)
    assert pd.pd_resolve_policy("auto", "bogus") == (pd.PD_POLICY_AUTO, 0)
    assert pd.pd_resolve_policy("bogus", None) == (pd.PD_POLICY_LEGACY, 0)
    assert pd.pd_resolve_policy(None, None) == (pd.PD_POLICY_LEGACY, 0)


def _run_child(code, env):
    e = dict(os.environ)
    e.update(env)
    e["PYTHONPATH"] = ROOT
    r = subprocess.run([sys.executable, "-c", code], env=e, capture_output=True, text=True, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    return r.stdout.strip()


def test_policy_from_env_reads_the_environment():
    code = ("from paged_kv_decode_splitk_gb300 import pd; import os; "
            "print(pd.pd_policy_from_env('auto')); os.environ['PD_ATTN_DECODE_SPLITK']='legacy'; "
            "print(pd.pd_policy_from_env('auto'))")
    out = _run_child(code, {"PD_ATTN_DECODE_SPLITK": " 5 "}).splitlines()
    assert out == ["(2, 5)", "(0, 0)"]


def test_gqa_pack_enabled_is_resolved_once():
    code = ("from paged_kv_decode_splitk_gb300 import pd; import os; a = pd.pd_gqa_pack_enabled(); "
            "os.environ['PD_ATTN_DECODE_GQA_PACK']='off'; print(a, pd.pd_gqa_pack_enabled())")
    assert _run_child(code, {"PD_ATTN_DECODE_GQA_PACK": "on"}) == "True True"
    assert _run_child(code.replace("'off'", "'on'"), {"PD_ATTN_DECODE_GQA_PACK": "nonsense"}) == "False False"


def test_workspace_bytes_agree_with_oracle():
    for rows in (1, 3, 256):
        for hq in (1, 4, 24, 32):
            for d in (8, 64, 128, 256):
                for n in (1, 2, 13, 16, 148):
                    assert pd.pd_workspace_bytes(rows, hq, d, n) == 4 * P.workspace_f32_values(rows, hq, d, n)
    assert pd.pd_workspace_bytes(0, 4, 64, 2) == 0


def test_pack_gate_and_ctas_agree_with_oracle():
    for hq in range(1, 40):
        for hkv in range(0, 6):
            for d in (128, 255, 256, 512):
                assert pd.pd_gqa_pack_shape_ok(hq, hkv, d) == P.gqa_pack_shape_ok(hq, hkv, d)
    assert pd.pd_gqa_pack_ctas(4, 12) == P.gqa_pack_ctas(4, 12) == 48


def test_split_chunk_agrees_with_oracle():
    for L in list(range(0, 600, 7)) + [2048, 2521, 4096, 16384, 32768, 100000]:
        for n in range(1, 17):
            for bs in (16, 32, 64):
                assert pd.pd_split_chunk_tokens(L, n, bs) == P.split_chunk_tokens(L, n, bs), (L, n, bs)


# ---- argument validation that happens before any CUDA call ----------------------------

def _call(L, **kw):
    a = dict(q=16, k=16, v=16, bt=16, maxb=4, cl=16, out=16, S=1, Hq=8, Hkv=2, D=128, bs=16, nb=8,
             scale=0.1, N=1, ws=None, wsb=0, pack=0)
    a.update(kw)
    P_ = ctypes.c_void_p
    return L.pd_decode_attn(P_(a["q"]), P_(a["k"]), P_(a["v"]), P_(a["bt"]), a["maxb"], P_(a["cl"]),
                            P_(a["out"]), a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["nb"],
                            a["scale"], a["N"], P_(a["ws"]) if a["ws"] else None, a["wsb"], a["pack"],
                            None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=6, Hkv=4), pd.PD_ERR_INVALID),
    (dict(Hkv=0), pd.PD_ERR_INVALID),
    (dict(D=300), pd.PD_ERR_INVALID),
    (dict(D=12), pd.PD_ERR_UNSUPPORTED),
    (dict(bs=8), pd.PD_ERR_UNSUPPORTED),
    (dict(bs=24), pd.PD_ERR_UNSUPPORTED),
    (dict(N=0), pd.PD_ERR_INVALID),
    (dict(S=-1), pd.PD_ERR_INVALID),
    (dict(scale=float("nan")), pd.PD_ERR_INVALID),
    (dict(q=0), pd.PD_ERR_INVALID),
    (dict(q=18), pd.PD_ERR_INVALID),            # misaligned
    (dict(maxb=0), pd.PD_ERR_INVALID),
    (dict(N=2), pd.PD_ERR_WORKSPACE),           # no workspace
    (dict(N=2, ws=16, wsb=100), pd.PD_ERR_WORKSPACE),
    (dict(pack=1), pd.PD_NOT_APPLICABLE),       # 8/2 heads at D=128: not the packed shape
    (dict(pack=1, Hq=16, Hkv=2, D=256, N=2), pd.PD_NOT_APPLICABLE),
    (dict(pack=2), pd.PD_NOT_APPLICABLE),       # the split-K packed mode keeps the shape gate
    (dict(pack=3), pd.PD_ERR_INVALID),
    (dict(pack=-1), pd.PD_ERR_INVALID),
])
def test_decode_attn_rejects(L, kw, code):
    assert _call(L, **kw) == code
    if code != pd.PD_OK:
        assert pd.last_error() != ""


def _call_fp8(L, ks=1.0, vs=1.0, **kw):
    a = dict(q=16, k=16, v=16, bt=16, maxb=4, cl=16, out=16, S=1, Hq=8, Hkv=2, D=128, bs=16, nb=8,
             scale=0.1, N=1, ws=None, wsb=0, pack=0)
    a.update(kw)
    P_ = ctypes.c_void_p
    return L.pd_decode_attn_fp8(P_(a["q"]), P_(a["k"]), P_(a["v"]), ks, vs, P_(a["bt"]), a["maxb"],
                                P_(a["cl"]), P_(a["out"]), a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["nb"],
                                a["scale"], a["N"], P_(a["ws"]) if a["ws"] else None, a["wsb"], a["pack"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=40), pd.PD_ERR_UNSUPPORTED),        # an FP8 row must be a whole number of 16-byte chunks
    (dict(ks=float("inf")), pd.PD_ERR_INVALID),
    (dict(vs=float("nan")), pd.PD_ERR_INVALID),
    (dict(Hq=6, Hkv=4), pd.PD_ERR_INVALID),
    (dict(N=2), pd.PD_ERR_WORKSPACE),
    (dict(pack=1), pd.PD_NOT_APPLICABLE),
])
def test_decode_attn_fp8_rejects(L, kw, code):
    assert _call_fp8(L, **kw) == code
    assert pd.last_error() != ""


def test_zero_sequences_is_a_no_op(L):
    assert _call(L, S=0, q=0, k=0, v=0) == pd.PD_OK


@pytest.mark.parametrize("dims,code", [
    ((4, 6, 4, 64, 16, 8), pd.PD_ERR_INVALID),
    ((4, 8, 0, 64, 16, 8), pd.PD_ERR_INVALID),
    ((4, 8, 2, 512, 16, 8), pd.PD_ERR_INVALID),
    ((4, 8, 2, 60, 16, 8), pd.PD_ERR_UNSUPPORTED),
    ((4, 8, 2, 64, 12, 8), pd.PD_ERR_UNSUPPORTED),
    ((-1, 8, 2, 64, 16, 8), pd.PD_ERR_INVALID),
    ((4, 8, 2, 64, 16, 8), pd.PD_OK),
])
def test_tiled_validate(dims, code):
    d = pd.pd_tiled_dims(*dims)
    assert pd.lib().pd_tiled_validate(ctypes.byref(d)) == code


def test_tiled_state_bytes_follow_the_dims_formula():
    d = pd.pd_tiled_dims(64, 16, 4, 256, 16, 64)
    b = pd.pd_tiled_state_bytes(d)
    assert b == {"m": 64 * 16 * 4, "l": 64 * 16 * 4, "o": 64 * 16 * 256 * 4, "output": 64 * 16 * 256 * 2}


def test_tiled_create_rejects_bad_dims_without_cuda():
    d = pd.pd_tiled_dims(4, 6, 4, 64, 16, 8)
    with pytest.raises(pd.PdError) as e:
        pd.pd_tiled_create(d)
    assert e.value.code == pd.PD_ERR_INVALID
