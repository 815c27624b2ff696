"""Pins of the oracle's launch-geometry rules (CPU only): the values the Module
attn_splitk page prints, and the invariants it states."""

import json
import os

import pytest

from oracle import policy as P

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "policy_worked_values.json")))


def test_worked_value_uncapped_auto():
    for case in GOLDEN["auto_uncapped"]:
        assert P.auto_splits_uncapped(case["sm_count"], case["num_q_heads"]) == case["splits"]
        # ... and the ceiling is what stops it
        assert P.auto_splits(case["sm_count"], case["num_q_heads"]) == P.MAX_DECODE_SPLITS


def test_worked_value_auto():
    for case in GOLDEN["auto"]:
        assert P.auto_splits(case["sm_count"], case["num_q_heads"]) == case["splits"]
        assert P.num_splits("auto", 0, case["sm_count"], case["num_q_heads"], 1, 1) == case["splits"]


def test_ceiling_admits_the_worked_auto_value():
    assert P.MAX_DECODE_SPLITS >= 13


def test_worked_value_pack_grid_fills_sms():
    for case in GOLDEN["gqa_pack_ctas_fill"]:
        n = case["first_num_seqs_that_fills"]
        assert P.gqa_pack_ctas(case["num_kv_heads"], n) >= case["sm_count"]
        assert P.gqa_pack_ctas(case["num_kv_heads"], n - 1) < case["sm_count"]


def test_pack_constants():
    assert P.DECODE_GQA_PACK_WIDTH == GOLDEN["pack_width"]["value"]
    assert P.DECODE_GQA_PACK_HEAD_DIM == GOLDEN["pack_head_dim"]["value"]


def test_legacy_rule_by_hand():
    # current_ctas = Hq * max(max_decode_seqs, num_seqs); >= SMs -> 1, else SMs // ctas
    assert P.num_splits("legacy", 0, 132, 1, 1, 1) == 132
    assert P.num_splits("legacy", 0, 132, 8, 2, 4) == 132 // 32
    assert P.num_splits("legacy", 0, 148, 24, 1, 0) == 6
    assert P.num_splits("legacy", 0, 148, 32, 5, 0) == 1     # 160 >= 148
    assert P.num_splits("legacy", 0, 148, 37, 4, 0) == 1     # exactly 148
    assert P.num_splits("legacy", 0, 148, 1, 1, 200) == 1    # max_decode_seqs dominates


def test_legacy_reads_the_batch_but_auto_and_pinned_do_not():
    sm, hq = 148, 8
    legacy = {P.num_splits("legacy", 0, sm, hq, s, 0) for s in range(1, 40)}
    assert len(legacy) > 1
    for pin in (0, 1, 3, 99):
        for pol in ("auto", "pinned"):
            vals = {P.num_splits(pol, pin, sm, hq, s, m) for s in range(1, 300, 7)
                    for m in (0, 1, 64, 512)}
            assert len(vals) == 1


def test_pinned_is_clamped():
    assert P.num_splits("pinned", 0, 148, 8, 1, 0) == 1
    assert P.num_splits("pinned", 1000, 148, 8, 1, 0) == P.MAX_DECODE_SPLITS
    assert P.num_splits("pinned", 5, 148, 8, 1, 0) == 5


def test_auto_sweep_bounds():
    for sm in (48, 132, 148, 152):
        for hq in range(1, 129):
            n = P.auto_splits(sm, hq)
            assert 1 <= n <= P.MAX_DECODE_SPLITS
            assert n == min(P.MAX_DECODE_SPLITS, -(-2 * sm // hq))


def test_workspace_formula():
    assert P.workspace_f32_values(1, 24, 128, 13) == 24 * 13 * 130
    assert P.workspace_f32_values(256, 32, 128, 10) * 4 == 42_598_400


def test_pack_shape_gate():
    assert P.gqa_pack_shape_ok(16, 2, 256)
    assert not P.gqa_pack_shape_ok(16, 2, 128)
    assert not P.gqa_pack_shape_ok(16, 4, 256)
    assert not P.gqa_pack_shape_ok(0, 0, 256)


@pytest.mark.parametrize("text,want", [
    ("legacy", ("legacy", 0)), (" AUTO ", ("auto", 0)), ("0", ("pinned", 1)),
    ("off", ("pinned", 1)), ("False", ("pinned", 1)), ("no", ("pinned", 1)),
    ("3", ("pinned", 3)), ("16", ("pinned", 16)), ("17", ("pinned", 16)),
    ("99999999999999999999", ("pinned", 16)), (" 007 ", ("pinned", 7)),
])
def test_parse_policy(text, want):
    assert P.parse_policy(text) == want


@pytest.mark.parametrize("text", ["", "  ", "-3", "+3", "3.0", "auto2", "yes", "0x10"])
def test_parse_policy_rejects(text):
    with pytest.raises(ValueError):
        P.parse_policy(text)


def test_parse_gqa_pack():
    for t in ("1", "on", " TRUE", "yes"):
        assert P.parse_gqa_pack(t) is True
    for t in ("0", "off", "false", "No "):
        assert P.parse_gqa_pack(t) is False
    with pytest.raises(ValueError):
        P.parse_gqa_pack("maybe")


@pytest.mark.parametrize("L", [0, 1, 15, 16, 17, 255, 256, 257, 2048, 2521, 32768, 16384])
@pytest.mark.parametrize("n", [1, 2, 3, 10, 13, 16])
def test_split_ranges_partition_the_sequence(L, n):
    rs = P.split_ranges(L, n, 16)
    assert len(rs) == n
    assert rs[0][0] == 0 and rs[-1][1] == L
    for (a, b), (c, d) in zip(rs, rs[1:]):
        assert b == c and a <= b
    chunk = P.split_chunk_tokens(L, n, 16)
    assert chunk % 16 == 0 and chunk >= P.MIN_KV_PER_SPLIT
    nonempty = [r for r in rs if r[1] > r[0]]
    for a, b in nonempty:
        assert a % 16 == 0
    for a, b in nonempty[:-1]:
        assert b - a == chunk


def test_long_context_split_geometry():
    # 32768 tokens in 13 splits: ceil(32768/13) = 2521 -> 2528 tokens (158 blocks)
    assert P.split_chunk_tokens(32768, 13, 16) == 2528
    rs = P.split_ranges(32768, 13, 16)
    assert rs[-1] == (12 * 2528, 32768)
