"""Launch-geometry policy of paged-decode attention, restated for the oracle.

TEST INFRASTRUCTURE ONLY: the product library carries its own implementation
of these rules; this module exists so that tests can check it against a
second, independent statement written from the pages.  Nothing on the product
path imports it.

Every rule below cites the item of the "Module attn_splitk" documentation page
(metrale_kernels::attn_splitk) that states it.
"""

from __future__ import annotations

# "MAX_DECODE_SPLITS" item: the ceiling on the split count under every policy
# but Legacy.  The page does not print its value; it implies at least 13
# (auto asks for 13 at 24 q heads on 148 SMs and the count is clamped to the
# ceiling).  Reading: 16.
MAX_DECODE_SPLITS = 16

# "SPLITK_TARGET_WAVES" item: waves of CTAs Auto aims for; the
# MAX_DECODE_SPLITS item's "2 * sm_count / num_q_heads" fixes it at 2.
SPLITK_TARGET_WAVES = 2

# "DECODE_GQA_PACK_WIDTH" item (the kernels' PD_GQA) and
# "DECODE_GQA_PACK_HEAD_DIM" item (the kernels' PD_HDIM).
DECODE_GQA_PACK_WIDTH = 8
DECODE_GQA_PACK_HEAD_DIM = 256

# Module description: each sequence's split size is floored at
# PD_MIN_KV_PER_SPLIT tokens computed from its own length.  The value is not
# printed.  Reading: 256 tokens, chunks rounded up to whole cache blocks.
MIN_KV_PER_SPLIT = 256

POLICY_LEGACY = "legacy"
POLICY_AUTO = "auto"
POLICY_PINNED = "pinned"


def split_ref_seqs(num_seqs: int, max_decode_seqs: int) -> int:
    """"legacy_splits" item: the reference batch is max(max_decode_seqs, num_seqs)."""
    return max(max_decode_seqs, num_seqs)


def legacy_splits(sm_count: int, num_q_heads: int, ref_seqs: int) -> int:
    """Module description, the SplitkPolicy::Legacy rule.

    current_ctas = num_q_heads * ref_seqs; one split when that already fills
    the SMs, else NUM_SMS / current_ctas by integer division.  Not clamped.
    """
    current_ctas = num_q_heads * ref_seqs
    if current_ctas >= sm_count:
        return 1
    return sm_count // current_ctas


def auto_splits_uncapped(sm_count: int, num_q_heads: int) -> int:
    """ceil(WAVES * sm_count / num_q_heads), before the clamp ("MAX_DECODE_SPLITS" item)."""
    return -(-(SPLITK_TARGET_WAVES * sm_count) // num_q_heads)


def auto_splits(sm_count: int, num_q_heads: int) -> int:
    """"auto_splits" item: clamp(ceil(WAVES*sm_count/num_q_heads), 1, MAX_DECODE_SPLITS)."""
    return min(max(auto_splits_uncapped(sm_count, num_q_heads), 1), MAX_DECODE_SPLITS)


def num_splits(policy: str, pin: int, sm_count: int, num_q_heads: int, num_seqs: int,
               max_decode_seqs: int) -> int:
    """"num_splits" item: the split count for a launch.

    Auto and Pinned read only (sm_count, num_q_heads) and the pin (module
    invariants); Legacy reads the reference batch.  A pinned count is clamped
    to 1..MAX_DECODE_SPLITS ("MAX_DECODE_SPLITS" and "parse" items).
    """
    if policy == POLICY_LEGACY:
        return legacy_splits(sm_count, num_q_heads, split_ref_seqs(num_seqs, max_decode_seqs))
    if policy == POLICY_AUTO:
        return auto_splits(sm_count, num_q_heads)
    if policy == POLICY_PINNED:
        return min(max(pin, 1), MAX_DECODE_SPLITS)
    raise ValueError(f"unknown policy {policy!r}")


def workspace_f32_values(rows: int, num_q_heads: int, head_dim: int, num_splits_: int) -> int:
    """"MAX_DECODE_SPLITS" item: rows * num_q_heads * num_splits * (head_dim + 2) F32 values,
    one [o[head_dim], m, l] slot ("workspace_slots" item) per (row, q head, split)."""
    return rows * num_q_heads * num_splits_ * (head_dim + 2)


def gqa_pack_shape_ok(num_q_heads: int, num_kv_heads: int, head_dim: int) -> bool:
    """Module invariants / "gqa_pack_shape_ok" item: only
    num_q_heads == num_kv_heads * PACK_WIDTH at head_dim == PACK_HEAD_DIM.
    Reading: num_kv_heads must also be positive (the page's list is cut off)."""
    return (num_kv_heads > 0 and num_q_heads == num_kv_heads * DECODE_GQA_PACK_WIDTH
            and head_dim == DECODE_GQA_PACK_HEAD_DIM)


def gqa_pack_ctas(num_kv_heads: int, num_seqs: int) -> int:
    """"gqa_pack_ctas" item: a packed launch puts num_kv_heads * num_seqs CTAs on the device."""
    return num_kv_heads * num_seqs


_OFF_WORDS = ("0", "off", "false", "no")


def parse_policy(text: str) -> tuple[str, int]:
    """"parse" item: legacy | auto | 0/off/false/no | a decimal count clamped to 1..MAX,
    trimmed and case-insensitive.  Returns (policy, pin); raises ValueError.

    Reading: the off words mean split-K off, i.e. Pinned(1).
    """
    word = text.strip().lower()
    if word == "legacy":
        return POLICY_LEGACY, 0
    if word == "auto":
        return POLICY_AUTO, 0
    if word in _OFF_WORDS:
        return POLICY_PINNED, 1
    if word and all(c in "0123456789" for c in word):
        return POLICY_PINNED, min(max(int(word), 1), MAX_DECODE_SPLITS)
    raise ValueError(f"not a split-K policy: {text!r}")


def parse_gqa_pack(text: str) -> bool:
    """"parse_gqa_pack" item: 1/on/true/yes | 0/off/false/no, trimmed, case-insensitive."""
    word = text.strip().lower()
    if word in ("1", "on", "true", "yes"):
        return True
    if word in _OFF_WORDS:
        return False
    raise ValueError(f"not a GQA-pack switch: {text!r}")


def split_chunk_tokens(context_len: int, num_splits_: int, block_size: int,
                       min_kv_per_split: int = MIN_KV_PER_SPLIT) -> int:
    """Tokens per split for one sequence (module description: the split size is
    floored at PD_MIN_KV_PER_SPLIT from the sequence's own length).

    Reading: chunk = roundup(max(ceil(L / N), MIN_KV_PER_SPLIT), block_size);
    split i covers [i*chunk, min((i+1)*chunk, L)), possibly empty.
    """
    per = -(-context_len // num_splits_) if context_len > 0 else 0
    c = max(per, min_kv_per_split)
    return -(-c // block_size) * block_size


def split_ranges(context_len: int, num_splits_: int, block_size: int,
                 min_kv_per_split: int = MIN_KV_PER_SPLIT) -> list[tuple[int, int]]:
    """The token range of every split of one sequence, empty ones included."""
    chunk = split_chunk_tokens(context_len, num_splits_, block_size, min_kv_per_split)
    out = []
    for i in range(num_splits_):
        a = min(i * chunk, context_len)
        b = min((i + 1) * chunk, context_len)
        out.append((a, b))
    return out


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


