"""pd_decode_attn_noalloc: the entry point for callers that cannot allocate
device memory on the decode path (their memory is reserved up front by their
own allocator, or cudaMalloc's synchronisation is not acceptable there).  Its
split-K workspace is a fixed array inside the library, shared by every call.

These tests call it through the C ABI and check it against pd_decode_attn,
which takes a caller workspace, bit for bit (the same kernels run on the same
inputs), on different launches in a row, so each call after the first runs on
whatever the one before left in the shared array; the oracle checks the
values as well.  This file is collected last on purpose; it passes alone in
a fresh process as well.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_splitk_gb300 import api, pd
from paged_kv_decode_splitk_gb300 import workloads as W

from helpers import assert_within_tolerance

pytestmark = pytest.mark.gpu

NOALLOC_LIMIT = 16 * 1024 * 1024  # PD_NOALLOC_WORKSPACE_BYTES


def _both(w, device, num_splits, gqa_pack=0):
    """Run the same launch through pd_decode_attn (caller workspace) and
    pd_decode_attn_noalloc; returns both outputs as BF16 tensors."""
    inp = api.PagedInputs(w, device)
    shape = (w.num_seqs, w.num_q_heads, w.head_dim)
    ref = torch.full(shape, 9.0, dtype=torch.bfloat16, device=device)
    got = torch.full(shape, -9.0, dtype=torch.bfloat16, device=device)
    ws = api.workspace(w.num_seqs, w.num_q_heads, w.head_dim, num_splits, device)
    assert pd.pd_decode_attn(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, ref,
                             w.inv_sqrt_d, num_splits, ws, gqa_pack) == pd.PD_OK
    assert pd.pd_decode_attn_noalloc(inp.q, inp.k, inp.v, inp.block_table, inp.context_lens, got,
                                     w.inv_sqrt_d, num_splits, gqa_pack) == pd.PD_OK
    torch.cuda.synchronize()
    assert pd.pd_device_status() == 0
    return got, ref


def test_noalloc_matches_the_caller_workspace_entry_point_on_two_calls(cuda_device):
    # Both entry points run the same kernels with the same split geometry, so
    # their outputs agree bit for bit; the second case runs on whatever the
    # first one left in the shared array.
    cases = [
        # 13 splits over head dim 128 (the long-context shape class), ragged lengths
        (W.custom([300, 4100, 17, 0, 2500], 24, 8, 128, seed=61), 13, 0),
        # then a different shape: head dim 256, 4 splits
        (W.custom([1000, 3000, 16], 16, 2, 256, seed=62), 4, 0),
        # then the packed pass with splits (gqa_pack 2): 8 query heads per KV head
        (W.custom([0, 700, 4097, 33], 16, 2, 256, seed=63), 5, pd.PD_GQA_PACK_SPLITK),
    ]
    for w, n, pack in cases:
        need = pd.pd_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim, n)
        assert 0 < need <= NOALLOC_LIMIT
        got, ref = _both(w, cuda_device, n, pack)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), \
            f"noalloc differs from the caller-workspace call (N={n}, gqa_pack={pack})"
        exact = oracle.decode_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens,
                                   w.inv_sqrt_d)
        assert_within_tolerance(api.bf16_to_f64(got), exact, f"noalloc vs oracle, N={n}, gqa_pack={pack}")


def test_noalloc_single_split_needs_no_workspace(cuda_device):
    w = W.tiny(pin=1)
    got, ref = _both(w, cuda_device, 1)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_a_workspace_beyond_its_limit(cuda_device):
    # 256 sequences x 32 heads x 16 splits x (128 + 2) floats = 68 MB > 16 MiB:
    # refused before anything is touched (the pointers below are never used)
    L = pd.lib()
    fake = ctypes.c_void_p(256)
    rc = L.pd_decode_attn_noalloc(fake, fake, fake, fake, 64, fake, fake, 256, 32, 8, 128, 16, 4096,
                                  0.088, 16, 0, None)
    assert rc == pd.PD_ERR_WORKSPACE
    assert "16777216" in pd.last_error()
