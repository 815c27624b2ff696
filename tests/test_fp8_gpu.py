"""FP8 E4M3 KV cache (Module attn_splitk page: the dispatch serves BF16 and FP8
paged-decode launches; read here as E4M3 codes with per-tensor FP32 scales):
GPU output against the FP64 oracle over the dequantised cache, element by
element within |gpu - ref| <= ulp_bf16(ref) + 1e-3, plus batch invariance."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_splitk_gb300 import api, pd
from paged_kv_decode_splitk_gb300 import workloads as W

from helpers import assert_within_tolerance, oracle_all_rows

pytestmark = pytest.mark.gpu


def _ref(w, seqs=None):
    seqs = np.arange(w.num_seqs) if seqs is None else np.asarray(seqs)
    return oracle.decode_attn_fp8(w.q[seqs], w.k_cache, w.v_cache, w.k_scale, w.v_scale, w.block_table[seqs],
                                  w.context_lens[seqs], w.inv_sqrt_d)


def _run(w, device, n, pack=0):
    out = api.run_paged(api.PagedInputs(w, device), num_splits=n, gqa_pack=pack)
    assert out is not None
    assert pd.pd_device_status() == 0
    return api.bf16_to_f64(out)


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 1, 64), (24, 8, 128), (16, 2, 128), (32, 2, 256), (16, 2, 256)])
@pytest.mark.parametrize("N", [1, 3])
def test_fp8_shapes_and_splits(cuda_device, Hq, Hkv, D, N):
    lens = [0, 1, 15, 16, 17, 255, 700, 2049]
    w = W.fp8_variant(W.custom(lens, Hq, Hkv, D, seed=90 + D), k_scale=0.37, v_scale=1.7, seed=D)
    got = _run(w, cuda_device, N)
    assert_within_tolerance(got, _ref(w), f"fp8 Hq{Hq} Hkv{Hkv} D{D} N{N}")
    assert np.all(got[0] == 0.0)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 80), (12, 4, 96), (8, 1, 112), (8, 2, 160), (16, 4, 208)])
@pytest.mark.parametrize("N", [1, 4])
def test_fp8_head_dims_below_the_padded_width(cuda_device, Hq, Hkv, D, N):
    # K is read in boxes of 128 codes that reach past head_dim (zero-filled
    # there, with q zero in the same columns); V in one box of the padded row
    lens = [1, 16, 33, 600, 1500]
    w = W.fp8_variant(W.custom(lens, Hq, Hkv, D, seed=190 + D), k_scale=0.6, v_scale=1.3, seed=D + 1)
    assert_within_tolerance(_run(w, cuda_device, N), _ref(w), f"fp8 Hq{Hq} Hkv{Hkv} D{D} N{N}")


@pytest.mark.parametrize("pack,N", [(1, 1), (2, 4)])
def test_fp8_packed(cuda_device, pack, N):
    w = W.fp8_variant(W.custom([0, 33, 512, 4000], 16, 2, 256, seed=95), seed=5)
    assert_within_tolerance(_run(w, cuda_device, N, pack), _ref(w), f"fp8 packed mode {pack}")


def test_fp8_subnormal_codes(cuda_device):
    """Keys made of zero and subnormal codes only (a large K scale makes them
    matter) and values mixing subnormal and normal codes: a conversion that
    flushed subnormals would turn every score into 0."""
    w = W.custom([40, 300], 8, 2, 128, seed=96)
    rng = np.random.default_rng(7)
    sub = np.array([0x00, 0x01, 0x02, 0x03, 0x04, 0x05, 0x06, 0x07,
                    0x81, 0x82, 0x83, 0x84, 0x85, 0x86, 0x87], dtype=np.uint8)
    k8 = rng.choice(sub, size=w.k_cache.shape)
    v8 = np.where(rng.random(w.v_cache.shape) < 0.5, rng.choice(sub, size=w.v_cache.shape),
                  rng.integers(0x08, 0x70, size=w.v_cache.shape, dtype=np.uint8)).astype(np.uint8)
    kw = dict(w.__dict__)
    kw.update(k_cache=k8, v_cache=v8, kv_dtype="e4m3", k_scale=64.0, v_scale=0.5)
    w8 = W.PagedWorkload(**kw)
    got = _run(w8, cuda_device, 2)
    ref = _ref(w8)
    assert_within_tolerance(got, ref, "fp8 subnormal codes")
    assert np.std(ref) > 1e-3   # not a degenerate (uniform-attention) case


def test_fp8_long_context_full_size(cuda_device):
    w = W.long_context_fp8()
    n = api.PagedInputs(w, cuda_device).splits()
    assert n == 13
    assert_within_tolerance(_run(w, cuda_device, n), _ref(w), "fp8 long context")


def test_fp8_gqa_packed_full_size(cuda_device):
    w = W.gqa_packed_fp8()
    assert_within_tolerance(_run(w, cuda_device, 1, 1), _ref(w), "fp8 gqa packed")


def test_fp8_large_batch_whole_output_and_batch_invariant(cuda_device):
    w = W.large_batch_fp8()
    n = api.PagedInputs(w, cuda_device).splits()
    full = api.run_paged(api.PagedInputs(w, cuda_device), num_splits=n)
    assert pd.pd_device_status() == 0
    got = api.bf16_to_f64(full)
    assert_within_tolerance(got, oracle_all_rows(w), "fp8 large batch whole output")
    bits = api.bf16_bits(full)
    for s in (int(np.argmax(w.context_lens)), 77):
        kw = dict(w.__dict__)
        kw.update(q=w.q[[s]], block_table=w.block_table[[s]], context_lens=w.context_lens[[s]])
        alone = api.run_paged(api.PagedInputs(W.PagedWorkload(**kw), cuda_device), num_splits=n)
        assert np.array_equal(api.bf16_bits(alone)[0], bits[s])


def test_fp8_argument_errors(cuda_device):
    w = W.fp8_variant(W.custom([50], 8, 2, 64, seed=97), seed=6)
    inp = api.PagedInputs(w, cuda_device)
    out = torch.empty((1, 8, 64), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(pd.PdError) as e:
        pd.pd_decode_attn_fp8(inp.q, inp.k, inp.v, float("inf"), 1.0, inp.block_table, inp.context_lens, out,
                              w.inv_sqrt_d, 1)
    assert e.value.code == pd.PD_ERR_INVALID
    w40 = W.fp8_variant(W.custom([50], 8, 2, 40, seed=98), seed=7)
    i40 = api.PagedInputs(w40, cuda_device)
    out40 = torch.empty((1, 8, 40), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(pd.PdError) as e:
        pd.pd_decode_attn_fp8(i40.q, i40.k, i40.v, 1.0, 1.0, i40.block_table, i40.context_lens, out40,
                              w40.inv_sqrt_d, 1)
    assert e.value.code == pd.PD_ERR_UNSUPPORTED


@pytest.mark.parametrize("bs", [32, 64, 256])
def test_fp8_block_sizes(cuda_device, bs):
    w = W.fp8_variant(W.custom([0, 1, 31, 33, 500, 1100], 16, 4, 128, block_size=bs, seed=99), seed=bs)
    got = _run(w, cuda_device, 3)
    assert_within_tolerance(got, _ref(w), f"fp8 block {bs}")
