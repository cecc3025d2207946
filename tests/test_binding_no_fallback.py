"""The product path has no CPU fallback: every call of the binding refuses
host tensors (and wrong dtypes) before anything runs, and the library it
loads is the in-tree build.  No GPU needed."""
import os

import pytest
import torch

import paged_kv_cache_125_gb300 as kvp

bf16, i32 = torch.bfloat16, torch.int32


def _cache():
    return torch.zeros((4, 16, 2, 64), dtype=bf16), torch.zeros((4, 16, 2, 64), dtype=bf16)


def test_library_is_the_in_tree_build():
    path = os.path.realpath(kvp.library_path())
    pkg = os.path.realpath(os.path.dirname(kvp.__file__))
    assert path.startswith(pkg + os.sep) and "site-packages" not in path


def test_kv_store_refuses_host_tensors():
    kc, vc = _cache()
    k = v = torch.zeros((3, 2, 64), dtype=bf16)
    with pytest.raises(ValueError, match="CUDA"):
        kvp.kv_store(k, v, torch.zeros(3, dtype=i32), kc, vc)
    with pytest.raises(TypeError):  # dtypes are checked first
        kvp.kv_store(k, v, torch.zeros(3, dtype=i32), kc.float(), vc)


def test_decode_refuses_host_tensors():
    kc, vc = _cache()
    q = torch.zeros((2, 4, 64), dtype=bf16)
    bt, ctx = torch.zeros((2, 3), dtype=i32), torch.ones(2, dtype=i32)
    with pytest.raises(ValueError, match="CUDA"):
        kvp.attn_decode_paged(q, kc, vc, bt, ctx, 48)
    with pytest.raises(ValueError, match="CUDA"):
        kvp.attn_decode_paged_append(q, torch.zeros((2, 2, 64), dtype=bf16),
                                     torch.zeros((2, 2, 64), dtype=bf16), torch.zeros(2, dtype=i32),
                                     kc, vc, bt, ctx, 48)
    with pytest.raises(ValueError, match="CUDA"):
        kvp.attn_decode_paged_noalloc(q, kc, vc, bt, ctx, 48, out=torch.zeros_like(q))


def test_prefill_refuses_host_tensors():
    q = torch.zeros((5, 4, 64), dtype=bf16)
    cu = torch.tensor([0, 5], dtype=i32)
    with pytest.raises(ValueError, match="CUDA"):
        kvp.attn_prefill_varlen(q, cu, cu, 5, 5, k=torch.zeros((5, 2, 64), dtype=bf16),
                                v=torch.zeros((5, 2, 64), dtype=bf16), num_kv_heads=2)


def test_copy_blocks_refuses_host_tensors():
    cache = torch.zeros((2, 1, 4, 16, 2, 64), dtype=bf16)
    with pytest.raises(ValueError, match="CUDA"):
        kvp.kv_copy_blocks(cache, torch.tensor([[0, 1]], dtype=i32))
