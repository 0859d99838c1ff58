"""The Python binding's shape agreement checks (CPU, no library call).

The C ABI receives bare pointers and trusts the extents it is given, so the binding must refuse
tensors that disagree before anything reaches the library: a pos vector shorter than the batch,
a v cache smaller than the k cache, an output of the wrong shape.  Shapes only matter here, so
the tests use CPU tensors and call the binding's checks directly.
"""
from __future__ import annotations

import pytest
import torch

import sliding_window_gqa_gb300 as wa


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def i32(n):
    return torch.zeros(n, dtype=torch.int32)


def test_decode_shapes_accept_a_consistent_call():
    q, k = bf16(3, 16, 256), bf16(3, 1536, 8, 256)
    assert wa._decode_shapes(q, k, bf16(3, 1536, 8, 256), i32(3), bf16(3, 16, 256)) == (3, 16, 8, 256, 1536)
    assert wa._decode_shapes(q, k, k.clone(), i32(3), None) == (3, 16, 8, 256, 1536)


@pytest.mark.parametrize("bad", ["pos_short", "pos_2d", "v_small", "k_rows", "k_dim", "out_shape", "out_dtype",
                                 "q_rank"])
def test_decode_shapes_refuse_disagreeing_tensors(bad):
    q, k, v, pos, out = bf16(3, 16, 256), bf16(3, 1536, 8, 256), bf16(3, 1536, 8, 256), i32(3), None
    if bad == "pos_short":
        pos = i32(2)
    elif bad == "pos_2d":
        pos = torch.zeros((3, 1), dtype=torch.int32)
    elif bad == "v_small":
        v = bf16(3, 1024, 8, 256)
    elif bad == "k_rows":
        k = v = bf16(2, 1536, 8, 256)
    elif bad == "k_dim":
        k = v = bf16(3, 1536, 8, 128)
    elif bad == "out_shape":
        out = bf16(3, 8, 256)
    elif bad == "out_dtype":
        out = torch.zeros((3, 16, 256), dtype=torch.float32)
    elif bad == "q_rank":
        q = bf16(3 * 16, 256)
    with pytest.raises(ValueError):
        wa._decode_shapes(q, k, v, pos, out)


def test_prompt_shapes_accept_a_consistent_call():
    q, k = bf16(512, 16, 256), bf16(1536, 8, 256)
    assert wa._prompt_shapes(q, k, bf16(1536, 8, 256), i32(512), None) == (512, 16, 8, 256, 1536)
    # the dense interleaved layout: strided views of one buffer
    qkv = bf16(100, 3 * 56 * 128)
    q = qkv[:, :7168].view(100, 56, 128)
    k = qkv[:, 7168:14336].view(100, 56, 128)
    v = qkv[:, 14336:].view(100, 56, 128)
    assert wa._prompt_shapes(q, k, v, None, bf16(100, 56, 128)) == (100, 56, 56, 128, 100)


@pytest.mark.parametrize("bad", ["v_short", "d_mismatch", "hi_short", "hi_dtype", "out_shape"])
def test_prompt_shapes_refuse_disagreeing_tensors(bad):
    q, k, v, hi, out = bf16(512, 16, 256), bf16(1536, 8, 256), bf16(1536, 8, 256), None, None
    if bad == "v_short":
        v = bf16(1000, 8, 256)
    elif bad == "d_mismatch":
        k = v = bf16(1536, 8, 128)
    elif bad == "hi_short":
        hi = i32(511)
    elif bad == "hi_dtype":
        hi = torch.zeros(512, dtype=torch.int64)
    elif bad == "out_shape":
        out = bf16(512, 8, 256)
    with pytest.raises((ValueError, TypeError)):
        wa._prompt_shapes(q, k, v, hi, out)


def test_prep_shapes_accept_shared_and_per_token_rings():
    src = bf16(4, (8 + 2 * 4) * 128)
    assert wa._prep_shapes(src, i32(4), bf16(4, 8, 128), bf16(64, 4, 128), bf16(64, 4, 128)) == (4, 8, 4, 128)
    assert wa._prep_shapes(src, i32(4), bf16(4, 8, 128), bf16(4, 64, 4, 128), None) == (4, 8, 4, 128)


@pytest.mark.parametrize("bad", ["src_narrow", "pos_short", "q_tokens", "rings_count", "v_shape"])
def test_prep_shapes_refuse_disagreeing_tensors(bad):
    src, pos, q_out, k, v = bf16(4, 16 * 128), i32(4), bf16(4, 8, 128), bf16(4, 64, 4, 128), None
    if bad == "src_narrow":
        src = bf16(4, 15 * 128)
    elif bad == "pos_short":
        pos = i32(3)
    elif bad == "q_tokens":
        q_out = bf16(5, 8, 128)
    elif bad == "rings_count":
        k = bf16(3, 64, 4, 128)
    elif bad == "v_shape":
        v = bf16(4, 32, 4, 128)
    with pytest.raises(ValueError):
        wa._prep_shapes(src, pos, q_out, k, v)


def test_workspace_must_be_a_device_tensor():
    with pytest.raises(TypeError):
        wa._workspace(256, torch.device("cpu"), torch.zeros(256, dtype=torch.uint8))
