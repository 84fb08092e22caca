"""The torch helpers validate their tensors before calling the C ABI, which reads
dense device memory and cannot tell a wrong dtype, stride or shape (CPU tensors
stand in here: every check before the device check is exercised without a GPU)."""
import pytest
import torch

import exact_attention_blackwell_gb300 as fa


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_fwd_checks_dtype_layout_shape_and_device():
    q, k, v = bf16(1, 128, 2, 64), bf16(1, 128, 2, 64), bf16(1, 128, 2, 64)
    with pytest.raises(ValueError, match="bfloat16"):
        fa.attention_fwd(q.float(), k, v)
    with pytest.raises(ValueError, match="contiguous"):
        fa.attention_fwd(q, k.transpose(1, 2).contiguous().transpose(1, 2), v)
    with pytest.raises(ValueError, match="shape"):
        fa.attention_fwd(q, k, bf16(1, 127, 2, 64))
    with pytest.raises(ValueError, match="shape"):
        fa.attention_fwd(q, k, v, lse=torch.zeros((1, 2, 127)))
    with pytest.raises(ValueError, match="CUDA"):
        fa.attention_fwd(q, k, v)
    with pytest.raises(ValueError, match="B, N, H, d"):
        fa.attention_fwd(bf16(128, 2, 64), k, v)


def test_bwd_checks_every_operand():
    q = bf16(1, 128, 4, 64)
    k = v = bf16(1, 128, 2, 64)
    lse = torch.zeros((1, 4, 128))
    with pytest.raises(ValueError, match="dO"):
        fa.attention_bwd(q, k, v, q, lse, bf16(1, 128, 2, 64))
    with pytest.raises(ValueError, match="lse"):
        fa.attention_bwd(q, k, v, q, lse.double(), q)
    with pytest.raises(ValueError, match="CUDA"):
        fa.attention_bwd(q, k, v, q, lse, q)


def test_packed_checks_the_offsets_table():
    q = bf16(300, 2, 128)
    k = v = bf16(300, 1, 128)
    with pytest.raises(ValueError, match="int32"):
        fa.attention_fwd_varlen(q, k, v, torch.tensor([0, 100, 300]), 200)
    with pytest.raises(ValueError, match="cu_seqlens"):
        fa.attention_fwd_varlen(q, k, v, torch.zeros((2, 2), dtype=torch.int32), 200)
    with pytest.raises(ValueError, match="CUDA"):
        fa.attention_fwd_varlen(q, k, v, torch.tensor([0, 100, 300], dtype=torch.int32), 200)


def test_fp8_checks_the_rotation_signs():
    q = k = v = bf16(1, 128, 2, 128)
    with pytest.raises(ValueError, match="rot_signs"):
        fa.attention_fwd_fp8(q, k, v, torch.ones(64))
