"""DecodeStep rejects bad arguments before it touches the GPU (CPU test)."""
import pytest
import torch

from sm_load_balancing_gb300.step import DecodeStep


def test_decode_step_argument_checks():
    q = torch.zeros(2, 1, 8, 64, dtype=torch.bfloat16)
    k_cpu = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="q_like"):
        DecodeStep(q.float(), k_cpu, None, 4, scale=0.1)
    with pytest.raises(ValueError, match="q_like"):
        DecodeStep(q[0], k_cpu, None, 4, scale=0.1)
    with pytest.raises(ValueError, match="CUDA"):
        DecodeStep(q, k_cpu, k_cpu, 4, scale=0.1)
