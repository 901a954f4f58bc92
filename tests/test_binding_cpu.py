"""The Python binding's argument checks, on the CPU: tensors that are not CUDA,
of the wrong dtype or shape, or on another device than the call's are rejected
before the library is called (no GPU needed)."""
import pytest
import torch

import online_softmax_merge_gb300 as ra


def _qkv(dev="cpu", dtype=torch.bfloat16):
    q = torch.zeros((1, 256, 4, 128), dtype=dtype, device=dev)
    k = torch.zeros((1, 256, 2, 128), dtype=dtype, device=dev)
    return q, k, k.clone()


def test_host_tensors_are_rejected_by_the_device_calls():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA tensor"):
        ra.fwd(q, k, v, 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ra.decode(q[:, :1], k, v, 2, 255)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ra.merge(torch.zeros((2, 1, 8, 4, 128)), torch.zeros((2, 1, 4, 8)))


def test_wrong_dtype_and_shape_are_rejected():
    q, k, v = _qkv(dtype=torch.float16)
    with pytest.raises(ValueError, match="bfloat16"):
        ra.fwd(q, k, v, 2)
    with pytest.raises(ValueError, match="shape"):
        ra.fwd_host(*_qkv()[:2], torch.zeros((1, 255, 2, 128), dtype=torch.bfloat16), 2)
    with pytest.raises(ValueError, match="layout"):
        ra.problem(1, 256, 4, 2, 128, 2, True, "diagonal")


def test_tensors_on_another_device_are_rejected():
    ref = torch.zeros(4)
    other = torch.zeros(4, device="meta")
    with pytest.raises(ValueError, match="out is on meta"):
        ra._same_device(ref, lse=torch.zeros(2), out=other)
    ra._same_device(ref, a=torch.zeros(1), b=torch.zeros(2))     # same device: accepted


def test_host_forward_rejects_device_inputs_before_any_work():
    q, k, v = _qkv(dev="meta")
    with pytest.raises(ValueError, match="host"):
        ra.fwd_host(q, k, v, 2)
