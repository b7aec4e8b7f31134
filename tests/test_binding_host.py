"""The Python binding's argument marshalling on the CPU: row pitch of strided
views, shape checks, and the type, device and activation checks that run before
any call into the library.  No GPU is involved: every case here raises (or
computes a pitch) before a device is touched."""
import pytest
import torch

from dense_fp32_gemm_02_gb300 import binding


def test_row_pitch_of_compact_padded_and_degenerate_views():
    base = torch.zeros(6, 10)
    assert binding._ld(base, 10) == 10
    assert binding._ld(base[:, :7], 7) == 10        # a view inside wider rows keeps the pitch
    assert binding._ld(base[2:5, 3:8], 5) == 10
    assert binding._ld(base[:1, :4], 4) == 4         # one row: the pitch is the width
    assert binding._ld(torch.zeros(0, 5), 5) == 5    # empty
    assert binding._ld(torch.zeros(3, 0), 0) == 1    # zero width: pitch at least 1


def test_row_pitch_rejects_strided_rows_and_other_ranks():
    with pytest.raises(ValueError, match="contiguous"):
        binding._ld(torch.zeros(4, 6).t(), 4)
    with pytest.raises(ValueError, match="contiguous"):
        binding._ld(torch.zeros(4, 6)[:, ::2], 3)
    with pytest.raises(ValueError, match="2-D"):
        binding._ld(torch.zeros(2, 3, 4), 4)


def test_shapes_must_agree():
    A, B, C = torch.zeros(3, 4), torch.zeros(4, 5), torch.zeros(3, 5)
    assert binding._shapes(A, B, C) == (3, 5, 4)
    with pytest.raises(ValueError, match="inner dimensions"):
        binding._shapes(A, torch.zeros(5, 5), C)
    with pytest.raises(ValueError, match="C must be"):
        binding._shapes(A, B, torch.zeros(5, 3))


@pytest.mark.parametrize("fn", [binding.sgemm_into, binding.sgemm_3xtf32_into,
                                binding.sgemm_noalloc_into, binding.sgemm_ex_into])
def test_device_entry_points_refuse_host_and_non_float32_tensors(fn):
    A, B, C = torch.zeros(3, 4), torch.zeros(4, 5), torch.zeros(3, 5)
    with pytest.raises(TypeError, match="A must be a CUDA float32 tensor"):
        fn(A, B, C)
    with pytest.raises(TypeError, match="must be a CUDA float32 tensor"):
        fn(A.double(), B, C)
    with pytest.raises(TypeError):
        fn(A.numpy(), B, C)


def test_new_output_needs_beta_zero():
    with pytest.raises(ValueError, match="beta != 0"):
        binding.sgemm(torch.zeros(2, 2), torch.zeros(2, 2), None, beta=1.0)


def test_host_entry_point_checks_types_and_shapes_before_any_device_call():
    A, B, C = torch.zeros(3, 4), torch.zeros(4, 5), torch.zeros(3, 5)
    with pytest.raises(TypeError, match="CPU float32"):
        binding.sgemm_host(A.double(), B, C)
    with pytest.raises(TypeError, match="CPU float32"):
        binding.sgemm_host(A, B.half(), C)
    with pytest.raises(ValueError, match="inner dimensions"):
        binding.sgemm_host(A, torch.zeros(3, 5), C)
    with pytest.raises(ValueError, match="C must be"):
        binding.sgemm_host(A, B, torch.zeros(5, 3))


def test_batched_views():
    t = torch.zeros(4, 3, 5)
    first, batch, stride = binding._batched(t, "A")
    assert tuple(first.shape) == (3, 5) and batch == 4 and stride == 15
    m = torch.zeros(3, 5)
    assert binding._batched(m, "B")[1:] == (1, 0)           # one matrix shared by every batch
    assert binding._batched(torch.zeros(1, 3, 5), "C")[1:] == (1, 0)
    with pytest.raises(ValueError, match="2-D or 3-D"):
        binding._batched(torch.zeros(2, 2, 2, 2), "C")


def test_activation_names():
    assert binding.ACTIVATIONS == {"none": 0, "relu": 1, "gelu": 2}
