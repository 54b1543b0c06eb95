"""Host logic of the Python binding that needs no GPU: the spatial_shapes
checks and the per-tensor cache of device copies that keeps the autograd
operator free of per-call host synchronisation."""
import pytest

torch = pytest.importorskip("torch")


def test_check_shapes_on_host():
    import scale_deformable_attention_gb300 as msda

    ss = torch.tensor([[2, 3], [1, 4]])
    msda._check_shapes(ss, 10)
    with pytest.raises(ValueError):
        msda._check_shapes(ss, 11)
    with pytest.raises(ValueError):
        msda._check_shapes(torch.tensor([[0, 3], [1, 4]]), 4)


def test_device_copy_is_cached_per_tensor_and_version():
    import scale_deformable_attention_gb300 as msda

    dev = torch.device("cpu")
    t64 = torch.tensor([[2, 3]], dtype=torch.int64)
    assert msda._on_device(t64, dev) is t64          # already int64 and contiguous: no copy
    t32 = torch.tensor([[2, 3], [4, 5]], dtype=torch.int32)
    a = msda._on_device(t32, dev)
    assert a.dtype == torch.int64 and a.tolist() == [[2, 3], [4, 5]]
    assert msda._on_device(t32, dev) is a           # the copy is reused
    t32[0, 0] = 7                                   # an in-place change bumps the version
    b = msda._on_device(t32, dev)
    assert b is not a and b.tolist() == [[7, 3], [4, 5]]
    other = torch.tensor([[7, 3], [4, 5]], dtype=torch.int32)
    assert msda._on_device(other, dev) is not b     # another tensor never gets this one's copy
