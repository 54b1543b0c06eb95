"""msda_reduction_ceiling, the measurement the backward's reduction roofline
is reported against: it runs, leaves no device error, and gives a rate of
the order of the L2's (tens to hundreds of G sectors/s) for every kind."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,row_bytes", [("bf16", 64), ("f16", 64), ("f32", 128), ("f32", 32), ("bf16", 512)])
def test_reduction_ceiling_runs(dtype, row_bytes):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import scale_deformable_attention_gb300 as msda

    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
    rate = msda.reduction_ceiling(tdt, row_bytes=row_bytes, blocks_per_sm=4, repeats=2)
    assert 1e10 < rate < 2e12, rate
    assert msda.device_errors() == 0
