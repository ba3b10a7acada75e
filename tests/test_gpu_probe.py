"""The benchmark's probes: the streaming read (a floor for weight-streaming kernels) reads what it is given,
leaves its sink alone and refuses unaligned arguments; the block-scaled MMA stream (a ceiling for the prefill
GEMMs) completes without running out its wait and refuses bad arguments."""
import pytest

torch = pytest.importorskip("torch")

from expert_offload_moe_gb300 import build as moe_build
from expert_offload_moe_gb300 import moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def test_stream_read_runs_and_leaves_the_sink(lib):
    buf = torch.arange(1 << 22, dtype=torch.int32, device="cuda")  # 16 MiB, xor of all words != the constant
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    for nblocks in (0, 1, 7):
        moe.stream_read(buf.data_ptr(), buf.numel() * 4, sink.data_ptr(), nblocks=nblocks)
        moe.stream_read(buf.data_ptr(), 48, sink.data_ptr(), nblocks=nblocks)  # fewer words than threads
    torch.cuda.synchronize()
    assert int(sink.abs().sum()) == 0


def test_stream_read_rejects_bad_arguments(lib):
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = moe.stream_ptr(None)
    assert lib.moe_debug_stream_read(moe._P(buf.data_ptr() + 4), 64, moe._P(sink.data_ptr()), 0, s) == moe.MOE_EINVAL
    assert lib.moe_debug_stream_read(moe._P(buf.data_ptr()), 20, moe._P(sink.data_ptr()), 0, s) == moe.MOE_EINVAL
    assert lib.moe_debug_stream_read(moe._P(buf.data_ptr()), 64, moe._P(sink.data_ptr()), -1, s) == moe.MOE_EINVAL


def test_mma_peak_completes_and_scales_with_iters(lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ms = {}
    for iters in (256, 2048):
        moe.mma_peak(iters, err.data_ptr())  # warm-up
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        moe.mma_peak(iters, err.data_ptr())
        e1.record()
        torch.cuda.synchronize()
        ms[iters] = e0.elapsed_time(e1)
    moe.mma_peak(1, err.data_ptr(), nblocks=3)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert ms[2048] > 2.0 * ms[256]  # the launch is MMA-bound, not launch-bound
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tflops = moe.mma_peak_flops(2048, sms) / (ms[2048] * 1e-3) / 1e12
    assert 500 < tflops < 20000


def test_mma_peak_rejects_bad_arguments(lib):
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = moe.stream_ptr(None)
    assert lib.moe_debug_mma_peak(0, 0, moe._P(err.data_ptr()), s) == moe.MOE_EINVAL
    assert lib.moe_debug_mma_peak(65537, 0, moe._P(err.data_ptr()), s) == moe.MOE_EINVAL
    assert lib.moe_debug_mma_peak(8, -1, moe._P(err.data_ptr()), s) == moe.MOE_EINVAL
    assert lib.moe_debug_mma_peak(8, 0, moe._P(err.data_ptr() + 2), s) == moe.MOE_EINVAL
    assert lib.moe_debug_mma_peak(8, 0, None, s) == moe.MOE_EINVAL
