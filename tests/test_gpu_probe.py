"""The streaming-read probe the benchmark uses as a floor: it reads what it is given, leaves its sink alone
and refuses unaligned arguments."""
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
