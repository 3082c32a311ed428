"""The calibration read (ub_stream_read): it reads what it is given and nothing else,
leaves the handle's status clean, replays from a CUDA graph, and rejects what it cannot
read (unaligned source or size, negative size)."""
import pytest
import torch

from gemm_overlap_gemms_gb300 import ub
from gpu_helpers import dev, is_sentinel, sentinel

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_bytes", [16, 4096, 32768 + 16, 3 * 1024 * 1024 + 48, 117 * 1024 * 1024])
def test_stream_read_runs_clean_and_writes_nothing(n_bytes):
    guard = 4096
    # the bytes to read, between two sentinel guards that must stay as they were
    buf_t = sentinel(((guard * 2 + n_bytes) // 2,))
    body = buf_t[guard // 2: guard // 2 + n_bytes // 2]
    body.view(torch.int16).fill_(7)
    with ub.UserBuffer([64, 64], 1) as buf:
        buf.stream_read(body)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    assert is_sentinel(buf_t[:guard // 2]) and is_sentinel(buf_t[guard // 2 + n_bytes // 2:])
    assert bool((body.view(torch.int16) == 7).all().item())


def test_stream_read_replays_from_a_graph():
    t = torch.zeros(8 * 1024 * 1024, dtype=torch.bfloat16, device=dev())
    with ub.UserBuffer([64, 64], 1) as buf:
        s = torch.cuda.Stream()
        buf.stream_read(t, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            buf.stream_read(t, stream=s)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK


def test_stream_read_rejects_what_it_cannot_read():
    t = torch.zeros(4096, dtype=torch.bfloat16, device=dev())
    with ub.UserBuffer([64, 64], 1) as buf:
        L = ub.load()
        p = t.data_ptr()
        assert L.ub_stream_read(buf._h, p + 2, 1024, None) == ub.CODES["UB_ERR_ALIGN"]
        assert L.ub_stream_read(buf._h, p, 1000, None) == ub.CODES["UB_ERR_ALIGN"]
        assert L.ub_stream_read(buf._h, p, -16, None) == ub.CODES["UB_ERR_ARG"]
        assert L.ub_stream_read(buf._h, None, 16, None) == ub.CODES["UB_ERR_ARG"]
        assert L.ub_stream_read(buf._h, p, 0, None) == ub.UB_OK
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
