"""The read-only floor kernel behind the decode workloads' floor measurement:
it reads the bytes it is given with the streaming kernel's launch shape,
reports the grid it used, and leaves the device error word clear."""
import pytest
import torch

from rank_gemv_gb300 import workloads as wl
from tests.gpu_helpers import check_error_word

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,ctas,cluster", [("decode-distinct", 128, 4),
                                               ("decode-zipf", 256, 4),
                                               ("llama7b-q", 128, 1), ("tiny", 64, 8)])
def test_read_floor_runs_with_the_streaming_shape(name, ctas, cluster):
    from rank_gemv_gb300 import sgmv

    w = wl.make(name, 0)
    nbytes = (w.bytes_moved() + 15) // 16 * 16
    src = torch.ones(nbytes // 4 + 64, dtype=torch.int32, device="cuda")
    got_ctas, got_cl = sgmv.sgmv_read_floor(src, nbytes, w.T, w.L, w.H1, w.H2, w.r, w.dtype,
                                            w.y_dtype)
    torch.cuda.synchronize()
    check_error_word(0)
    assert got_cl == cluster
    assert got_ctas == ctas
    assert bool((src == 1).all())  # nothing written
