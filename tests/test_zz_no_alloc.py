"""psgd_project_q_static: the allocation-free Q = M^T P entry point.

Some callers cannot let the library call cudaMalloc (a job that reserved
nearly all device memory up front, code whose memory must come from a
framework's allocator, latency-sensitive code).  This entry point keeps its
partial sums in a static device array instead.  The test checks, through the
C ABI, that it reproduces the Q that psgd_step computes (read back with
psgd_get_q, from the P read back with psgd_get_p) on two calls in a row.
The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest

from parity_util import REL_TOL, rel

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _static_q(L, m_dev, p_host, rows, cols, rank):
    p_dev = torch.from_numpy(np.ascontiguousarray(p_host, dtype=np.float32)).to(DEV)
    q_dev = torch.full((cols, rank), float("nan"), dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.psgd_project_q_static(ctypes.c_void_p(m_dev.data_ptr()), ctypes.c_void_p(p_dev.data_ptr()),
                                 ctypes.c_void_p(q_dev.data_ptr()), rows, cols, rank,
                                 ctypes.c_void_p(stream))
    assert rc == 0, L.psgd_last_error()
    torch.cuda.synchronize()
    return q_dev.cpu().numpy()


# Every padded-rank instantiation of the kernel (1, 2, 4, 8, 16, 32 -- 4, 2
# and 1 columns per thread), each with a column count that is not a multiple
# of 4 (the element-by-element path) and a partial last row block; ranks 4
# and 32 also with aligned columns (the vector path), rank 16 with a column
# tile narrower than one thread's share at the edge.
@pytest.mark.parametrize("rows,cols,rank", [
    (513, 130, 1), (513, 131, 1),
    (650, 1001, 2),
    (1100, 700, 4), (777, 1030, 3),
    (900, 517, 5),
    (700, 333, 8),
    (1100, 900, 16), (1100, 901, 16),
    (600, 2000, 32), (600, 2001, 32),
])
def test_static_projection_matches_step(rows, cols, rank):
    from powersgd_rank_gradient_gb300 import PowerSGDState, _lib

    L = _lib.lib()
    st = PowerSGDState([(rows, cols)], 1, matrix_approximation_rank=rank, start_powerSGD_iter=0,
                       min_compression_rate=1.0, use_error_feedback=False, device=DEV)
    rng = np.random.default_rng(rows)
    st.set_q(0, rng.standard_normal((cols, rank)).astype(np.float32), is_draw=True)
    for call in range(2):
        m = torch.from_numpy(rng.standard_normal(rows * cols).astype(np.float32)).to(DEV)
        st.step([m])
        assert not st.status()
        p = st.get_p(0).numpy()
        q_step = st.get_q(0).double().numpy()
        q_static = _static_q(L, m, p, rows, cols, rank)
        assert np.all(np.isfinite(q_static))
        assert rel(q_static.astype(np.float64), q_step) <= REL_TOL, f"call {call}"
    st.close()


def test_static_projection_rejects_oversize():
    from powersgd_rank_gradient_gb300 import _lib

    L = _lib.lib()
    x = torch.zeros(16, device=DEV)
    ptr = ctypes.c_void_p(x.data_ptr())
    # ceil(5000 / 512) * 32 * 8192 partial sums exceed the 2 Mi-float array
    rc = L.psgd_project_q_static(ptr, ptr, ptr, 5000, 8192, 32, None)
    assert rc == _lib.PSGD_EINVAL
    assert b"static scratch" in L.psgd_last_error()
    # sizes whose product would overflow 64 bits are rejected, not launched
    rc = L.psgd_project_q_static(ptr, ptr, ptr, 2**62, 2**40, 32, None)
    assert rc == _lib.PSGD_EINVAL
    assert b"static scratch" in L.psgd_last_error()
    assert L.psgd_project_q_static(None, ptr, ptr, 4, 4, 1, None) == _lib.PSGD_EINVAL
