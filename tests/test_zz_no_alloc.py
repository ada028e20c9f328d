"""The allocation-free RMSNorm backward (sf_op_rmsnorm_bwd_noalloc).

It is for callers that cannot allocate device memory: it keeps its scratch
in a fixed array of the library instead of a caller buffer.  Checked through
the C ABI against the scratch-taking entry point, bit for bit, on two calls
in a row (the second one sees the array as the first one left it).  This
file is collected last so that a run stopping at the first failure has run
every other test.
"""
import pytest
import torch

import inputs
from tests.gpu_util import bf16_values, cuda, host, stream, sync
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu
sf = pytest.importorskip("offloaded_fine_tuning_gb300")


def _case(seed, rows, d):
    x = inputs.normal(seed, 1, rows * d, 0.0, 2.0).reshape(rows, d)
    g = bf16_values(1.0 + 0.1 * inputs.normal(seed, 2, d))
    dy = inputs.normal(seed, 3, rows * d).reshape(rows, d)
    dres = inputs.normal(seed, 4, rows * d).reshape(rows, d)
    X, G, DY, DR = cuda(x, torch.float32), cuda(g, torch.bfloat16), cuda(dy, torch.float32), cuda(dres, torch.float32)
    RS = torch.empty(rows, dtype=torch.float32, device="cuda")
    Y = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    assert sf.op_rmsnorm_fwd(X.data_ptr(), G.data_ptr(), Y.data_ptr(), RS.data_ptr(), rows, d, 1e-5, stream()) == 0
    return X, G, RS, DY, DR


def _outputs(rows, d):
    return (torch.empty((rows, d), dtype=torch.float32, device="cuda"),
            torch.empty((rows, d), dtype=torch.bfloat16, device="cuda"),
            torch.empty(d, dtype=torch.bfloat16, device="cuda"))


def test_noalloc_matches_scratch_entry_point_on_two_calls_in_a_row():
    """Both entry points run the same kernels over the same row partition, so
    their results must agree bit for bit; a partition mismatch would show."""
    sf.lib(build_if_needed=True)
    cases = [(11, 300, 4096), (12, 1000, 768)]  # second call: other shape and contents
    for seed, rows, d in cases:
        X, G, RS, DY, DR = _case(seed, rows, d)
        dx0, dxb0, dg0 = _outputs(rows, d)
        scratch = torch.empty(sf.rmsnorm_bwd_scratch(rows, d), dtype=torch.float32, device="cuda")
        assert sf.op_rmsnorm_bwd(X.data_ptr(), G.data_ptr(), RS.data_ptr(), DY.data_ptr(), DR.data_ptr(),
                                 dx0.data_ptr(), dxb0.data_ptr(), dg0.data_ptr(), scratch.data_ptr(),
                                 rows, d, stream()) == 0
        dx1, dxb1, dg1 = _outputs(rows, d)
        sync()
        alloc, reserved = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
        free_before = torch.cuda.mem_get_info()[0]
        assert sf.op_rmsnorm_bwd_noalloc(X.data_ptr(), G.data_ptr(), RS.data_ptr(), DY.data_ptr(),
                                         DR.data_ptr(), dx1.data_ptr(), dxb1.data_ptr(), dg1.data_ptr(),
                                         rows, d, stream()) == 0
        sync()
        # nothing was taken from torch's allocator, on either call
        assert torch.cuda.memory_allocated() == alloc and torch.cuda.memory_reserved() == reserved
        if seed != cases[0][0]:  # after the first call's one-time set-up, no device memory moves
            assert torch.cuda.mem_get_info()[0] == free_before
        for a, b in ((dx1, dx0), (dxb1, dxb0), (dg1, dg0)):
            assert torch.equal(a.view(torch.int32 if a.dtype == torch.float32 else torch.int16),
                               b.view(torch.int32 if b.dtype == torch.float32 else torch.int16))
        assert rel_l2(host(dx1), host(dx0)) == 0.0


def test_noalloc_rejects_sizes_beyond_its_array():
    sf.lib(build_if_needed=True)
    parts = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    d = 16384
    if parts * d <= sf.STATIC_SCRATCH_FLOATS:
        pytest.skip("this GPU's row partition fits the array at every size")
    rows = parts
    buf = torch.empty((rows, d), dtype=torch.float32, device="cuda")
    b16 = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    rs = torch.ones(rows, dtype=torch.float32, device="cuda")
    st = sf.op_rmsnorm_bwd_noalloc(buf.data_ptr(), g.data_ptr(), rs.data_ptr(), buf.data_ptr(), 0,
                                   buf.data_ptr(), b16.data_ptr(), g.data_ptr(), rows, d, stream())
    assert st == sf.SF_EINVAL
