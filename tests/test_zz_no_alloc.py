"""rmsnorm_bwd_noalloc: the backward for callers that cannot allocate device
memory when they call (engines that reserve all memory up front, plug-in
hosts that give an op no workspace, code running under a global-mode stream
capture). It keeps the dW partial rows in a fixed array inside the library.

Called through the C ABI, twice in a row on different inputs, its dx and dw
must agree with rmsnorm_bwd (which gets its own workspace) within the
tolerances the parity tests use: dx within 1 bf16 ulp, dw within 4e-3
relative. A size whose workspace exceeds the array must be refused without
a launch. This file sorts last so that a run stopping at the first failure
has already run every other test.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_ulp_distance, to_dev, to_host
from row_wise_normalization_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rn():
    from row_wise_normalization_rmsnorm_gb300 import build
    build.build()
    import row_wise_normalization_rmsnorm_gb300 as pkg
    return pkg


def test_noalloc_backward_matches_rmsnorm_bwd_on_two_calls(rn):
    L = rn.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, seed in ((4096, 8192, 301), (1000, 2048, 302)):
        d = inputs.make_inputs(M, N, "bf16", seed)
        x, dy, w = (to_dev(d[k], "bf16") for k in ("x", "dy", "w"))
        _, rstd = rn.rmsnorm_fwd(x, w)
        dx_ref, dw_ref = rn.rmsnorm_bwd(dy, x, w, rstd)
        dx = torch.full_like(x, float("nan"))
        dw = torch.full_like(w, float("nan"))
        st = L.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), w.data_ptr(), rstd.data_ptr(), dx.data_ptr(),
                                   dw.data_ptr(), M, N, 1, 1e-6, 0.0, stream)
        assert st == 0, rn.lib().rmsnorm_status_string(st)
        torch.cuda.synchronize()
        assert bf16_ulp_distance(to_host(dx, "bf16"), to_host(dx_ref, "bf16")).max() <= 1
        a = dw.float().cpu().numpy().astype(np.float64)
        b = dw_ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        assert np.all(np.abs(a - b) <= 4e-3 * np.abs(b) + 1e-6)


def test_noalloc_refuses_sizes_beyond_its_array(rn):
    """A call whose partial rows do not fit is refused before any launch.
    Every buffer passed is real and large enough for the call, so nothing
    could go out of bounds even if it were not refused. Bases one element
    past an aligned allocation select the generic backward, which keeps at
    least one partial row per SM: >= 152 rows x 65536 x 4 B > 32 MiB."""
    L = rn.lib()
    limit = 32 << 20
    M, N = 2048, 65536
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = rn.plan_query(rn.OP_BWD, M, N, rn.RMSNORM_BF16, aligned=False, num_sms=sms, ctas_per_sm=1)
    assert plan["path_name"] == "generic" and plan["workspace_bytes"] > limit

    def buf(n, dtype=torch.bfloat16):
        return torch.zeros(n + 1, dtype=dtype, device="cuda")[1:]

    x, dy, dx = buf(M * N), buf(M * N), buf(M * N)
    w, dw = buf(N), buf(N)
    r = torch.ones(M, dtype=torch.float32, device="cuda")
    st = L.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), w.data_ptr(), r.data_ptr(), dx.data_ptr(),
                               dw.data_ptr(), M, N, 1, 1e-6, 0.0, torch.cuda.current_stream().cuda_stream)
    assert st == 3          # RMSNORM_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
