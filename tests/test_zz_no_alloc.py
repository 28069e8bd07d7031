"""rmsnorm_bwd_noalloc: the backward for callers that cannot allocate device
memory when they call (engines that reserve all device memory up front,
plug-in hosts that give an op no workspace). It keeps the dW partial rows
in a fixed array inside the library.

Called through the C ABI twice in a row, the second time on a smaller
problem (so stale partial rows left by the first call in the shared array
would show), its dx and dw must equal rmsnorm_bwd's bit for bit: the two
run the same plan, the same CTA count and the same fixed-order finalizer,
and only the workspace address differs. Every storage type rmsnorm_bwd
takes is covered. A size whose workspace exceeds the array must be refused
without a launch. This file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import pytest
import torch

from helpers import cuda_bits_equal, to_dev
from row_wise_normalization_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu

# (storage type name for the inputs, weight type name, ABI dtype code)
DTYPES = [("bf16", "bf16", 1), ("f32", "f32", 0), ("f16", "f16", 2), ("bf16", "f32", 0x101), ("f16", "f32", 0x102)]


@pytest.fixture(scope="module")
def rn():
    from row_wise_normalization_rmsnorm_gb300 import build
    build.build()
    import row_wise_normalization_rmsnorm_gb300 as pkg
    return pkg


@pytest.mark.parametrize("dt,wdt,code", DTYPES)
def test_noalloc_backward_equals_rmsnorm_bwd_on_two_calls(rn, dt, wdt, code):
    L = rn.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, seed in ((4096, 8192, 301), (1000, 2048, 302)):
        d = inputs.make_inputs(M, N, dt, seed, wdtype=wdt)
        x, dy = to_dev(d["x"], dt), to_dev(d["dy"], dt)
        w = to_dev(d["w"], wdt)
        _, rstd = rn.rmsnorm_fwd(x, w)
        dx_ref, dw_ref = rn.rmsnorm_bwd(dy, x, w, rstd)
        dx = torch.full_like(x, float("nan"))
        dw = torch.full_like(w, float("nan"))
        st = L.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), w.data_ptr(), rstd.data_ptr(), dx.data_ptr(),
                                   dw.data_ptr(), M, N, code, 1e-6, 0.0, stream)
        assert st == 0, L.rmsnorm_status_string(st)
        torch.cuda.synchronize()
        assert cuda_bits_equal(dx, dx_ref), (dt, wdt, M, N)
        assert cuda_bits_equal(dw, dw_ref), (dt, wdt, M, N)


def test_noalloc_refuses_sizes_beyond_its_array(rn):
    """A call whose partial rows do not fit is refused before any launch.
    Every buffer passed is real and large enough for the call, so nothing
    could go out of bounds even if it were not refused. x and dy at
    different addresses mod 16 (one and two elements past aligned
    allocations) select the generic backward, which keeps at least one
    partial row per SM: >= 152 rows x 65536 x 4 B > 32 MiB."""
    L = rn.lib()
    limit = 32 << 20
    M, N = 2048, 65536
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = rn.plan_query(rn.OP_BWD, M, N, rn.RMSNORM_BF16, aligned=False, num_sms=sms, ctas_per_sm=1)
    assert plan["path_name"] == "generic" and plan["workspace_bytes"] > limit

    def buf(n, dtype=torch.bfloat16, off=1):
        return torch.zeros(n + off, dtype=dtype, device="cuda")[off:]

    x, dy, dx = buf(M * N), buf(M * N, off=2), buf(M * N)
    w, dw = buf(N), buf(N)
    r = torch.ones(M, dtype=torch.float32, device="cuda")
    st = L.rmsnorm_bwd_noalloc(dy.data_ptr(), x.data_ptr(), w.data_ptr(), r.data_ptr(), dx.data_ptr(),
                               dw.data_ptr(), M, N, 1, 1e-6, 0.0, torch.cuda.current_stream().cuda_stream)
    assert st == 3          # RMSNORM_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
