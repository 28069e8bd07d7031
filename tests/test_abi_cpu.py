"""Host-side tests of the C ABI that need no GPU: the library loads, exports
every entry point the header declares, its plan table passes the self-check,
plan selection follows the table, and argument errors are reported as
status codes before any CUDA call."""
import ctypes
import os
import re

import pytest

from row_wise_normalization_rmsnorm_gb300 import build as rn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rmsnorm.h")


@pytest.fixture(scope="module")
def rn():
    rn_build.build()
    import row_wise_normalization_rmsnorm_gb300 as pkg
    return pkg


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rmsnorm_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_add_fwd", "rmsnorm_add_bwd",
                     "rmsnorm_bwd_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(rn):
    h = ctypes.CDLL(rn.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(h, n)]
    assert not missing, missing
    # and the binding declares a signature for each
    from row_wise_normalization_rmsnorm_gb300._binding import SIGNATURES
    assert set(declared_functions()) <= set(SIGNATURES)


def test_plan_table_self_check(rn):
    assert rn.lib().rmsnorm_self_check() == 0
    ids = [rn.lib().rmsnorm_plan_id_at(i) for i in range(rn.lib().rmsnorm_plan_count())]
    assert len(ids) == len(set(ids))
    assert rn.lib().rmsnorm_plan_id_at(len(ids)) == -1


@pytest.mark.parametrize("dt,N,tpr,v,cs", [
    (1, 128, 16, 1, 1), (1, 2048, 64, 4, 1), (1, 4096, 128, 4, 1), (1, 7168, 256, 4, 1), (1, 8192, 256, 4, 1),
    (1, 16384, 512, 4, 1), (0, 256, 32, 2, 1), (0, 2048, 128, 4, 1), (0, 6144, 512, 4, 1),
    (0, 65536, 512, 4, 8),
])
def test_fwd_default_plans(rn, dt, N, tpr, v, cs):
    p = rn.plan_query(rn.OP_FWD, 4096, N, dt)
    assert p["path_name"] == "vector"
    assert (p["threads_per_row"], p["chunks_per_thread"], p["cluster_size"]) == (tpr, v, cs)
    # the row fits the registers of the plan's CTA (or cluster of CTAs)
    per_chunk = 8 if dt == 1 else 4
    assert tpr * v * cs * per_chunk >= N
    assert p["ctas"] == 4096 // p["rows_per_cta"] * cs


@pytest.mark.parametrize("dt,N,cs,v", [(0, 16384, 2, 4), (1, 32768, 2, 4), (1, 65536, 4, 4), (1, 20480, 2, 3),
                                       (1, 40960, 4, 3), (0, 32768, 4, 4), (2, 24576, 2, 3)])
def test_fwd_wide_rows_stream_through_staged_clusters(rn, dt, N, cs, v):
    """Forward rows of 2049..8192 chunks: a persistent grid of clusters whose
    CTAs stream equal slices through two shared-memory stages (x only, or
    x and the residual for the fused variant); no workspace. The E4M3
    outputs keep the register cluster plans."""
    p = rn.plan_query(rn.OP_FWD, 16384, N, dt, num_sms=152, ctas_per_sm=3)
    assert p["path_name"] == "staged" and p["cluster_size"] == cs and p["chunks_per_thread"] == v
    assert p["threads_per_row"] == 512 and p["workspace_bytes"] == 0
    assert p["ctas"] == p["ws_rows"] * cs and p["ws_rows"] == 3 * 152 // cs
    es = 4 if dt == 0 else 2
    slice_bytes = -(-N * es // (16 * cs)) * 16
    assert p["smem_bytes"] == 2 * slice_bytes


@pytest.mark.parametrize("dt,N,cs,v,stages", [(0, 16384, 2, 4, 2), (1, 32768, 2, 4, 2), (1, 65536, 4, 4, 2),
                                              (0, 32768, 4, 4, 2), (1, 20480, 2, 3, 3), (1, 40960, 4, 3, 3)])
@pytest.mark.parametrize("op", ["bwd", "ln"])
def test_bwd_wide_rows_use_clusters(rn, dt, N, cs, v, stages, op):
    """Rows wider than 2048 chunks: a cluster of cs staged CTAs shares each
    row, each streaming an equal slice (a cs-th of the row, whole chunks)
    into its stages; the cluster owns one partial row (two for LayerNorm)."""
    code = rn.OP_BWD if op == "bwd" else rn.OP_LN_BWD
    p = rn.plan_query(code, 16384, N, dt, num_sms=152, ctas_per_sm=1)
    assert p["path_name"] == "staged" and p["cluster_size"] == cs and p["chunks_per_thread"] == v
    assert p["ws_rows"] == 152 // cs and p["ctas"] == p["ws_rows"] * cs
    rows = 1 if op == "bwd" else 2
    assert p["workspace_bytes"] == (p["ws_rows"] * rows * N * 4 + 255) // 256 * 256
    es = 4 if dt == 0 else 2
    slice_bytes = -(-N * es // (16 * cs)) * 16
    assert p["smem_bytes"] == (2 * stages + (op == "ln")) * slice_bytes


@pytest.mark.parametrize("dt,N", [(1, 4097), (1, 8191), (1, 8193), (0, 4097), (1, 65535), (0, 32767), (1, 1), (0, 3)])
def test_fwd_generic_when_vector_cannot_serve(rn, dt, N):
    p = rn.plan_query(rn.OP_FWD, 100, N, dt)
    assert p["path_name"] == "generic"


def test_staged_backward_defaults(rn):
    """Rows of 257..2048 chunks take the staged (bulk-copy pipeline)
    backward: one row team per CTA, `depth` shared-memory stages of x and dy
    rows, a partial row per CTA."""
    for dt, N, tpr, v, stages in ((1, 4096, 256, 2, 4), (1, 8192, 512, 2, 4), (0, 4096, 512, 2, 4),
                                  (1, 12288, 512, 3, 3), (1, 16384, 512, 4, 2), (0, 8192, 512, 4, 2),
                                  (2, 8192, 512, 2, 4), (2, 16384, 512, 4, 2)):
        p = rn.plan_query(rn.OP_BWD, 16384, N, dt, num_sms=152, ctas_per_sm=1)
        assert p["path_name"] == "staged", (dt, N, p)
        assert (p["threads_per_row"], p["chunks_per_thread"], p["cluster_size"]) == (tpr, v, 1)
        es = 4 if dt == 0 else 2
        assert p["smem_bytes"] == stages * 2 * N * es        # plain variant: x and dy rows
        assert p["ctas"] == 152 and p["ws_rows"] == 152
    # the LayerNorm backward's re-read stages keep gamma after the stages
    for dt, N, stages, extra in ((1, 16384, 2, 1), (2, 12288, 2, 1), (0, 6144, 3, 0)):
        p = rn.plan_query(rn.OP_LN_BWD, 16384, N, dt, num_sms=152, ctas_per_sm=1)
        es = 4 if dt == 0 else 2
        assert p["path_name"] == "staged" and p["smem_bytes"] == (2 * stages + extra) * N * es, (dt, N, p)
    # the same rows with an fp32 weight take the same plans
    assert rn.plan_query(rn.OP_BWD, 16384, 8192, rn.RMSNORM_BF16 | rn.RMSNORM_WEIGHT_F32)["path_name"] == "staged"
    # misaligned rows still take the generic kernel; short rows stay in registers
    assert rn.plan_query(rn.OP_BWD, 4096, 8192, 1, aligned=False)["path_name"] == "generic"
    assert rn.plan_query(rn.OP_BWD, 4096, 2048, 1)["path_name"] == "vector"
    # a staged plan is refused for the forward and for rows it cannot hold
    with pytest.raises(rn.RMSNormError):
        rn.plan_query(rn.OP_FWD, 10, 8192, 1, force_plan=88)
    with pytest.raises(rn.RMSNormError):
        rn.plan_query(rn.OP_BWD, 10, 16384, 1, force_plan=88)


def test_fp32_weight_flag_plans(rn):
    """dt | RMSNORM_WEIGHT_F32 selects the activations' default plans; forced
    alternative vector plans are refused (not compiled for that pairing);
    the flag on fp32 activations is the same as fp32. (The register cluster
    plans stay table defaults, for the E4M3 outputs, so they are compiled
    for every pairing although a plain forward streams those rows.)"""
    W = rn.RMSNORM_WEIGHT_F32
    for op in (rn.OP_FWD, rn.OP_BWD):
        for N in (128, 2048, 8192, 16384):
            for base in (rn.RMSNORM_BF16, rn.RMSNORM_F16):
                a = rn.plan_query(op, 4096, N, base, num_sms=152, ctas_per_sm=1)
                b = rn.plan_query(op, 4096, N, base | W, num_sms=152, ctas_per_sm=1)
                assert a == b
            assert (rn.plan_query(op, 4096, N, rn.RMSNORM_F32 | W, num_sms=152, ctas_per_sm=1) ==
                    rn.plan_query(op, 4096, N, rn.RMSNORM_F32, num_sms=152, ctas_per_sm=1))
    default = rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_BF16)["plan_id"]
    defaults = {rn.plan_query(rn.OP_FWD, 64, n, t)["plan_id"] for n in range(8, 65537, 8) for t in (0, 1, 2)}
    refused = 0
    for i in range(rn.lib().rmsnorm_plan_count()):
        pid = rn.lib().rmsnorm_plan_id_at(i)
        try:
            p = rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_BF16, force_plan=pid)
        except rn.RMSNormError:
            continue
        if p["path_name"] == "vector" and p["cluster_size"] == 1 and pid not in defaults:
            with pytest.raises(rn.RMSNormError):
                rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_BF16 | W, force_plan=pid)
            refused += 1
    assert refused > 0
    assert rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_BF16 | W, force_plan=default)["plan_id"] == default
    # the generic plan serves any pairing
    assert rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_F16 | W, force_plan=16)["path_name"] == "generic"
    # unknown flag bits are rejected
    with pytest.raises(rn.RMSNormError):
        rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_BF16 | 0x200)


@pytest.mark.parametrize("dt,N,tpr,v,cs", [(1, 64, 8, 1, 1), (1, 1024, 128, 1, 1), (1, 2048, 128, 2, 1),
                                           (1, 4096, 256, 2, 1), (1, 8192, 256, 4, 1), (0, 8192, 512, 4, 1),
                                           (1, 16384, 512, 4, 1), (1, 12288, 512, 3, 1),
                                           (1, 32768, 512, 4, 2), (1, 65536, 512, 4, 4), (1, 20480, 512, 3, 2)])
def test_layernorm_backward_plans(rn, dt, N, tpr, v, cs):
    p = rn.plan_query(rn.OP_LN_BWD, 16384, N, dt, num_sms=152, ctas_per_sm=1)
    assert p["path_name"] in ("vector", "staged")
    assert (p["threads_per_row"], p["chunks_per_thread"], p["cluster_size"]) == (tpr, v, cs)
    # two partial rows (dgamma | dbeta) per unit
    assert p["workspace_bytes"] == (p["ws_rows"] * 2 * N * 4 + 255) // 256 * 256
    assert rn.plan_query(rn.OP_LN_BWD, 100, N - 1, dt)["path_name"] == "generic"


def test_layernorm_invalid_arguments_without_gpu(rn):
    L = rn.lib()
    x = ctypes.c_void_p(256)
    r = ctypes.c_void_p(512)
    # forward: residual without residual_out, missing mean, an fp32 gamma or
    # beta not 4-byte aligned
    assert L.layernorm_fwd(x, x, x, None, x, None, r, r, 4, 8, 1, 1e-5, 0.0, None) == 1
    assert L.layernorm_fwd(x, None, x, None, x, None, None, r, 4, 8, 1, 1e-5, 0.0, None) == 1
    assert L.layernorm_fwd(x, None, ctypes.c_void_p(258), None, x, None, r, r, 4, 8, 0x101, 1e-5, 0.0, None) == 1
    assert L.layernorm_fwd(x, None, x, ctypes.c_void_p(258), x, None, r, r, 4, 8, 0x101, 1e-5, 0.0, None) == 1
    assert L.layernorm_fwd(x, None, x, None, x, None, r, r, 0, 8, 1, 1e-5, 0.0, None) == 0
    # backward: dgamma without gamma, odd bf16 address, negative eps
    assert L.layernorm_bwd(x, None, x, None, r, r, x, x, None, None, 0, 4, 8, 1, 1e-5, 0.0, None) == 1
    assert L.layernorm_bwd(x, None, ctypes.c_void_p(257), x, r, r, x, x, x, None, 0, 4, 8, 1, 1e-5, 0.0,
                           None) == 1
    assert L.layernorm_bwd(x, None, x, x, r, r, x, x, x, None, 0, 4, 8, 1, -1.0, 0.0, None) == 1
    # a forced alternative forward plan is not compiled for LayerNorm
    assert L.layernorm_fwd_ex(x, None, x, None, x, None, r, r, 4, 2048, 1, 1e-5, 0.0, None, 9, None) == 2


def test_misaligned_pointers_take_generic(rn):
    assert rn.plan_query(rn.OP_FWD, 4096, 7168, 1, aligned=False)["path_name"] == "generic"
    assert rn.plan_query(rn.OP_BWD, 4096, 2048, 0, aligned=False)["path_name"] == "generic"


def test_generic_backward_plan_by_row_length(rn):
    """Rows no vectorised kernel takes (odd N, or arrays at different
    addresses mod 16) run the streamed generic backward whose range holds N,
    with its stages (two slots a stage, each a 16-byte cover of a row at its
    worst offset) in shared memory; longer rows the one-CTA-a-row kernel."""
    expect = ((1, 58), (256, 58), (257, 57), (1024, 57), (1025, 56), (2048, 56), (2049, 43), (4096, 43),
              (4097, 37), (7169, 37), (8192, 37), (8193, 36), (65536, 36))
    for N, pid in expect:
        for dt, es in ((1, 2), (0, 4)):
            p = rn.plan_query(rn.OP_BWD, 4096, N, dt, aligned=False, num_sms=152)
            assert p["plan_id"] == pid and p["path_name"] == "generic", (N, dt, p)
            if pid != 36:
                slot = (N * es + 30) // 16 * 16
                assert p["smem_bytes"] % (2 * slot) == 0 and 2 <= p["smem_bytes"] // (2 * slot) <= 8, (N, dt, p)
                assert p["smem_bytes"] <= 226 * 1024 and p["chunks_per_thread"] == 0
    # one CTA an SM for the widest rows: one partial row an SM
    p = rn.plan_query(rn.OP_BWD, 4096, 7169, 1, aligned=False, num_sms=152)
    assert p["ctas"] == 152 and p["ws_rows"] == 152 and p["workspace_bytes"] == (152 * 7169 * 4 + 255) // 256 * 256
    # aligned rows keep the vectorised plans; the streamed plan may be forced on any layout
    assert rn.plan_query(rn.OP_BWD, 4096, 7168, 1)["path_name"] in ("vector", "staged")
    assert rn.plan_query(rn.OP_BWD, 4096, 7168, 1, force_plan=37)["plan_id"] == 37
    with pytest.raises(rn.RMSNormError):  # a row longer than the plan holds
        rn.plan_query(rn.OP_BWD, 4096, 8193, 1, aligned=False, force_plan=37)


def test_generic_forward_plan_by_row_length(rn):
    """The forward's counterpart: streamed plans (one slot a stage, x's
    cover) up to 16384 elements, the one-CTA-a-row kernel beyond and where
    two stages of the fused variant (x and residual) would not fit: fp32
    rows of 16384 elements."""
    expect = ((1, 104), (256, 104), (257, 105), (1024, 105), (1025, 106), (2048, 106), (2049, 107),
              (4096, 107), (4097, 108), (8192, 108), (8193, 109), (16384, 109), (16385, 16), (65536, 16))
    for N, pid in expect:
        for dt, es in ((1, 2), (0, 4)):
            if es == 4 and N == 16384:
                pid = 16
            p = rn.plan_query(rn.OP_FWD, 4096, N, dt, aligned=False, num_sms=152)
            assert p["plan_id"] == pid and p["path_name"] == "generic", (N, dt, p)
            if pid != 16:
                slot = (N * es + 30) // 16 * 16
                assert p["smem_bytes"] % slot == 0 and 2 <= p["smem_bytes"] // slot <= 6, (N, dt, p)
                assert p["workspace_bytes"] == 0 and p["ctas"] == p["ws_rows"], (N, dt, p)
            else:
                assert p["ctas"] == 4096


def test_plan_independent_of_m(rn):
    for N in (128, 2048, 8192):
        ids = {rn.plan_query(op, M, N, 1)["plan_id"] for op in (0,) for M in (1, 7, 4096, 524288)}
        assert len(ids) == 1
        ids = {rn.plan_query(1, M, N, 1)["plan_id"] for M in (1, 7, 4096, 524288)}
        assert len(ids) == 1


def test_bwd_cta_count_and_workspace(rn):
    p = rn.plan_query(rn.OP_BWD, 16384, 8192, 1, num_sms=152, ctas_per_sm=2)
    assert p["ctas"] == 304 and p["ctas_per_sm"] == 2 and p["ws_rows"] == 304
    assert p["workspace_bytes"] == 304 * 8192 * 4
    # capped by the rows available (rows_per_cta rows per CTA)
    q = rn.plan_query(rn.OP_BWD, 10, 2048, 1, num_sms=152, ctas_per_sm=2)
    assert q["ctas"] == -(-10 // q["rows_per_cta"])
    # forced CTA count
    r = rn.plan_query(rn.OP_BWD, 16384, 8192, 1, num_sms=152, ctas_per_sm=2, force_ctas=77)
    assert r["ctas"] == 77 and r["workspace_bytes"] == (77 * 8192 * 4 + 255) // 256 * 256


def test_forced_plan_rules(rn):
    # a forward plan id is not a backward plan
    with pytest.raises(rn.RMSNormError):
        rn.plan_query(rn.OP_BWD, 10, 8192, 1, force_plan=7)
    # a vector plan too small for the row is refused
    with pytest.raises(rn.RMSNormError):
        rn.plan_query(rn.OP_FWD, 10, 8192, 1, force_plan=0)
    # the generic plan serves anything
    assert rn.plan_query(rn.OP_FWD, 10, 8192, 1, force_plan=16)["path_name"] == "generic"
    assert rn.plan_query(rn.OP_BWD, 10, 5, 0, force_plan=36)["path_name"] == "generic"


def test_invalid_arguments_without_gpu(rn):
    L = rn.lib()
    x = ctypes.c_void_p(256)
    r = ctypes.c_void_p(512)
    # N out of range, null pointers, negative eps, non-finite scalars: all
    # rejected before any CUDA call
    assert L.rmsnorm_fwd(x, x, x, r, 4, 0, 1, 1e-6, 0.0, None) == 1
    assert L.rmsnorm_fwd(x, x, x, r, 4, 65537, 1, 1e-6, 0.0, None) == 1
    assert L.rmsnorm_fwd(None, x, x, r, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert L.rmsnorm_fwd(x, x, x, r, 4, 8, 1, -1.0, 0.0, None) == 1
    assert L.rmsnorm_fwd(x, x, x, r, 4, 8, 1, float("nan"), 0.0, None) == 1
    assert L.rmsnorm_fwd(x, x, x, r, 4, 8, 1, 1e-6, float("inf"), None) == 1
    assert L.rmsnorm_fwd(x, x, x, r, 4, 8, 7, 1e-6, 0.0, None) == 1           # unknown dtype
    assert L.rmsnorm_fwd(x, x, x, r, 4, 8, 0x201, 1e-6, 0.0, None) == 1       # unknown flag
    # an fp32 weight must be 4-byte aligned
    assert L.rmsnorm_fwd(x, ctypes.c_void_p(258), x, r, 4, 8, 0x101, 1e-6, 0.0, None) == 1
    assert L.rmsnorm_fwd(x, x, x, r, -1, 8, 1, 1e-6, 0.0, None) == 1          # negative M
    assert L.rmsnorm_fwd(ctypes.c_void_p(257), x, x, r, 4, 8, 1, 1e-6, 0.0, None) == 1  # odd bf16 address
    assert L.rmsnorm_add_fwd(x, None, x, x, x, r, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert L.rmsnorm_bwd(x, x, x, r, x, None, None, 0, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert L.rmsnorm_bwd(x, x, x, r, x, x, ctypes.c_void_p(264), 1 << 20, 4, 8, 1, 1e-6, 0.0, None) == 3
    # E4M3 forward: unknown scaling, per-tensor without a scale, per-row
    # with a given scale or without scale_inv, an fp32 weight not 4-byte aligned
    f8 = L.rmsnorm_fwd_fp8
    assert f8(x, None, x, x, None, r, 2, None, r, None, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert f8(x, None, x, x, None, r, 0, None, r, None, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert f8(x, None, x, x, None, r, 1, r, r, None, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert f8(x, None, x, x, None, r, 1, None, None, None, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert f8(x, None, x, x, None, r, 0, ctypes.c_void_p(514), None, None, 4, 8, 1, 1e-6, 0.0, None) == 1
    assert f8(x, None, ctypes.c_void_p(258), x, None, r, 1, None, r, None, 4, 8, 0x101, 1e-6, 0.0, None) == 1
    assert f8(x, x, x, x, None, r, 1, None, r, None, 4, 8, 1, 1e-6, 0.0, None) == 1   # residual without out
    # M == 0 forward is a no-op that needs no device
    assert L.rmsnorm_fwd(x, x, x, r, 0, 8, 1, 1e-6, 0.0, None) == 0
    assert L.rmsnorm_status_string(3) == b"workspace too small or misaligned"


def test_workspace_query_without_device_is_zero(rn):
    import torch
    if torch.cuda.is_available():
        pytest.skip("host has a GPU")
    assert rn.rmsnorm_bwd_workspace_bytes(4096, 2048, 1) == 0
    assert rn.rmsnorm_bwd_workspace_bytes(0, 2048, 1) == 0


def test_generic_note_is_optional_and_printed_once(rn, capfd):
    """The generic-kernel note: off by default; once switched on, the first
    call of a kind that falls to the generic kernel prints one line to
    stderr and later ones print nothing; switching it on again re-arms it.
    On a host without a GPU the call then fails at its launch (status 4)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host has a GPU: these addresses are not device memory")
    L = rn.lib()
    # bf16 x and y at different offsets past a 16-byte boundary (at one
    # common offset they would take the vectorised kernels)
    x, y, r = ctypes.c_void_p(258), ctypes.c_void_p(260), ctypes.c_void_p(512)
    L.rmsnorm_set_generic_note(0)
    assert L.rmsnorm_fwd(x, None, y, r, 4, 8, 1, 1e-6, 0.0, None) == 4
    assert "generic kernel" not in capfd.readouterr().err
    L.rmsnorm_set_generic_note(1)
    assert L.rmsnorm_fwd(x, None, y, r, 4, 8, 1, 1e-6, 0.0, None) == 4
    err = capfd.readouterr().err
    assert err.count("falling back to the generic kernel") == 1 and "N=8" in err and "bf16" in err
    assert L.rmsnorm_fwd(x, None, y, r, 4, 8, 1, 1e-6, 0.0, None) == 4
    assert "generic kernel" not in capfd.readouterr().err
    # a row of 7 bf16 elements is not a whole number of 16-byte chunks
    L.rmsnorm_set_generic_note(1)
    assert L.rmsnorm_fwd(ctypes.c_void_p(256), None, ctypes.c_void_p(256), r, 4, 7, 1, 1e-6, 0.0, None) == 4
    assert "whole number of 16-byte chunks" in capfd.readouterr().err
    L.rmsnorm_set_generic_note(0)


def test_common_offset_rows_refuse_forced_alternative_plans(rn):
    """The kernels for rows at a common offset are compiled for the plans of
    the default ranges only: forcing a plan the defaults select on such rows
    is accepted, alternative (tuning) plans are refused, and the generic plan
    still serves them."""
    defaults = {rn.plan_query(op, 64, n, t)["plan_id"] for op in (rn.OP_FWD, rn.OP_BWD, rn.OP_LN_BWD)
                for n in range(8, 65537, 8) for t in (0, 1, 2)}
    refused = accepted = 0
    for op in (rn.OP_FWD, rn.OP_BWD, rn.OP_LN_BWD):
        for i in range(rn.lib().rmsnorm_plan_count()):
            pid = rn.lib().rmsnorm_plan_id_at(i)
            try:
                a = rn.plan_query(op, 64, 2048, rn.RMSNORM_BF16, force_plan=pid)
            except rn.RMSNormError:
                continue
            if a["path_name"] == "generic":
                continue
            if pid in defaults:
                assert rn.plan_query(op, 64, 2048, rn.RMSNORM_BF16, aligned=2, force_plan=pid)["peel"] == 1
                accepted += 1
            else:
                try:
                    p = rn.plan_query(op, 64, 2048, rn.RMSNORM_BF16, aligned=2, force_plan=pid)
                except rn.RMSNormError:
                    refused += 1
                    continue
                # a plan of the default ranges that another one shadows (the
                # register cluster forward beside the staged one)
                assert p["peel"] == 1 and p["cluster_size"] > 1, p
    assert refused > 0 and accepted > 0
    assert rn.plan_query(rn.OP_BWD, 64, 2048, rn.RMSNORM_BF16, aligned=2, force_plan=36)["path_name"] == "generic"


@pytest.mark.parametrize("dt,N,k", [(1, 7168, 1), (1, 8192, 7), (0, 2048, 3), (2, 128, 5), (1, 32768, 2)])
def test_common_offset_plans_match_aligned_plans(rn, dt, N, k):
    """Rows at one common offset (every array k elements past a 16-byte
    boundary) take the plan, CTA count and workspace of aligned rows, with
    the offset reported; an offset that is not a whole element of a chunk
    (k >= 16 / element size) takes the generic kernels."""
    for op in (rn.OP_FWD, rn.OP_BWD, rn.OP_LN_BWD):
        a = rn.plan_query(op, 4096, N, dt, aligned=1, ctas_per_sm=1)
        p = rn.plan_query(op, 4096, N, dt, aligned=1 + k, ctas_per_sm=1)
        assert p["peel"] == k and a["peel"] == 0
        for key in ("plan_id", "ctas", "ws_rows", "workspace_bytes", "threads_per_row", "chunks_per_thread"):
            assert p[key] == a[key], (op, key, p, a)
        if p["path_name"] == "staged":
            # one more 16-byte slot a row buffer (the aligned block that ends the row)
            assert p["smem_bytes"] > a["smem_bytes"]
    es = 4 if dt == 0 else 2
    assert rn.plan_query(rn.OP_BWD, 4096, N, dt, aligned=1 + 16 // es)["path_name"] == "generic"
