"""The no-allocation entry point, mla_decode_run_noalloc.

It serves callers that cannot allocate device memory for a workspace (for
example a C client running inside a process whose framework owns the device
allocator): the library's own fixed device array stands in for the
workspace.  These tests call it through the C ABI and compare its output
with the regular entry point's on the same inputs, on two calls in a row.
Both run the same plan through the same kernels, so the results must be
bitwise equal: any difference would be a stale table or leftover partials in
the shared array.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20    # bytes of the library's array


def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_decode_stage1_gb300 as mla
    import workloads
    return mla, workloads


def _regular(mla, plan, w, d):
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    rows = w.bs * w.q_len
    out = torch.empty(rows, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(rows, 16, dtype=torch.float32, device="cuda")
    mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, lse=lse, q_scale=d.q_scale,
                       kv_scale=d.kv_scale, kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices)
    mla.mla_decode_check(plan, ws)
    return out, lse


def _noalloc(mla, plan, w, d):
    rows = w.bs * w.q_len
    out = torch.full((rows, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((rows, 16), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_run_noalloc(plan, d.q, d.kv, out, lse=lse, q_scale=d.q_scale,
                               kv_scale=d.kv_scale, kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices)
    return out, lse


@pytest.mark.parametrize("kv_dtype,page_size", [("fp8", 16), ("mxfp4", 1)])
def test_noalloc_matches_regular_entry_point_twice(kv_dtype, page_size):
    mla, workloads = _setup()
    w = workloads.make_workload(bs=5, lengths=[700, 1, 0, 2049, 300], page_size=page_size,
                                q_dtype="bf16", kv_dtype=kv_dtype, permute_pages=page_size > 1,
                                seed=31)
    d = w.to("cuda")
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=w.page_size,
                               q_dtype=w.q_dtype, kv_dtype=w.kv_dtype)
    assert plan.info().num_partials > 0          # the split path uses the workspace
    ref, ref_lse = _regular(mla, plan, w, d)

    # a different plan uses the shared array in between: the next call must
    # not see its leftovers
    other = workloads.make_workload(bs=2, lengths=[4096, 33], page_size=1, q_dtype="fp8",
                                    kv_dtype="fp8", seed=32).to("cuda")
    oplan = mla.mla_decode_plan(other.kv_indptr, None, page_size=1, q_dtype="fp8", kv_dtype="fp8")
    for _ in range(2):
        out, lse = _noalloc(mla, plan, w, d)
        mla.mla_decode_check(plan, None)
        tmp = torch.empty(2, 16, 512, dtype=torch.bfloat16, device="cuda")
        mla.mla_decode_run_noalloc(oplan, other.q, other.kv, tmp, q_scale=other.q_scale,
                                   kv_scale=other.kv_scale)
        mla.mla_decode_check(oplan, None)
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_noalloc_plan_just_under_the_limit_matches_the_oracle():
    # fixed splits put about 15 MiB of partials in the array
    mla, workloads = _setup()
    import oracle
    w = workloads.make_workload(bs=60, lengths=[1024] * 60, page_size=8, q_dtype="bf16",
                                kv_dtype="fp8", permute_pages=True, seed=33)
    plan = mla.mla_decode_plan(w.kv_indptr, None, page_size=8, q_dtype="bf16", kv_dtype="fp8",
                               num_splits=8)
    assert LIMIT - (2 << 20) < plan.workspace_bytes <= LIMIT
    d = w.to("cuda")
    out, lse = _noalloc(mla, plan, w, d)
    mla.mla_decode_check(plan, None)
    ref, ref_lse = _regular(mla, plan, w, d)
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    sel = [0, 17, 59]
    o_ref, l_ref = oracle.mla_decode(**workloads.oracle_args(w, select=sel))
    o = out.float().cpu().numpy()[sel]
    assert np.allclose(o, o_ref, atol=5e-2, rtol=5e-2)
    assert np.allclose(lse.cpu().numpy()[sel], l_ref, atol=1e-2, rtol=1e-3)


def test_noalloc_reports_a_page_outside_the_pool():
    # device-side errors of a no-allocation call are read with
    # mla_decode_check(plan, None); the next call starts clean
    mla, workloads = _setup()
    w = workloads.make_workload(bs=2, lengths=[300, 200], page_size=8, q_dtype="bf16",
                                kv_dtype="fp8", permute_pages=True, seed=34)
    good = w.to("cuda")
    ind = w.kv_indices.clone()
    ind[int(w.kv_indptr[1])] = w.pool_rows // 8 + 3
    bad = w.to("cuda")
    bad.kv_indices = ind.to("cuda")
    plan = mla.mla_decode_plan(w.kv_indptr, None, page_size=8, q_dtype="bf16", kv_dtype="fp8")
    _noalloc(mla, plan, w, bad)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_check(plan, None)
    assert e.value.status == 1                    # MLA_ERR_INVALID_ARG
    out, lse = _noalloc(mla, plan, w, good)
    mla.mla_decode_check(plan, None)
    ref, ref_lse = _regular(mla, plan, w, good)
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_plans_over_the_limit():
    mla, workloads = _setup()
    # 256 requests x 32 fixed splits x 32 KB partials is far above 16 MiB
    indptr = np.arange(257, dtype=np.int32) * 8192
    plan = mla.mla_decode_plan(indptr, None, page_size=1, q_dtype="fp8", kv_dtype="fp8",
                               num_splits=32)
    assert plan.workspace_bytes > LIMIT
    q = torch.zeros(256, 16, 576, dtype=torch.uint8, device="cuda")
    kv = torch.zeros(16, 576, dtype=torch.uint8, device="cuda")
    out = torch.empty(256, 16, 512, dtype=torch.bfloat16, device="cuda")
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_run_noalloc(plan, q, kv, out, q_scale=s, kv_scale=s)
    assert e.value.status == 3


def test_noalloc_cluster_merge_plan_matches_regular_entry_point():
    # a plan whose split requests merge inside thread-block clusters (no
    # stage 2, no partials in the array) through the no-allocation entry
    mla, workloads = _setup()
    w = workloads.make_workload(bs=4, lengths=[1024] * 4, page_size=1, q_dtype="bf16",
                                kv_dtype="bf16", seed=35)
    plan = mla.mla_decode_plan(w.kv_indptr, None, page_size=1, q_dtype="bf16", kv_dtype="bf16",
                               num_sms=152)
    assert plan.info().cluster_size == 8
    d = w.to("cuda")
    ref, ref_lse = _regular(mla, plan, w, d)
    for _ in range(2):
        out, lse = _noalloc(mla, plan, w, d)
        mla.mla_decode_check(plan, None)
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
