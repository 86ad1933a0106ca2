"""The no-allocation entry point, mla_decode_run_noalloc.

It serves callers that cannot allocate device memory for a workspace (for
example a C client running inside a process whose framework owns the device
allocator): the library's own fixed device array stands in for the
workspace.  These tests call it through the C ABI and compare its output
with the regular entry point's on the same inputs, on two calls in a row.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 5e-2          # the fp8-KV tolerance of the parity tests


def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_decode_stage1_gb300 as mla
    from mla_decode_stage1_gb300 import synth
    return mla, synth


def test_noalloc_matches_regular_entry_point_twice():
    mla, synth = _setup()
    w = synth.make_workload(bs=5, lengths=[700, 1, 0, 2049, 300], page_size=16, q_dtype="bf16",
                            kv_dtype="fp8", permute_pages=True, seed=31)
    d = w.to("cuda")
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=w.page_size,
                               q_dtype=w.q_dtype, kv_dtype=w.kv_dtype)
    assert plan.info().num_partials > 0          # the split path uses the workspace
    kw = dict(q_scale=d.q_scale, kv_scale=d.kv_scale, kv_indices=d.kv_indices)

    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty(w.bs, 16, 512, dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(w.bs, 16, dtype=torch.float32, device="cuda")
    mla.mla_decode_run(plan, d.q, d.kv, ref, workspace=ws, lse=ref_lse, **kw)

    # a different plan uses the shared array in between: the next call must
    # not see its leftovers
    other = synth.make_workload(bs=2, lengths=[4096, 33], page_size=1, q_dtype="fp8",
                                kv_dtype="fp8", seed=32).to("cuda")
    oplan = mla.mla_decode_plan(other.kv_indptr, None, page_size=1, q_dtype="fp8", kv_dtype="fp8")
    outs = []
    for i in range(2):
        out = torch.full((w.bs, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.bs, 16), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_run_noalloc(plan, d.q, d.kv, out, lse=lse, **kw)
        tmp = torch.empty(2, 16, 512, dtype=torch.bfloat16, device="cuda")
        mla.mla_decode_run_noalloc(oplan, other.q, other.kv, tmp, q_scale=other.q_scale,
                                   kv_scale=other.kv_scale)
        torch.cuda.synchronize()
        outs.append((out.float().cpu().numpy(), lse.cpu().numpy()))
    r = ref.float().cpu().numpy()
    rl = ref_lse.cpu().numpy()
    for o, l in outs:
        assert np.allclose(o, r, atol=TOL, rtol=TOL)
        assert np.array_equal(np.isneginf(l), np.isneginf(rl))
        fin = np.isfinite(rl)
        assert np.allclose(l[fin], rl[fin], atol=1e-2, rtol=1e-3)


def test_noalloc_rejects_plans_over_the_limit():
    mla, synth = _setup()
    # 256 requests x 32 fixed splits x 32 KB partials is far above 16 MiB
    indptr = np.arange(257, dtype=np.int32) * 8192
    plan = mla.mla_decode_plan(indptr, None, page_size=1, q_dtype="fp8", kv_dtype="fp8",
                               num_splits=32)
    assert plan.workspace_bytes > (16 << 20)
    q = torch.zeros(256, 16, 576, dtype=torch.uint8, device="cuda")
    kv = torch.zeros(16, 576, dtype=torch.uint8, device="cuda")
    out = torch.empty(256, 16, 512, dtype=torch.bfloat16, device="cuda")
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_run_noalloc(plan, q, kv, out, q_scale=s, kv_scale=s)
    assert e.value.status == 3
