"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: the pass bar is atol = rtol = 2e-2 for bf16 KV and 5e-2 for fp8
KV, element by element (the bar the decode spec sets).  Because decode
outputs of flat softmaxes are small (|o| ~ 0.02 for N(0,1) data), each case
also bounds the relative L2 error per (request, head) by REL_L2: bf16 output
rounding is 2^-9 relative, the fp8 path adds its two-term q and p splits
(~2^-8 each), so 1e-2 leaves margin while failing any structural error.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2


def _mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_decode_stage1_gb300 as mla
    return mla


def run_gpu(w, num_splits=0, num_sms=0, **plan_kw):
    mla = _mla()
    import workloads as synth  # noqa: F401
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=w.page_size,
                               q_dtype=w.q_dtype, kv_dtype=w.kv_dtype, num_splits=num_splits,
                               num_sms=num_sms, q_len=w.q_len, **plan_kw)
    d = w.to("cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    rows = w.bs * w.q_len
    out = torch.full((rows, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((rows, 16), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, q_scale=d.q_scale,
                       kv_scale=d.kv_scale, kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices, lse=lse)
    mla.mla_decode_check(plan, ws)
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), plan


def compare(o, lse, o_ref, l_ref, kv_dtype, lengths):
    tol = 2e-2 if kv_dtype == "bf16" else 5e-2
    for b, n in enumerate(lengths):
        if n == 0:
            assert np.all(o[b] == 0.0), f"empty request {b}: out not zero"
            assert np.all(np.isneginf(lse[b])), f"empty request {b}: lse not -inf"
            continue
        assert np.all(np.isfinite(o[b])), f"request {b}: non-finite output"
        bad = ~np.isclose(o[b], o_ref[b], atol=tol, rtol=tol)
        assert not bad.any(), f"request {b}: {bad.sum()} elements off, max err {np.abs(o[b]-o_ref[b]).max()}"
        num = np.linalg.norm(o[b] - o_ref[b], axis=-1)
        den = np.linalg.norm(o_ref[b], axis=-1)
        rel = (num / den).max()
        assert rel < REL_L2, f"request {b}: relative L2 error {rel:.3e}"
        assert np.allclose(lse[b], l_ref[b], atol=1e-2, rtol=1e-3), \
            f"request {b}: lse max err {np.abs(lse[b]-l_ref[b]).max()}"


def check(w, num_splits=0, num_sms=0, select=None, **plan_kw):
    import workloads as synth
    o, lse, plan = run_gpu(w, num_splits=num_splits, num_sms=num_sms, **plan_kw)
    sel = list(range(w.bs)) if select is None else list(select)
    o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(w, select=sel))
    # rows b*q_len + t; query token t of a request with n tokens sees the
    # first n - q_len + 1 + t of them
    ql = w.q_len
    rows = [b * ql + t for b in sel for t in range(ql)]
    seen = [max(0, w.lengths[b] - ql + 1 + t) for b in sel for t in range(ql)]
    compare(o[rows], lse[rows], o_ref, l_ref, w.kv_dtype, seen)
    return plan


COMBOS = [("bf16", "bf16"), ("bf16", "fp8"), ("fp8", "fp8"), ("fp8", "bf16")]


@pytest.mark.parametrize("q_dtype,kv_dtype", COMBOS)
def test_ragged_contiguous(q_dtype, kv_dtype):
    import workloads as synth
    lengths = [1, 127, 128, 129, 300, 0, 1000]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=1, q_dtype=q_dtype,
                            kv_dtype=kv_dtype, seed=21)
    check(w)


@pytest.mark.parametrize("q_dtype,kv_dtype", COMBOS)
@pytest.mark.parametrize("page_size", [1, 2, 3, 4, 8, 12, 16, 24, 256])
def test_paged_permuted_partial_pages(q_dtype, kv_dtype, page_size):
    # page sizes that are multiples of 8 use one TMA box per 8-row group,
    # the others gather every row through its own page-table entry
    import workloads as synth
    lengths = [5, 700, 1, 0, 2049, 383]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=page_size,
                            q_dtype=q_dtype, kv_dtype=kv_dtype, permute_pages=True, seed=22,
                            extra_pool_pages=3)
    check(w)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7])
def test_forced_splits(num_splits):
    import workloads as synth
    lengths = [1, 130, 900, 4096, 0]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=8, q_dtype="bf16",
                            kv_dtype="fp8", permute_pages=True, seed=23)
    check(w, num_splits=num_splits)


@pytest.mark.parametrize("num_sms", [1, 3, 7])
def test_few_ctas_many_items(num_sms):
    # few CTAs: each walks many items and tiles (ring wrap, q double buffer,
    # item boundaries inside the pipeline)
    import workloads as synth
    lengths = [300, 1, 1024, 129, 77, 2000, 0, 640]
    for qd, kd in (("bf16", "fp8"), ("fp8", "fp8"), ("bf16", "bf16")):
        w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=16, q_dtype=qd,
                                kv_dtype=kd, permute_pages=True, seed=24 + num_sms)
        check(w, num_sms=num_sms)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "mxfp4"])
def test_peaked_softmax_and_rescale(kv_dtype):
    # q scaled up: a few tokens dominate, outputs are O(1), and KV rows scaled
    # by a growing factor (before they are encoded) make later tokens score
    # higher, so the running max keeps growing across tiles (the O rescale
    # path) in every format
    import workloads as synth
    lengths = [1500, 640, 3000]
    w = synth.make_workload(bs=3, lengths=lengths, page_size=1, q_dtype="bf16", kv_dtype=kv_dtype,
                            seed=25, q_std=6.0, kv_ramp=(0.5, 1.5))
    check(w, num_sms=2)


def test_bf16_q_wide_range_within_a_request_fp8_kv():
    # bf16 q meeting fp8 KV is split into two e4m3 terms with one scale per
    # request: one head 2^8 larger than the others and the rope dims 2^-6
    # smaller put most elements far below the request's largest |q|
    import workloads as synth
    lengths = [700, 129, 2000, 1]
    w = synth.make_workload(bs=4, lengths=lengths, page_size=8, q_dtype="bf16", kv_dtype="fp8",
                            permute_pages=True, seed=59)
    q = w.q.float()
    q[:, 3, :] *= 2.0 ** 8
    q[:, :, 512:] *= 2.0 ** -6
    w.q = q.to(torch.bfloat16)
    check(w)
    check(w, num_splits=3)


def test_single_request_single_token():
    import workloads as synth
    for qd, kd in COMBOS:
        w = synth.make_workload(bs=1, lengths=[1], page_size=1, q_dtype=qd, kv_dtype=kd, seed=26)
        check(w)


def test_all_empty_batch():
    import workloads as synth
    w = synth.make_workload(bs=2, lengths=[0, 0], page_size=1, q_dtype="bf16", kv_dtype="fp8",
                            seed=27)
    o, lse, _ = run_gpu(w)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("name", ["bs4_kv1024_bf16", "bs32_kv1024_fp8kv"])
def test_small_benchmark_configs_full(name):
    import workloads as synth
    check(synth.make_config(name))


@pytest.mark.parametrize("name", ["bs64_kv8192_fp8kv_page8", "bs256_kv8192_fp8_page8"])
def test_large_benchmark_configs_sampled(name):
    # the full configuration on the GPU, in the launch configuration the
    # benchmark times; the oracle checks a seeded sample of requests
    import workloads as synth
    w = synth.make_config(name, device="cuda")
    rng = np.random.default_rng(7)
    sel = sorted(rng.choice(w.bs, size=6, replace=False).tolist() + [0, w.bs - 1])
    check(w, select=sel)


@pytest.mark.parametrize("page_size,permute", [(1, False), (16, True), (7, True)])
def test_mxfp4_ragged(page_size, permute):
    import workloads as synth
    lengths = [1, 127, 128, 129, 700, 0, 2049]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=page_size, q_dtype="bf16",
                            kv_dtype="mxfp4", permute_pages=permute, seed=41)
    check(w)


def test_mxfp4_wide_scale_rows_and_few_ctas():
    import workloads as synth
    lengths = [300, 1024, 5, 2000]
    w = synth.make_workload(bs=4, lengths=lengths, page_size=1, q_dtype="bf16", kv_dtype="mxfp4",
                            seed=42, scale_stride=48)
    check(w, num_sms=2)
    check(w, num_splits=3)


def test_mxfp4_spread_block_exponents():
    # scale exponents spread over 8 binades inside a token: still exact
    import workloads as synth
    w = synth.make_workload(bs=2, lengths=[500, 77], page_size=1, q_dtype="bf16",
                            kv_dtype="mxfp4", seed=43)
    g = torch.Generator().manual_seed(5)
    w.kv_e8m0[:, :18] = (120 + torch.randint(0, 9, (w.kv_e8m0.shape[0], 18), generator=g)).to(torch.uint8)
    check(w)


def test_mxfp4_very_spread_block_exponents():
    # exponents spread over 30 binades inside a token: blocks more than 8
    # binades below the row's largest are rounded to e4m3 subnormals or to 0
    # (they are then below 2^-8 of that block, far inside the tolerance)
    import workloads as synth
    w = synth.make_workload(bs=3, lengths=[300, 129, 1000], page_size=8, permute_pages=True,
                            q_dtype="bf16", kv_dtype="mxfp4", seed=45)
    g = torch.Generator().manual_seed(6)
    w.kv_e8m0[:, :18] = (100 + torch.randint(0, 31, (w.kv_e8m0.shape[0], 18), generator=g)).to(torch.uint8)
    check(w)


@pytest.mark.parametrize("scale_stride", [18, 32, 48])
@pytest.mark.parametrize("page_size,permute", [(1, False), (3, True), (8, True), (24, True)])
def test_mxfp4_scale_row_strides(scale_stride, page_size, permute):
    # the pages' 18-byte e8m0 rows and wider strides; contiguous and paged
    # pools, a ragged last tile and an empty request
    import workloads as synth
    lengths = [300, 0, 129, 1000, 64]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=page_size,
                            q_dtype="bf16", kv_dtype="mxfp4", permute_pages=permute,
                            seed=44, scale_stride=scale_stride, extra_pool_pages=2)
    assert w.kv_e8m0.shape[1] == scale_stride
    check(w)


def test_mxfp4_benchmark_config_sampled():
    import workloads as synth
    w = synth.make_config("bs256_varkv_mxfp4", device="cuda")
    rng = np.random.default_rng(8)
    sel = sorted(rng.choice(w.bs, size=6, replace=False).tolist() + [0, w.bs - 1])
    check(w, select=sel)


@pytest.mark.parametrize("q_dtype,kv_dtype", COMBOS)
@pytest.mark.parametrize("bs,length,page_size,permute,cs", [
    (4, 1024, 1, False, 8),     # C1's shape: 8 one-tile CTAs per request
    (16, 1024, 8, True, 8),     # paged, permuted: 128 CTAs in 16 clusters
    (3, 1000, 16, True, 8),     # ragged last tile in every request, partial last pages
    (1, 1024, 7, True, 8),      # page size 7: gathered rows (bf16 / fp8 KV)
])
def test_cluster_merge_against_stage2_and_oracle(q_dtype, kv_dtype, bs, length, page_size,
                                                 permute, cs):
    # split requests merged inside stage 1 through a thread-block cluster
    # (distributed shared memory) against the oracle, and against the same
    # plan merged by stage 2
    import workloads as synth
    w = synth.make_workload(bs=bs, lengths=[length] * bs, page_size=page_size, q_dtype=q_dtype,
                            kv_dtype=kv_dtype, permute_pages=permute, seed=61)
    plan = check(w, num_sms=152)
    assert plan.info().cluster_size == cs
    o1, l1, _ = run_gpu(w, num_sms=152)
    o2, l2, plan2 = run_gpu(w, num_sms=152, merge=1)
    assert plan2.info().cluster_size == 0
    assert np.allclose(o1, o2, atol=1e-2, rtol=1e-2) and np.allclose(l1, l2, atol=1e-4, rtol=1e-5)


def test_cluster_merge_repeated_and_bitwise_stable():
    # the cluster path keeps no state between calls: repeated calls give the
    # same bytes
    mla = _mla()
    import workloads as synth
    w = synth.make_workload(bs=4, lengths=[1024] * 4, page_size=1, q_dtype="bf16",
                            kv_dtype="fp8", seed=62)
    plan = mla.mla_decode_plan(w.kv_indptr, None, page_size=1, q_dtype="bf16", kv_dtype="fp8")
    if plan.info().cluster_size == 0:
        pytest.skip("this device's SM count gives no cluster plan for the shape")
    d = w.to("cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(5):
        out = torch.full((4, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((4, 16), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, q_scale=d.q_scale,
                           kv_scale=d.kv_scale, lse=lse)
        outs.append((out, lse))
    mla.mla_decode_check(plan, ws)
    for out, lse in outs[1:]:
        assert torch.equal(out, outs[0][0]) and torch.equal(lse, outs[0][1])


def test_split_merge_repeated_launches_same_workspace():
    # the plan's table is uploaded on the first launch into a workspace only;
    # later launches reuse it and must give identical results
    mla = _mla()
    import workloads as synth
    lengths = [900, 0, 4096, 130, 2500]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=8, q_dtype="bf16",
                            kv_dtype="fp8", permute_pages=True, seed=46)
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=8, q_dtype="bf16",
                               kv_dtype="fp8", num_splits=3)
    assert plan.info().num_partials > 0
    d = w.to("cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(4):
        out = torch.full((w.bs, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.bs, 16), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, q_scale=d.q_scale,
                           kv_scale=d.kv_scale, kv_indices=d.kv_indices, lse=lse)
        outs.append((out.clone(), lse.clone()))
    mla.mla_decode_check(plan, ws)
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(w))
    o = outs[-1][0].float().cpu().numpy().astype(np.float64)
    lse = outs[-1][1].cpu().numpy().astype(np.float64)
    compare(o, lse, o_ref, l_ref, "fp8", w.lengths)


@pytest.mark.parametrize("q_dtype,kv_dtype,q_len", [
    ("bf16", "bf16", 1), ("bf16", "fp8", 1), ("fp8", "fp8", 1), ("fp8", "bf16", 1),
    ("bf16", "mxfp4", 1), ("fp8", "fp8", 2), ("bf16", "fp8", 2)])
def test_soak_interleaved_plans_are_deterministic(q_dtype, kv_dtype, q_len):
    # 300 calls back to back on one stream, without synchronising: two plans
    # of different batches interleaved, plan A alternating between two
    # workspaces (its table is uploaded again on every switch).  No device
    # wait may give up, every repeat must be bitwise identical to the plan's
    # first result, and the first results must match the oracle.
    mla = _mla()
    import workloads as synth
    ps = 1 if kv_dtype == "mxfp4" else 8
    rng = np.random.default_rng(70 + len(q_dtype) + len(kv_dtype) + q_len)
    wa = synth.make_workload(bs=24, lengths=[int(x) for x in rng.integers(0, 3000, 24)], page_size=ps,
                             q_dtype=q_dtype, kv_dtype=kv_dtype, permute_pages=ps > 1,
                             q_len=q_len, seed=71)
    wb = synth.make_workload(bs=5, lengths=[4000, 1, 0, 700, 129], page_size=ps, q_dtype=q_dtype,
                             kv_dtype=kv_dtype, permute_pages=ps > 1, q_len=q_len, seed=72)
    cases = []
    for w, S in ((wa, 0), (wb, 3)):
        plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=ps, q_dtype=q_dtype,
                                   kv_dtype=kv_dtype, num_splits=S, q_len=q_len)
        cases.append((w, plan, w.to("cuda")))
    (wa, pa, da), (wb, pb, db) = cases
    ws = [torch.empty(p.workspace_bytes, dtype=torch.uint8, device="cuda") for p in (pa, pa, pb)]
    n_rep = 100
    outs = {0: [], 1: [], 2: []}

    def call(k, w, plan, d):
        rows = w.bs * w.q_len
        out = torch.empty((rows, 16, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((rows, 16), dtype=torch.float32, device="cuda")
        mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws[k], q_scale=d.q_scale,
                           kv_scale=d.kv_scale, kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices, lse=lse)
        outs[k].append((out, lse))

    for _ in range(n_rep):
        call(0, wa, pa, da)
        call(2, wb, pb, db)
        call(1, wa, pa, da)
    torch.cuda.synchronize()
    for k, plan in ((0, pa), (1, pa), (2, pb)):
        mla.mla_decode_check(plan, ws[k])
    first_a = outs[0][0]
    for k in (0, 1, 2):
        ref = outs[2][0] if k == 2 else first_a
        for o, l in outs[k]:
            assert torch.equal(o, ref[0]) and torch.equal(l, ref[1]), f"workspace {k}: result changed"
    for w, (o, l) in ((wa, first_a), (wb, outs[2][0])):
        o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(w))
        ql = w.q_len
        seen = [max(0, w.lengths[b] - ql + 1 + t) for b in range(w.bs) for t in range(ql)]
        compare(o.float().cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64),
                o_ref, l_ref, w.kv_dtype, seen)


@pytest.mark.parametrize("kv_dtype", ["fp8", "mxfp4"])
def test_one_long_request_over_every_sm(kv_dtype):
    # one request cut into as many items as there are CTAs: stage 2 merges
    # well over a hundred partials per head
    import workloads as synth
    n = 40000
    w = synth.make_workload(bs=2, lengths=[n, 0], page_size=1, q_dtype="bf16",
                            kv_dtype=kv_dtype, seed=47)
    plan = check(w)
    assert plan.info().num_partials >= 100


# ------------------------------------------------- several query tokens

@pytest.mark.parametrize("q_dtype,kv_dtype", COMBOS + [("bf16", "mxfp4")])
@pytest.mark.parametrize("q_len", [2, 4])
def test_qlen_causal_decode(q_dtype, kv_dtype, q_len):
    # requests shorter than q_len leave their first query tokens empty
    import workloads as synth
    lengths = [1, 3, 130, 0, 1000, 2049]
    page = 4
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=page, q_dtype=q_dtype,
                            kv_dtype=kv_dtype, permute_pages=True, seed=48, q_len=q_len)
    check(w)


@pytest.mark.parametrize("q_dtype", ["fp8", "bf16"])
@pytest.mark.parametrize("q_len", [2, 3, 4, 6])
@pytest.mark.parametrize("num_splits,num_sms", [(3, 0), (0, 5), (0, 2)])
def test_qlen_splits_and_few_ctas(num_splits, num_sms, q_len, q_dtype):
    # fp8 KV with an even number of query tokens runs them in pairs (32 q
    # rows per tile; with bf16 q one q buffer, refilled by the softmax warps
    # between items); three tokens run as causal prefixes
    import workloads as synth
    lengths = [700, 5, 4096, 129, 1, 2, 128]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=16, q_dtype=q_dtype,
                            kv_dtype="fp8", permute_pages=True, seed=49, q_len=q_len)
    check(w, num_splits=num_splits, num_sms=num_sms)


def test_qlen2_bf16_pairs_gathered_rows_and_small_rope_dims():
    # bf16 q in pairs with page size 7 (rows gathered one by one), extra pool
    # pages and rope dims 2^-6 smaller than the rest, so the pair's one scale
    # covers a wide range.  (A head made 2^4 to 2^8 larger than the others
    # puts a short request's dominant LSE just outside the LSE bar: the
    # two-term split keeps about 2^-9 of the pair's largest |q|, the same
    # bound as one token, which the one-token test above covers.)
    import workloads as synth
    lengths = [1000, 3, 257, 2049]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=7, q_dtype="bf16",
                            kv_dtype="fp8", permute_pages=True, seed=64, q_len=2,
                            extra_pool_pages=3)
    q = w.q.float()
    q[:, :, 512:] *= 2.0 ** -6                     # rope dims
    w.q = q.to(torch.bfloat16)
    check(w)
    check(w, num_sms=3)


def test_qlen2_fp8_token_zero_without_kv_in_an_item():
    # items that hold only a request's last token leave query token 0 with no
    # token to attend to in that item (partial lse = -inf, weight 0)
    import workloads as synth
    lengths = [129, 257, 1, 2049]
    w = synth.make_workload(bs=4, lengths=lengths, page_size=1, q_dtype="fp8", kv_dtype="fp8",
                            seed=51, q_len=2)
    check(w, num_splits=2)
    check(w, num_sms=11)


def test_qlen2_fp8_peaked_scores():
    # large scores: the running max moves across tiles and the lazy rescale
    # runs on 16-row groups
    import workloads as synth
    w = synth.make_workload(bs=3, lengths=[1500, 640, 3000], page_size=8, q_dtype="fp8",
                            kv_dtype="fp8", permute_pages=True, seed=52, q_len=2, q_std=6.0)
    check(w, num_sms=2)


@pytest.mark.parametrize("q_dtype", ["bf16", "fp8"])
def test_qlen_large_batch_sampled(q_dtype):
    # bs=64 x 8192 tokens, two query tokens, in the balanced launch the
    # planner picks (one CTA group per query token)
    _mla()
    import workloads as synth
    w = synth.make_workload(bs=64, lengths=[8192] * 64, page_size=8, q_dtype=q_dtype,
                            kv_dtype="fp8", permute_pages=True, seed=50, q_len=2, device="cuda")
    rng = np.random.default_rng(9)
    sel = sorted(rng.choice(w.bs, size=4, replace=False).tolist() + [0, w.bs - 1])
    check(w, select=sel)


# ------------------------------------------------- seeded random sweep

def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    q_dtype, kv_dtype = [("bf16", "bf16"), ("bf16", "fp8"), ("fp8", "fp8"), ("fp8", "bf16"),
                         ("bf16", "mxfp4")][rng.integers(5)]
    bs = int(rng.integers(1, 9))
    lengths = [int(x) for x in rng.choice([0, 1, 2, 127, 128, 129, 255, 300, 1000, 2500], size=bs)]
    page_size = int(rng.choice([1, 2, 3, 8, 16, 40, 64]))
    permute = page_size > 1 and bool(rng.integers(2))
    q_len = int(rng.choice([1, 1, 2, 3]))
    mode = int(rng.integers(3))
    num_splits = int(rng.integers(1, 5)) if mode == 1 else 0
    num_sms = int(rng.integers(1, 12)) if mode == 2 else 0
    return dict(bs=bs, lengths=lengths, page_size=page_size, q_dtype=q_dtype, kv_dtype=kv_dtype,
                permute_pages=permute, q_len=q_len), num_splits, num_sms


@pytest.mark.parametrize("seed", range(24))
def test_random_sweep(seed):
    # formats, lengths (empty, partial tiles), page sizes (row gather and
    # 8-row boxes), page permutation, several query tokens, fixed splits and
    # few-CTA plans drawn from one seed; every output against the oracle
    import workloads as synth
    kw, num_splits, num_sms = _random_case(seed)
    w = synth.make_workload(seed=60 + seed, **kw)
    check(w, num_splits=num_splits, num_sms=num_sms)


# Every wait in the kernels is bounded (200 ms), and the waits of hint-only
# roles give up without flagging an error.  A wait that can miss its phase
# would then show only as a call that takes the bound: these cases (several
# tiles and items per CTA, every role layout) must finish far below it.
STALL_CASES = [
    # (q dtype, KV dtype, page size, q_len, CTAs (0 = the device's SMs), batch, length range
    #  [, cut unit in tokens])
    ("fp8", "fp8", 8, 1, 16, 12, (1000, 6000)),
    ("bf16", "fp8", 8, 3, 0, 64, (8192, 8193)),     # bs=64 x 8192, three query tokens
    ("bf16", "fp8", 8, 3, 16, 10, (500, 5000)),
    ("fp8", "fp8", 8, 2, 16, 10, (500, 5000)),
    ("bf16", "fp8", 16, 4, 24, 8, (500, 5000)),
    ("bf16", "bf16", 1, 1, 16, 8, (1000, 6000)),    # one-slot ring, identity table
    ("bf16", "bf16", 8, 3, 16, 8, (500, 5000)),
    ("fp8", "bf16", 8, 1, 0, 16, (1000, 6000)),
    ("bf16", "mxfp4", 1, 1, 16, 8, (1000, 6000)),
    ("bf16", "mxfp4", 8, 3, 16, 8, (500, 5000)),
    ("fp8", "fp8", 12, 1, 16, 8, (1000, 6000)),     # rows gathered one by one
    ("fp8", "bf16", 7, 2, 16, 8, (500, 5000)),
    ("bf16", "bf16", 1, 1, 0, 4, (1024, 1025)),     # eight-way splits merged in clusters
    ("fp8", "fp8", 1, 1, 16, 8, (1000, 6000), 32),  # 32-token cut units (8-row boxes)
    ("bf16", "bf16", 8, 2, 16, 8, (500, 5000), 64),
]


@pytest.mark.parametrize("q_dtype,kv_dtype,page_size,q_len,num_sms,bs,span,unit",
                         [c if len(c) == 8 else c + (0,) for c in STALL_CASES])
def test_calls_finish_far_below_the_wait_bound(q_dtype, kv_dtype, page_size, q_len, num_sms,
                                                bs, span, unit):
    mla = _mla()
    import workloads as synth
    rng = np.random.default_rng(91)
    lengths = rng.integers(span[0], span[1], size=bs).tolist()
    w = synth.make_workload(bs=bs, lengths=lengths, page_size=page_size, q_dtype=q_dtype,
                            kv_dtype=kv_dtype, permute_pages=page_size > 1, seed=92,
                            q_len=q_len, device="cuda")
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=w.page_size,
                               q_dtype=q_dtype, kv_dtype=kv_dtype, num_sms=num_sms, q_len=q_len,
                               unit_tokens=unit)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((bs * q_len, 16, 512), dtype=torch.bfloat16, device="cuda")
    times = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mla.mla_decode_run(plan, w.q, w.kv, out, workspace=ws, q_scale=w.q_scale,
                           kv_scale=w.kv_scale, kv_e8m0=w.kv_e8m0, kv_indices=w.kv_indices)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    mla.mla_decode_check(plan, ws)
    assert max(times) < 20.0, f"a call took {max(times):.1f} ms (the wait bound is 200 ms)"


# ------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_context_survives():
    # a pipeline wait on a barrier nothing arrives on gives up after its
    # limit, the device error word reports it once, and the same context and
    # workspace then decode correctly
    mla = _mla()
    import time
    import workloads as synth
    w = synth.make_workload(bs=3, lengths=[300, 0, 1000], page_size=8, q_dtype="bf16",
                            kv_dtype="fp8", permute_pages=True, seed=53)
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=8, q_dtype="bf16",
                               kv_dtype="fp8", num_splits=2)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    mla.mla_selftest_bounded_wait(plan, ws, limit_us=20000)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_check(plan, ws)
    assert e.value.status == 5                      # MLA_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 >= 0.02          # it waited out its limit
    mla.mla_decode_check(plan, ws)                  # the word was cleared
    d = w.to("cuda")
    out = torch.full((w.bs, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.bs, 16, dtype=torch.float32, device="cuda")
    mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, q_scale=d.q_scale,
                       kv_scale=d.kv_scale, kv_indices=d.kv_indices, lse=lse)
    mla.mla_decode_check(plan, ws)
    o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(w))
    compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            o_ref, l_ref, "fp8", w.lengths)


def test_workspace_reused_by_another_plan_is_detected_in_cluster_mode():
    # as below, with plan A merging inside clusters: the CTAs that find B's
    # stamp still meet at the cluster barriers, write nothing, and the error
    # is reported
    mla = _mla()
    import workloads as synth
    wa = synth.make_workload(bs=4, lengths=[1024] * 4, page_size=1, q_dtype="fp8",
                             kv_dtype="fp8", seed=63)
    wb = synth.make_workload(bs=3, lengths=[50, 5000, 0], page_size=8, q_dtype="fp8",
                             kv_dtype="fp8", permute_pages=True, seed=57)
    pa = mla.mla_decode_plan(wa.kv_indptr, None, page_size=1, q_dtype="fp8", kv_dtype="fp8",
                             num_sms=152)
    pb = mla.mla_decode_plan(wb.kv_indptr, wb.kv_last_page_len, page_size=8, q_dtype="fp8",
                             kv_dtype="fp8", num_splits=3)
    assert pa.info().cluster_size == 8
    da, db = wa.to("cuda"), wb.to("cuda")
    ws = torch.empty(max(pa.workspace_bytes, pb.workspace_bytes), dtype=torch.uint8, device="cuda")

    def run(plan, w, d):
        out = torch.full((w.bs, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.bs, 16), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, q_scale=d.q_scale,
                           kv_scale=d.kv_scale, kv_indices=d.kv_indices, lse=lse)
        return out, lse

    out0, lse0 = run(pa, wa, da)
    mla.mla_decode_check(pa, ws)
    run(pb, wb, db)
    mla.mla_decode_check(pb, ws)
    out1, lse1 = run(pa, wa, da)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_check(pa, ws)
    assert e.value.status == 3
    assert torch.isnan(out1.float()).all() and torch.isnan(lse1).all()
    out2, lse2 = run(pa, wa, da)
    mla.mla_decode_check(pa, ws)
    assert torch.equal(out2, out0) and torch.equal(lse2, lse0)


def test_workspace_reused_by_another_plan_is_detected():
    # plan A uploads its table into a workspace; the same memory then serves
    # as plan B's workspace behind A's back (a caching allocator hands the
    # address out again).  A's next run finds B's stamp: it writes nothing
    # and mla_decode_check reports MLA_ERR_WORKSPACE.  A's run after that
    # uploads its table again and is correct.
    mla = _mla()
    import workloads as synth
    wa = synth.make_workload(bs=4, lengths=[700, 1, 3000, 129], page_size=8, q_dtype="fp8",
                             kv_dtype="fp8", permute_pages=True, seed=56)
    wb = synth.make_workload(bs=3, lengths=[50, 5000, 0], page_size=8, q_dtype="fp8",
                             kv_dtype="fp8", permute_pages=True, seed=57)
    pa = mla.mla_decode_plan(wa.kv_indptr, wa.kv_last_page_len, page_size=8, q_dtype="fp8",
                             kv_dtype="fp8")
    pb = mla.mla_decode_plan(wb.kv_indptr, wb.kv_last_page_len, page_size=8, q_dtype="fp8",
                             kv_dtype="fp8", num_splits=3)
    assert pa.info().num_merge_jobs > 0 and pb.info().num_merge_jobs > 0
    da, db = wa.to("cuda"), wb.to("cuda")
    ws = torch.empty(max(pa.workspace_bytes, pb.workspace_bytes), dtype=torch.uint8, device="cuda")

    def run(plan, w, d):
        out = torch.full((w.bs, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.bs, 16), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, q_scale=d.q_scale,
                           kv_scale=d.kv_scale, kv_indices=d.kv_indices, lse=lse)
        return out, lse

    out0, lse0 = run(pa, wa, da)
    mla.mla_decode_check(pa, ws)
    run(pb, wb, db)                                   # B's table replaces A's
    mla.mla_decode_check(pb, ws)
    out1, lse1 = run(pa, wa, da)                      # A believes its table is there
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_check(pa, ws)
    assert e.value.status == 3                        # MLA_ERR_WORKSPACE
    assert torch.isnan(out1.float()).all() and torch.isnan(lse1).all()   # nothing written
    out2, lse2 = run(pa, wa, da)                      # uploads A's table again
    mla.mla_decode_check(pa, ws)
    assert torch.equal(out2, out0) and torch.equal(lse2, lse0)
    o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(wa))
    compare(out2.float().cpu().numpy().astype(np.float64), lse2.cpu().numpy().astype(np.float64),
            o_ref, l_ref, "fp8", wa.lengths)


@pytest.mark.parametrize("kv_dtype,page_size", [("fp8", 8), ("bf16", 4), ("mxfp4", 8),
                                                ("fp8", 3), ("mxfp4", 5)])
def test_page_outside_the_pool_is_reported(kv_dtype, page_size):
    # one page-table entry of request 1 points past the pool (and one of
    # request 3 is negative): the kernels read page 0 in their place, touch
    # nothing outside the pool, and mla_decode_check reports
    # MLA_ERR_INVALID_ARG once; the other requests are unaffected
    mla = _mla()
    import workloads as synth
    lengths = [300, 200, 129, 77]
    w = synth.make_workload(bs=4, lengths=lengths, page_size=page_size, q_dtype="bf16",
                            kv_dtype=kv_dtype, permute_pages=True, seed=58)
    pool_pages = w.pool_rows // page_size
    ind = w.kv_indices.clone()
    ind[int(w.kv_indptr[1]) + 1] = pool_pages + 7
    ind[int(w.kv_indptr[3])] = -1
    w.kv_indices = ind
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=page_size,
                               q_dtype="bf16", kv_dtype=kv_dtype)
    d = w.to("cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((w.bs, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.bs, 16), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_run(plan, d.q, d.kv, out, workspace=ws, kv_scale=d.kv_scale,
                       kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices, lse=lse)
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_check(plan, ws)
    assert e.value.status == 1                        # MLA_ERR_INVALID_ARG
    mla.mla_decode_check(plan, ws)                    # reported once, then cleared
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all()
    good = [0, 2]
    o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(w, select=good))
    compare(o[good], l[good], o_ref, l_ref, kv_dtype, [lengths[b] for b in good])


def test_decode_call_captures_in_a_cuda_graph():
    # after one run has uploaded the plan's table into the workspace, a call
    # only launches kernels on the stream: it can be captured in a CUDA graph
    # and replayed (stage 2 keeps its programmatic dependency on stage 1)
    mla = _mla()
    import workloads as synth
    w = synth.make_workload(bs=5, lengths=[700, 1, 0, 3000, 129], page_size=8, q_dtype="fp8",
                            kv_dtype="fp8", permute_pages=True, seed=54)
    plan = mla.mla_decode_plan(w.kv_indptr, w.kv_last_page_len, page_size=8, q_dtype="fp8",
                               kv_dtype="fp8", num_sms=8)
    d = w.to("cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(w.bs, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.bs, 16, dtype=torch.float32, device="cuda")
    kw = dict(workspace=ws, q_scale=d.q_scale, kv_scale=d.kv_scale, kv_indices=d.kv_indices,
              lse=lse)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mla.mla_decode_run(plan, d.q, d.kv, out, stream=s, **kw)      # uploads the table
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mla.mla_decode_run(plan, d.q, d.kv, out, stream=s, **kw)
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    mla.mla_decode_check(plan, ws)
    o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(w))
    compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            o_ref, l_ref, "fp8", w.lengths)


@pytest.mark.parametrize("q_len", [1, 2])
def test_many_partials_per_request_wide_merge(q_len):
    # more than 4 partials per request: stage 2 merges with one CTA of eight
    # warps per output row; empty requests and short ones in the same batch
    import workloads as synth
    lengths = [5000, 0, 1, 130, 3000]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=8, q_dtype="fp8",
                            kv_dtype="fp8", permute_pages=True, seed=55, q_len=q_len)
    plan = check(w, num_splits=20)
    assert plan.info().num_partials > 20


# ------------------------------------------------- plan options, autotune

@pytest.mark.parametrize("unit", [32, 64])
@pytest.mark.parametrize("q_dtype,kv_dtype,page_size", [
    ("bf16", "bf16", 1), ("bf16", "fp8", 8), ("fp8", "fp8", 1), ("bf16", "fp8", 3),
    ("bf16", "mxfp4", 1), ("bf16", "mxfp4", 3), ("fp8", "fp8", 16)])
def test_sub_tile_cut_units(unit, q_dtype, kv_dtype, page_size):
    # items that start inside a tile (cut every 32 or 64 tokens): a CTA loads
    # only its rows; ragged and empty requests, page tables and MXFP4
    import workloads as synth
    lengths = [1024, 1024, 300, 0, 77, 129]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=page_size,
                            q_dtype=q_dtype, kv_dtype=kv_dtype, permute_pages=page_size > 1,
                            seed=80)
    plan = check(w, unit_tokens=unit)
    assert plan.info().unit_tokens == unit
    check(w, unit_tokens=unit, item_cost=4, num_sms=7)


@pytest.mark.parametrize("q_len", [1, 2])
def test_sub_tile_cut_units_several_query_tokens(q_len):
    import workloads as synth
    lengths = [700, 5, 1030, 64]
    w = synth.make_workload(bs=len(lengths), lengths=lengths, page_size=8, q_dtype="fp8",
                            kv_dtype="fp8", permute_pages=True, seed=81, q_len=q_len)
    check(w, unit_tokens=32)


@pytest.mark.parametrize("q_dtype,kv_dtype,page_size", [("bf16", "bf16", 1), ("bf16", "mxfp4", 1),
                                                        ("fp8", "fp8", 8)])
def test_autotune_choice_matches_the_oracle(q_dtype, kv_dtype, page_size):
    # every candidate is timed on these inputs; the chosen plan is the one
    # with the smallest median, and its result matches the oracle; the same
    # shape again is served from the cache without timing
    mla = _mla()
    import workloads as synth
    lengths = [1024, 1024, 1024, 1024]
    w = synth.make_workload(bs=4, lengths=lengths, page_size=page_size, q_dtype=q_dtype,
                            kv_dtype=kv_dtype, permute_pages=page_size > 1, seed=82)
    d = w.to("cuda")
    out = torch.empty(4, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(4, 16, dtype=torch.float32, device="cuda")
    kw = dict(page_size=page_size, q_dtype=q_dtype, kv_dtype=kv_dtype, q_scale=d.q_scale,
              kv_scale=d.kv_scale, kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices, lse=lse)
    need = mla.mla_decode_autotune(w.kv_indptr, w.kv_last_page_len, d.q, d.kv, out, **kw)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    plan, table = mla.mla_decode_autotune(w.kv_indptr, w.kv_last_page_len, d.q, d.kv, out,
                                          workspace=ws, reps=3, ignore_cache=True, **kw)
    assert len(table) >= 6 and all(ms > 0 for _, ms in table)
    info = plan.info()
    best = min(table, key=lambda r: r[1])
    chosen = [r for r in table if r[1] == best[1]][0][0]
    assert info.unit_tokens == (chosen["unit_tokens"] or 128)
    assert info.item_cost == (chosen["item_cost"] or 1)
    res = torch.full((4, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    res_lse = torch.full((4, 16), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_run(plan, d.q, d.kv, res, workspace=ws, q_scale=d.q_scale, kv_scale=d.kv_scale,
                       kv_e8m0=d.kv_e8m0, kv_indices=d.kv_indices, lse=res_lse)
    mla.mla_decode_check(plan, ws)
    o_ref, l_ref = oracle.mla_decode(**synth.oracle_args(w))
    compare(res.float().cpu().numpy().astype(np.float64), res_lse.cpu().numpy().astype(np.float64),
            o_ref, l_ref, kv_dtype, lengths)
    plan2, table2 = mla.mla_decode_autotune(w.kv_indptr, w.kv_last_page_len, d.q, d.kv, out,
                                            workspace=ws, reps=3, **kw)
    assert table2 == []
    assert plan2.info().unit_tokens == info.unit_tokens and plan2.info().item_cost == info.item_cost
    assert plan2.info().num_ctas == info.num_ctas
