"""CPU tests of the C ABI: the library loads, exports every declared symbol,
validates its arguments, and the planner's work table is a correct and
balanced partition.  No kernel is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")


@pytest.fixture(scope="module")
def mla():
    import __graft_entry__
    __graft_entry__._builder().build()
    import mla_decode_stage1_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(mla):
    names = declared_functions()
    assert len(names) >= 8
    lib = ctypes.CDLL(mla.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mla_decode.h but not exported"
    assert set(names) == set(mla.EXPORTS)


def test_status_strings(mla):
    for code, name in mla.STATUS.items():
        assert mla.mla_status_string(code) == name
    assert mla.mla_status_string(99) == "MLA_ERR_UNKNOWN"


def plan(mla, indptr, last=None, ps=1, qd="bf16", kd="fp8", S=0, sms=148):
    return mla.mla_decode_plan(np.asarray(indptr, np.int32), last, page_size=ps, q_dtype=qd,
                               kv_dtype=kd, num_splits=S, num_sms=sms)


@pytest.mark.parametrize("indptr,last,ps,err", [
    ([0, 5, 3], None, 1, 1),          # decreasing
    ([-1, 5], None, 1, 1),            # negative start
    ([0, 2], [0], 8, 1),              # last page length 0
    ([0, 2], [9], 8, 1),              # last page length > page size
])
def test_plan_rejects_bad_input(mla, indptr, last, ps, err):
    with pytest.raises(mla.MlaError) as e:
        plan(mla, indptr, None if last is None else np.asarray(last, np.int32), ps=ps)
    assert e.value.status == err


def test_plan_rejects_bad_scalars(mla):
    lib = mla._lib
    h = ctypes.c_void_p()
    ind = np.array([0, 4], np.int32)
    p = ind.ctypes.data_as(ctypes.c_void_p)
    assert lib.mla_decode_plan(None, None, 1, 1, 0, 0, 0, 1, ctypes.byref(h)) == 1
    assert lib.mla_decode_plan(p, None, 0, 1, 0, 0, 0, 1, ctypes.byref(h)) == 1
    assert lib.mla_decode_plan(p, None, 1, 0, 0, 0, 0, 1, ctypes.byref(h)) == 1
    assert lib.mla_decode_plan(p, None, 1, 1, 0, 0, -1, 1, ctypes.byref(h)) == 1
    assert lib.mla_decode_plan(p, None, 1, 1, 7, 0, 0, 1, ctypes.byref(h)) == 1
    assert lib.mla_decode_plan(p, None, 1, 1, 0, 0, 0, 1, None) == 1
    assert lib.mla_plan_get_info(None, None) == 1
    assert lib.mla_plan_workspace_size(None, None) == 1


def test_run_rejects_bad_arguments_without_launching(mla):
    pl = plan(mla, [0, 16], ps=1)
    lib = mla._lib
    buf = ctypes.create_string_buffer(1 << 16)
    a = ctypes.addressof(buf)
    a256 = ctypes.c_void_p((a + 255) & ~255)
    # null q / kv / out / workspace
    assert lib.mla_decode_run(pl.handle, None, None, a256, a256, None, 0, 16, None, a256,
                              1 << 12, a256, None, None) == 1
    # misaligned kv
    assert lib.mla_decode_run(pl.handle, a256, None, ctypes.c_void_p(a256.value + 8), a256, None,
                              0, 16, None, a256, 1 << 12, a256, None, None) == 1
    # fp8 KV without a scale pointer
    assert lib.mla_decode_run(pl.handle, a256, None, a256, None, None, 0, 16, None, a256,
                              1 << 12, a256, None, None) == 1
    # workspace too small
    assert lib.mla_decode_run(pl.handle, a256, None, a256, a256, None, 0, 16, None, a256,
                              0, a256, None, None) == 3
    # with a page table, a pool that is not whole pages is invalid
    pl4 = plan(mla, [0, 4], ps=4, qd="bf16", kd="mxfp4")
    assert lib.mla_decode_run(pl4.handle, a256, None, a256, None, a256, 32, 18, a256, a256,
                              1 << 14, a256, None, None) == 1
    # without a page table the requests' rows must lie inside the pool
    assert lib.mla_decode_run(pl.handle, a256, None, a256, a256, None, 0, 15, None, a256,
                              1 << 12, a256, None, None) == 1
    # MXFP4 scale rows: 18 bytes (the pages' rows) and more are accepted; a
    # narrower row is invalid, an odd stride unsupported (rows are read two
    # bytes at a time), a missing scale pointer invalid
    plm = plan(mla, [0, 16], ps=1, qd="bf16", kd="mxfp4")
    assert lib.mla_decode_run(plm.handle, a256, None, a256, None, a256, 16, 16, None, a256,
                              1 << 14, a256, None, None) == 1
    assert lib.mla_decode_run(plm.handle, a256, None, a256, None, a256, 19, 16, None, a256,
                              1 << 14, a256, None, None) == 2
    assert lib.mla_decode_run(plm.handle, a256, None, a256, None,
                              ctypes.c_void_p(a256.value + 1), 18, 16, None, a256,
                              1 << 14, a256, None, None) == 2
    assert lib.mla_decode_run(plm.handle, a256, None, a256, None, None, 18, 16, None, a256,
                              1 << 14, a256, None, None) == 1


def test_unsupported_combinations(mla):
    for qd, kd in (("mxfp4", "fp8"), ("fp8", "mxfp4"), ("mxfp4", "mxfp4")):
        with pytest.raises(mla.MlaError) as e:
            plan(mla, [0, 4], qd=qd, kd=kd)
        assert e.value.status == 2
    plan(mla, [0, 4], qd="bf16", kd="mxfp4")     # supported


def lengths_of(indptr, last, ps):
    n = np.diff(np.asarray(indptr)).astype(np.int64) * ps
    if last is not None:
        n -= np.where(n > 0, ps - np.asarray(last), 0)
    return n


def check_partition(pl, lengths, unit=128):
    ind, items = pl.work()
    info = pl.info()
    assert ind[0] == 0 and ind[-1] == info.num_items and np.all(np.diff(ind) >= 1)
    covered = {b: [] for b in range(len(lengths))}
    for b, t0, t1, slot in items:
        assert 0 <= t0 < t1 <= lengths[b] and t0 % unit == 0
        covered[b].append((t0, t1, slot))
    nslots = set()
    for b, rngs in covered.items():
        rngs.sort()
        if lengths[b] == 0:
            assert rngs == []
            continue
        assert rngs[0][0] == 0 and rngs[-1][1] == lengths[b]
        for (a0, a1, _), (b0, b1, _) in zip(rngs, rngs[1:]):
            assert a1 == b0, "gap or overlap"
        slots = [s for _, _, s in rngs]
        if len(rngs) == 1:
            assert slots == [-1]
        else:
            assert slots == list(range(slots[0], slots[0] + len(slots)))
            nslots.update(slots)
    assert len(nslots) == info.num_partials
    n_split = sum(1 for r in covered.values() if len(r) >= 2)
    n_empty = sum(1 for n in lengths if n == 0)
    assert info.num_merge_jobs == n_split + n_empty
    assert info.total_tokens == sum(lengths)
    return ind, items


def plan_costs(ind, items):
    """Per CTA: 2 per tile plus 1 per item past its first (the planner's cost)."""
    costs = []
    for c in range(len(ind) - 1):
        rng = items[ind[c]:ind[c + 1]]
        costs.append(2 * sum((t1 - t0 + 127) // 128 for _, t0, t1, _ in rng) + len(rng) - 1)
    return costs


def uniform_split_max_cost(lengths, G):
    """The same cost for G equal contiguous tile ranges (the plain split)."""
    tiles = [(n + 127) // 128 for n in lengths]
    owner = [b for b, t in enumerate(tiles) for _ in range(t)]
    T = len(owner)
    G = min(G, T)
    worst = 0
    for i in range(G):
        seg = owner[T * i // G: T * (i + 1) // G]
        worst = max(worst, 2 * len(seg) + len(set(seg)) - 1)
    return worst


@pytest.mark.parametrize("bs,kv,ps,sms", [(256, 8192, 8, 148), (256, 8192, 8, 152), (64, 8192, 8, 152),
                                          (32, 1024, 1, 152), (4, 1024, 1, 152), (3, 100, 1, 152)])
def test_balanced_plan_regular(mla, bs, kv, ps, sms):
    indptr = np.arange(bs + 1) * (kv // ps)
    pl = plan(mla, indptr, ps=ps, sms=sms)
    ind, items = check_partition(pl, [kv] * bs)
    info = pl.info()
    tiles = bs * ((kv + 127) // 128)
    assert 1 <= info.num_ctas <= min(sms, tiles)
    costs = plan_costs(ind, items)
    # never worse than the plain equal split, and within a tile and an item
    # of the ideal share
    assert max(costs) <= uniform_split_max_cost([kv] * bs, sms)
    assert max(costs) <= -(-2 * tiles // min(sms, tiles)) + 3


def test_balanced_plan_avoids_straddling_when_free(mla):
    # 32 requests of 8 tiles on 152 SMs: two tiles of one request per CTA
    # (128 CTAs, no CTA holds two requests) beats 1-2 tiles straddling them
    indptr = np.arange(33) * 1024
    pl = plan(mla, indptr, ps=1, sms=152)
    ind, items = check_partition(pl, [1024] * 32)
    assert pl.info().num_ctas == 128 and np.all(np.diff(ind) == 1)


def test_balanced_plan_ragged_with_last_pages(mla):
    rng = np.random.default_rng(0)
    ps = 16
    lens = rng.integers(0, 5000, 97)
    lens[::13] = 0
    npages = (lens + ps - 1) // ps
    indptr = np.concatenate([[0], np.cumsum(npages)])
    last = np.where(npages > 0, lens - (npages - 1) * ps, ps).astype(np.int32)
    pl = plan(mla, indptr, last, ps=ps, sms=152)
    check_partition(pl, lens_of := lengths_of(indptr, last, ps))
    assert np.array_equal(lens_of, lens)


@pytest.mark.parametrize("S", [1, 2, 3, 7, 32])
def test_fixed_split_plan(mla, S):
    lens = [1, 130, 900, 4096, 0, 128]
    indptr = np.concatenate([[0], np.cumsum(lens)])
    pl = plan(mla, indptr, ps=1, S=S)
    ind, items = check_partition(pl, lens)
    assert np.all(np.diff(ind) == 1)     # one item per CTA
    for b, n in enumerate(lens):
        tiles = (n + 127) // 128
        per = (tiles + S - 1) // S if tiles else 0
        got = [(t0, t1) for bb, t0, t1, _ in items if bb == b]
        exp = [(s * per * 128, min((s + 1) * per * 128, n)) for s in range(S)
               if per and s * per < tiles]
        assert got == exp


def test_workspace_size_covers_partials(mla):
    lens = [4096] * 8
    indptr = np.concatenate([[0], np.cumsum(lens)])
    pl = plan(mla, indptr, ps=1, S=4)
    info = pl.info()
    assert info.num_partials == 32
    assert pl.workspace_bytes >= 32 * 16 * 512 * 4 + 32 * 16 * 4


def test_all_empty_batch_has_no_ctas_and_only_fill_jobs(mla):
    # no tile to stream: stage 1 is not launched; stage 2 writes out = 0 and
    # lse = -inf for every request
    pl = plan(mla, np.array([0, 0, 0, 0]), ps=1)
    info = pl.info()
    assert info.num_ctas == 0 and info.num_items == 0 and info.num_partials == 0
    assert info.num_merge_jobs == 3


# ------------------------------------------------- several query tokens

def plan_q(mla, indptr, q_len, last=None, ps=1, S=0, sms=148):
    # bf16 q and KV: every query token is planned on its own (fp8 KV pairs them)
    return mla.mla_decode_plan(np.asarray(indptr, np.int32), last, page_size=ps, q_dtype="bf16",
                               kv_dtype="bf16", num_splits=S, num_sms=sms, q_len=q_len)


def virtual_lengths(lengths, q_len):
    return [max(0, n - q_len + 1 + t) for n in lengths for t in range(q_len)]


@pytest.mark.parametrize("q_len,S,sms", [(2, 0, 152), (3, 0, 12), (4, 0, 3), (3, 2, 152)])
def test_qlen_plan_covers_causal_prefixes(mla, q_len, S, sms):
    # query token t of request b is row b*q_len + t and covers the request's
    # first n - q_len + 1 + t tokens
    lens = [0, 1, 2, 3, 300, 1000, 4096, 129]
    indptr = np.concatenate([[0], np.cumsum(lens)])
    pl = plan_q(mla, indptr, q_len, S=S, sms=sms)
    info = pl.info()
    assert info.batch_size == len(lens) and info.q_len == q_len
    check_partition(pl, virtual_lengths(lens, q_len))


def test_qlen_plan_groups_ctas_by_query_token(mla):
    # every query token gets its own group of CTAs, each balanced over all
    # requests, so CTA i of each group reads the same KV ranges
    q_len, sms, bs, kv = 3, 12, 8, 2048
    indptr = np.arange(bs + 1) * kv
    pl = plan_q(mla, indptr, q_len, sms=sms)
    ind, items = pl.work()
    info = pl.info()
    assert info.num_ctas == sms
    per = sms // q_len
    for c in range(sms):
        toks = {int(r) % q_len for r, _, _, _ in items[ind[c]:ind[c + 1]]}
        assert toks == {c // per}
    for i in range(per):
        ranges = [[(int(r) // q_len, int(t0)) for r, t0, _, _ in items[ind[g * per + i]:ind[g * per + i + 1]]]
                  for g in range(q_len)]
        assert ranges[0] == ranges[1] == ranges[2]


def test_qlen_plan_rejects_bad_q_len(mla):
    for q_len in (0, -1, 65):
        with pytest.raises(mla.MlaError) as e:
            plan_q(mla, [0, 10], q_len)
        assert e.value.status == 1


@pytest.mark.parametrize("qd", ["fp8", "bf16"])
@pytest.mark.parametrize("S,sms", [(0, 152), (0, 7), (3, 152)])
def test_qlen2_fp8_plans_whole_requests(mla, S, sms, qd):
    # two query tokens with fp8 KV (fp8 or bf16 q) share every tile: the plan
    # covers each request's tokens once, and a partial holds 32 rows (2 x 16
    # heads)
    lens = [0, 1, 2, 300, 1000, 4096, 129]
    indptr = np.concatenate([[0], np.cumsum(lens)])
    pl = mla.mla_decode_plan(np.asarray(indptr, np.int32), None, page_size=1, q_dtype=qd,
                             kv_dtype="fp8", num_splits=S, num_sms=sms, q_len=2)
    info = pl.info()
    assert info.batch_size == len(lens) and info.q_len == 2
    check_partition(pl, lens)
    assert pl.workspace_bytes >= info.num_partials * 32 * (512 + 1) * 4


@pytest.mark.parametrize("qd", ["fp8", "bf16"])
def test_even_qlen_fp8_plans_pairs_of_query_tokens(mla, qd):
    # q_len = 4 with fp8 KV: pair p of request b is planned request 2b + p,
    # covering the tokens its second query token sees
    lens = [0, 1, 3, 4, 300, 1000]
    indptr = np.concatenate([[0], np.cumsum(lens)])
    pl = mla.mla_decode_plan(np.asarray(indptr, np.int32), None, page_size=1, q_dtype=qd,
                             kv_dtype="fp8", num_sms=20, q_len=4)
    pair_lens = [max(0, n - 4 + 2 + 2 * p) for n in lens for p in range(2)]
    check_partition(pl, pair_lens)
    assert pl.info().batch_size == len(lens) and pl.info().q_len == 4


# ------------------------------------------------- randomized plan sweep

def _random_batch(rng):
    bs = int(rng.choice([1, 2, 5, 17, 64, 300]))
    kind = rng.integers(0, 3)
    if kind == 0:        # short requests, many empty
        lens = rng.integers(0, 300, bs)
    elif kind == 1:      # long requests
        lens = rng.integers(1000, 20000, bs)
    else:                # a mix with empties
        lens = np.where(rng.random(bs) < 0.2, 0, rng.integers(1, 9000, bs))
    return lens.astype(np.int64)


@pytest.mark.parametrize("seed", range(120))
def test_randomized_plans_partition_every_query_token(mla, seed):
    """Any batch, page size, last-page layout, SM count, forced split and
    q_len: the work table covers every planned request's visible tokens
    exactly once, with consecutive partial slots and enough workspace.  The
    balanced plan's most expensive CTA never costs more than with the plain
    equal split of the tiles."""
    rng = np.random.default_rng(1000 + seed)
    lens = _random_batch(rng)
    ps = int(rng.choice([1, 2, 3, 8, 16, 64, 256]))
    npages = (lens + ps - 1) // ps
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    use_last = ps > 1 and rng.random() < 0.7
    last = (np.where(npages > 0, lens - (npages - 1) * ps, ps).astype(np.int32)
            if use_last else None)
    n = lens if use_last else npages * ps                   # tokens the plan sees
    sms = int(rng.choice([1, 3, 17, 148, 152]))
    S = int(rng.choice([0, 0, 0, 1, 2, 5, 32]))
    q_len = int(rng.choice([1, 1, 2, 3, 4]))
    qd, kd = [("bf16", "fp8"), ("fp8", "fp8"), ("bf16", "bf16"), ("bf16", "mxfp4")][rng.integers(0, 4)]
    pl = mla.mla_decode_plan(indptr, last, page_size=ps, q_dtype=qd, kv_dtype=kd, num_splits=S,
                             num_sms=sms, q_len=q_len)
    info = pl.info()
    assert info.batch_size == len(lens) and info.q_len == q_len
    pairs = q_len % 2 == 0 and kd == "fp8"
    if pairs:
        vlens = [max(0, int(x) - q_len + 2 + 2 * p) for x in n for p in range(q_len // 2)]
    else:
        vlens = virtual_lengths([int(x) for x in n], q_len)
    ind, items = check_partition(pl, vlens)
    if S == 0:
        assert info.num_ctas <= sms
    rows = 32 if pairs else 16
    assert pl.workspace_bytes >= info.num_partials * rows * (512 + 1) * 4
    if S == 0 and q_len == 1 and info.num_ctas > 0:
        assert max(plan_costs(ind, items)) <= uniform_split_max_cost(vlens, sms)


# ------------------------------------------------- plan options and autotune

def plan_ex(mla, indptr, ps=1, qd="bf16", kd="fp8", S=0, sms=152, item_cost=0, unit=0):
    return mla.mla_decode_plan(np.asarray(indptr, np.int32), None, page_size=ps, q_dtype=qd,
                               kv_dtype=kd, num_splits=S, num_sms=sms, item_cost=item_cost,
                               unit_tokens=unit)


@pytest.mark.parametrize("unit", [32, 64, 128])
@pytest.mark.parametrize("bs,kv", [(4, 1024), (32, 1024), (5, 777), (64, 8192)])
def test_plan_cut_units(mla, unit, bs, kv):
    # finer cut points: every item starts on a unit boundary, the partition
    # still covers every token once, and a small batch spreads over more CTAs
    indptr = np.arange(bs + 1) * kv
    pl = plan_ex(mla, indptr, unit=unit)
    check_partition(pl, [kv] * bs, unit=unit)
    info = pl.info()
    assert info.unit_tokens == unit
    units = bs * -(-kv // unit)
    if units <= 152:
        assert info.num_ctas == units          # one unit per CTA
    else:
        assert 1 <= info.num_ctas <= 152
    assert info.total_tiles == bs * -(-kv // 128)


def test_plan_item_cost_bounds(mla):
    # under its own item cost, the balanced plan's most expensive CTA is
    # never dearer than that of the plain equal split of the tiles (the bound
    # the planner's bisection starts from)
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 3000, 300)
    indptr = np.concatenate([[0], np.cumsum(lens)])
    tiles = [(n + 127) // 128 for n in lens]
    owner = [b for b, t in enumerate(tiles) for _ in range(t)]
    T, G = len(owner), 152
    for cost in (1, 2, 4, 16):
        pl = plan_ex(mla, indptr, item_cost=cost)
        ind, items = check_partition(pl, lens)
        assert pl.info().item_cost == cost
        worst = max(2 * sum((t1 - t0 + 127) // 128 for _, t0, t1, _ in items[ind[c]:ind[c + 1]])
                    + cost * (ind[c + 1] - ind[c] - 1) for c in range(len(ind) - 1))
        equal = max(2 * len(seg) + cost * (len(set(seg)) - 1)
                    for seg in (owner[T * i // G: T * (i + 1) // G] for i in range(G)) if seg)
        assert worst <= equal


def test_plan_options_validated(mla):
    indptr = np.array([0, 100], np.int32)
    for kw in (dict(unit=48), dict(unit=256), dict(item_cost=-1), dict(item_cost=65)):
        with pytest.raises(mla.MlaError) as e:
            plan_ex(mla, indptr, **kw)
        assert e.value.status == 1
    # all zero is the default plan
    a, b = plan_ex(mla, indptr).work(), plan(mla, indptr, sms=152).work()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_autotune_selects_the_smallest_median(mla):
    sel = mla.mla_autotune_select
    assert sel([[3.0, 1.0, 2.0], [2.5, 2.4, 2.6], [9.0, 0.1, 9.0]]) == 0   # medians 2, 2.5, 9
    assert sel([[3.0, 3.1, 2.9], [2.5, 2.4, 2.6], [0.1, 9.0, 9.0]]) == 1   # medians 3, 2.5, 9
    assert sel([[5.0, 5.0, 5.0], [-1.0, 0.1, 0.1], [4.0, 6.0, 4.5]]) == 2  # a run with -1 is skipped
    assert sel([[2.0, 2.0], [2.0, 2.0], [1.0, 3.0]]) == 0                  # ties: the first
    assert sel([[1.0, 4.0], [2.0, 2.2]]) == 1                              # even reps: mean of the middle two
    assert sel([[float("nan"), 1.0], [7.0, 7.0]]) == 1                     # NaN: not run
    with pytest.raises(mla.MlaError):
        sel([[-1.0], [-2.0]])


def test_autotune_workspace_query_without_a_gpu(mla):
    # workspace NULL: the plans are built and the largest workspace reported;
    # nothing is launched (so this runs on a host without a GPU)
    lib = mla._lib
    indptr = np.arange(5, dtype=np.int32) * 1024
    need = ctypes.c_size_t()
    nres = ctypes.c_int32()
    st = lib.mla_decode_autotune(indptr.ctypes.data_as(ctypes.c_void_p), None, 4, 1, 1, 0, 1,
                                 None, None, None, None, None, 0, 4096, None, None, 0, None, None,
                                 3, 0, None, None, 0, ctypes.byref(nres), ctypes.byref(need),
                                 None)
    # (num_sms 0 needs the device: without a GPU the query reports MLA_ERR_CUDA)
    assert st in (0, 4)
    if st == 0:
        assert need.value > 0 and nres.value == 0


def expected_cluster(cta_indptr, items, bs):
    """The rule, restated: every CTA holds one item and every request is split
    over 8 consecutive CTAs (one cluster per request)."""
    if len(cta_indptr) < 3 or not np.all(np.diff(cta_indptr) == 1):
        return 0
    b = items[:, 0]
    per_req = np.bincount(b, minlength=bs)
    cs = int(per_req[0])
    if cs != 8 or np.any(per_req != cs) or np.any(items[:, 3] < 0):
        return 0
    for k in range(len(b) // cs):
        if len(set(b[k * cs:(k + 1) * cs].tolist())) != 1:
            return 0
    return cs


@pytest.mark.parametrize("bs,kv,sms,qd,kd,want", [
    (4, 1024, 152, "bf16", "bf16", 8),     # 32 one-tile CTAs, 8 per request
    (32, 1024, 152, "bf16", "fp8", 0),     # 4 CTAs of 2 tiles per request: stage 2 is faster
    (8, 512, 152, "fp8", "fp8", 0),        # 4 one-tile CTAs per request
    (16, 1024, 152, "fp8", "fp8", 8),      # 128 one-tile CTAs, 8 per request
    (64, 8192, 152, "bf16", "fp8", 0),     # CTAs straddle requests: stage 2
    (1, 2048, 8, "bf16", "fp8", 8),        # 8 CTAs of 2 tiles
    (3, 1000, 152, "bf16", "fp8", 8),      # 24 CTAs, the last tile of each request ragged
    (5, 300, 152, "bf16", "fp8", 0),       # 3 tiles per request: no cluster size fits
])
def test_cluster_merge_plans(mla, bs, kv, sms, qd, kd, want):
    indptr = np.arange(bs + 1, dtype=np.int32) * kv
    pl = plan(mla, indptr, qd=qd, kd=kd, sms=sms)
    info = pl.info()
    cta_indptr, items = pl.work()
    assert expected_cluster(cta_indptr, items, bs) == want
    assert info.cluster_size == want
    # the stage-2 form of the same plan on request (merge=1)
    pl2 = mla.mla_decode_plan(indptr, None, page_size=1, q_dtype=qd, kv_dtype=kd, num_sms=sms,
                              merge=1)
    assert pl2.info().cluster_size == 0
    assert np.array_equal(pl2.work()[1], items)


@pytest.mark.parametrize("seed", range(40))
def test_cluster_merge_rule_on_random_batches(mla, seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.integers(1, 20))
    equal = rng.random() < 0.6
    lens = np.full(bs, int(rng.integers(1, 2048))) if equal else rng.integers(0, 2048, bs)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sms = int(rng.choice([4, 16, 64, 152]))
    pl = plan(mla, indptr, sms=sms)
    cta_indptr, items = pl.work()
    assert pl.info().cluster_size == expected_cluster(cta_indptr, items, bs)


def test_no_cluster_merge_for_mxfp4_or_several_tokens(mla):
    eq = np.arange(5, dtype=np.int32) * 1024
    assert plan(mla, eq, sms=152).info().cluster_size == 8
    assert plan(mla, eq, kd="mxfp4", sms=152).info().cluster_size == 0
    pq = mla.mla_decode_plan(eq, None, page_size=1, q_dtype="fp8", kv_dtype="fp8", num_sms=152,
                             q_len=2)
    assert pq.info().cluster_size == 0
    pq = mla.mla_decode_plan(eq, None, page_size=1, q_dtype="bf16", kv_dtype="fp8", num_sms=152,
                             q_len=3)
    assert pq.info().cluster_size == 0
    # an empty request keeps stage 2 (it zero-fills that request)
    with_empty = np.array([0, 1024, 1024, 2048, 3072, 4096], np.int32)
    assert plan(mla, with_empty, sms=152).info().cluster_size == 0
