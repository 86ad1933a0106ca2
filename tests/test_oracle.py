"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: a format table the
pages print, a library decoder, a closed form of softmax attention, or an
invariant the definition implies.  Together they are chosen so that a
plausible slip in the oracle (a dropped rope dimension, a wrong scale, a
swapped nibble, a head/token index mix-up, a wrong V slice, a sign error in
the merge) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden

H, D, DV = 16, 576, 512
BF16, FP8, MXFP4 = 0, 1, 2


def bf16_bits(x):
    """float array -> bf16 bit patterns (values must already be bf16-exact)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def rand_bf16(rng, shape, scale=1.0):
    t = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.float().numpy().astype(np.float64)


def run(q_bits, kv_bits, lengths, page_size=1, kv_indices=None, last=None, num_splits=0,
        q_dtype=BF16, kv_dtype=BF16, **kw):
    bs = len(lengths)
    npages = [(n + page_size - 1) // page_size for n in lengths]
    indptr = np.zeros(bs + 1, np.int32)
    indptr[1:] = np.cumsum(npages)
    return oracle.mla_decode(bs=bs, page_size=page_size, q_dtype=q_dtype, kv_dtype=kv_dtype,
                             q=q_bits, kv=kv_bits, kv_indptr=indptr, kv_indices=kv_indices,
                             kv_last_page_len=last, num_splits=num_splits, nthreads=4, **kw)


# ---------------------------------------------------------------- formats

def test_constants_match_pages():
    c = {k: int(v) for k, v in golden("mla_constants.txt")}
    assert (oracle.HEADS, oracle.QK_DIM, oracle.V_DIM) == (c["num_heads"], c["qk_head_dim"], c["v_head_dim"])
    assert c["kv_lora_rank"] + c["qk_rope_head_dim"] == c["qk_head_dim"]
    # one token, q = e_0 * 24, k = e_0: the score is exactly 1 if sm_scale = 1/24
    q = np.zeros((1, H, D), np.float32); q[0, :, 0] = 24.0
    kv = np.zeros((1, D), np.float32); kv[0, 0] = 1.0
    _, lse = run(bf16_bits(q), bf16_bits(kv), [1])
    assert np.allclose(lse, 1.0 / c["sm_scale_inverse"] * 24.0, rtol=0, atol=1e-15)


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode("e4m3", codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e2m1_matches_page_lut():
    rows = golden("e2m1_lut.txt")
    codes = np.array([int(r[0]) for r in rows], np.uint8)
    vals = np.array([float(r[1]) for r in rows])
    ours = oracle.decode("e2m1", codes)
    assert np.array_equal(ours, vals)
    # the sign of the zero at code 8 follows the format (see the file's header)
    assert np.array_equal(np.signbit(ours), np.signbit(vals))


def test_e8m0_is_power_of_two():
    e = np.arange(256, dtype=np.uint8)
    ours = oracle.decode("e8m0", e)
    for i in range(255):
        assert ours[i] == math.ldexp(1.0, i - 127)
    assert np.isnan(ours[255])


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, 4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]          # drop inf/NaN patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.decode("bf16", bits), ref)


def test_mxfp4_nibble_order_and_scale_blocks():
    # one row: element 2i in the low nibble of byte i, 2i+1 in the high nibble;
    # scale byte j multiplies elements 32j .. 32j+31.  Row stride 32 with junk
    # after the 18 used scale bytes.
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 16, (2, D)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = rng.integers(120, 135, (2, 32)).astype(np.uint8)
    sc[:, 18:] = 0xFF                                 # must never be read
    out = oracle.dequant_kv(MXFP4, packed, e8m0=sc, e8m0_stride=32)
    lut = {int(r[0]): float(r[1]) for r in golden("e2m1_lut.txt")}
    for r in range(2):
        for d in range(D):
            assert out[r, d] == lut[int(codes[r, d])] * 2.0 ** (int(sc[r, d // 32]) - 127)
    # a single high nibble set lands on the odd element only
    one = np.zeros((1, D // 2), np.uint8); one[0, 5] = 0x20       # code 2 (=1.0) at element 11
    s = np.full((1, 18), 127, np.uint8); s[0, 0] = 128             # block 0 scaled by 2
    v = oracle.dequant_kv(MXFP4, one, e8m0=s, e8m0_stride=18)[0]
    assert v[11] == 2.0 and np.count_nonzero(v) == 1


def test_fp8_kv_scale_applied():
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    rows = np.resize(codes, (2, D)).astype(np.uint8)
    out = oracle.dequant_kv(FP8, rows, kv_scale=0.375)
    ref = torch.from_numpy(rows).view(torch.float8_e4m3fn).to(torch.float64).numpy() * 0.375
    assert np.array_equal(out, ref)


# ---------------------------------------------------------- closed forms

def test_zero_query_gives_mean_of_v():
    rng = np.random.default_rng(2)
    for n in (1, 5, 33):
        kvb, kvf = rand_bf16(rng, (n, D))
        q = np.zeros((1, H, D), np.uint16)
        o, lse = run(q, kvb, [n])
        assert np.allclose(o[0], kvf[:, :DV].mean(0)[None, :], rtol=0, atol=1e-14)
        assert np.allclose(lse, math.log(n), rtol=0, atol=1e-14)


def test_single_token_returns_v_row_and_its_score():
    # q[h] = a_h * e_{d_h}: the score is a_h * k[d_h] / 24, exactly known.
    rng = np.random.default_rng(3)
    kvb, kvf = rand_bf16(rng, (1, D))
    q = np.zeros((1, H, D), np.float32)
    dims = [0, 100, 511, 512, 540, 575] + list(range(200, 210))
    a = [float(2 ** (h % 5)) * (-1) ** h for h in range(H)]
    for h in range(H):
        q[0, h, dims[h]] = a[h]
    o, lse = run(bf16_bits(q), kvb, [1])
    for h in range(H):
        assert np.array_equal(o[0, h], kvf[0, :DV])
        assert abs(lse[0, h] - a[h] * kvf[0, dims[h]] / 24.0) < 1e-14


def test_two_tokens_sigmoid_weights():
    # s_j = a_h k_j[d_h] / 24 with d_h in both latent and rope dims; the output
    # is sigma(s0 - s1) v0 + sigma(s1 - s0) v1 and v is the first 512 dims only.
    rng = np.random.default_rng(4)
    kvb, kvf = rand_bf16(rng, (2, D), scale=3.0)
    q = np.zeros((1, H, D), np.float32)
    dims = [h * 37 % D for h in range(H)]
    dims[3], dims[7], dims[11] = 512, 560, 575
    a = [float(1 + h) for h in range(H)]
    for h in range(H):
        q[0, h, dims[h]] = a[h]
    o, lse = run(bf16_bits(q), kvb, [2])
    for h in range(H):
        s0, s1 = a[h] * kvf[0, dims[h]] / 24.0, a[h] * kvf[1, dims[h]] / 24.0
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        exp_o = w0 * kvf[0, :DV] + (1.0 - w0) * kvf[1, :DV]
        assert np.allclose(o[0, h], exp_o, rtol=1e-13, atol=1e-13)
        m = max(s0, s1)
        assert abs(lse[0, h] - (m + math.log(math.exp(s0 - m) + math.exp(s1 - m)))) < 1e-13


def test_constant_v_rows_give_that_value():
    rng = np.random.default_rng(5)
    n = 40
    kvb, kvf = rand_bf16(rng, (n, D))
    c = kvf[0, :DV].copy()
    kvb[:, :DV] = kvb[0, :DV]          # V identical; rope dims still differ per token
    qb, _ = rand_bf16(rng, (1, H, D))
    o, _ = run(qb, kvb, [n])
    assert np.allclose(o[0], c[None, :], rtol=0, atol=1e-13)


def test_dominant_token_and_large_scores():
    # huge scores must not overflow; the token with the largest score wins.
    rng = np.random.default_rng(6)
    n = 9
    kvb, kvf = rand_bf16(rng, (n, D))
    q = np.zeros((1, H, D), np.float32)
    q[0, :, 540] = 2.0 ** 20
    o, lse = run(bf16_bits(q), kvb, [n])
    j = int(np.argmax(kvf[:, 540]))
    assert np.allclose(o[0], kvf[j, :DV][None, :], rtol=0, atol=1e-12)
    assert np.all(np.isfinite(lse))


def test_empty_request():
    rng = np.random.default_rng(7)
    kvb, _ = rand_bf16(rng, (3, D))
    qb, _ = rand_bf16(rng, (2, H, D))
    o, lse = run(qb, kvb, [0, 3])
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# ------------------------------------------------------------ invariants

def test_page_permutation_and_partial_last_page():
    rng = np.random.default_rng(8)
    ps, n = 4, 23                               # 6 pages, last one holds 3 tokens
    kvb, _ = rand_bf16(rng, (n, D))
    qb, _ = rand_bf16(rng, (1, H, D))
    o_ref, l_ref = run(qb, kvb, [n])            # contiguous, page size 1
    perm = rng.permutation(6)
    pool = np.zeros((6 * ps, D), np.uint16)
    for logical, phys in enumerate(perm):
        src = kvb[logical * ps: (logical + 1) * ps]
        pool[phys * ps: phys * ps + len(src)] = src
    # garbage in the unused slot of the last page must not matter
    pool[perm[5] * ps + 3] = bf16_bits(np.full(D, 7.0, np.float32))
    o, l = run(qb, pool, [n], page_size=ps, kv_indices=perm.astype(np.int32),
               last=np.array([3], np.int32))
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12) and np.allclose(l, l_ref, rtol=0, atol=1e-12)


def test_token_order_invariance():
    rng = np.random.default_rng(9)
    n = 17
    kvb, _ = rand_bf16(rng, (n, D))
    qb, _ = rand_bf16(rng, (1, H, D))
    o1, l1 = run(qb, kvb, [n])
    o2, l2 = run(qb, kvb[rng.permutation(n)], [n])
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S", [2, 3, 7, 32])
def test_split_merge_invariance(S):
    rng = np.random.default_rng(10 + S)
    lengths = [1, 5, 29, 64]
    kvb, _ = rand_bf16(rng, (sum(lengths), D))
    qb, _ = rand_bf16(rng, (len(lengths), H, D))
    o1, l1 = run(qb, kvb, lengths)
    o2, l2 = run(qb, kvb, lengths, num_splits=S)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)


def test_kv_and_q_rescaling():
    # scale KV rows by 2 and q by 1/2: scores unchanged, o doubles, lse unchanged.
    rng = np.random.default_rng(11)
    n = 12
    kvb, kvf = rand_bf16(rng, (n, D))
    qb, qf = rand_bf16(rng, (1, H, D))
    o1, l1 = run(qb, kvb, [n])
    o2, l2 = run(bf16_bits(qf * 0.5), bf16_bits(kvf * 2.0), [n])
    assert np.allclose(o2, 2.0 * o1, rtol=1e-13, atol=0) and np.allclose(l1, l2, rtol=0, atol=1e-13)


def test_fp8_scales_enter_scores_and_values():
    # fp8 KV with kv_scale s and fp8 q with q_scale t equal bf16 runs on the
    # decoded values times the scales.
    rng = np.random.default_rng(12)
    n = 10
    kv_codes = rng.integers(0, 256, (n, D)).astype(np.uint8)
    kv_codes[(kv_codes & 0x7F) == 0x7F] = 0x10
    q_codes = rng.integers(0, 256, (1, H, D)).astype(np.uint8)
    q_codes[(q_codes & 0x7F) == 0x7F] = 0x11
    s, t = 0.125, 0.0078125
    kvf = torch.from_numpy(kv_codes).view(torch.float8_e4m3fn).float().numpy() * s
    qf = torch.from_numpy(q_codes).view(torch.float8_e4m3fn).float().numpy() * t
    o1, l1 = run(q_codes, kv_codes, [n], q_dtype=FP8, kv_dtype=FP8, q_scale=t, kv_scale=s)
    o2, l2 = run(bf16_bits(qf), bf16_bits(kvf), [n])   # products of powers of 2: exact in bf16
    assert np.allclose(o1, o2, rtol=0, atol=1e-13) and np.allclose(l1, l2, rtol=0, atol=1e-13)


def test_mxfp4_single_token_is_decoded_row():
    rng = np.random.default_rng(13)
    codes = rng.integers(0, 16, (1, D)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sc = rng.integers(124, 131, (1, 18)).astype(np.uint8)
    lut = {int(r[0]): float(r[1]) for r in golden("e2m1_lut.txt")}
    row = np.array([lut[int(c)] * 2.0 ** (int(sc[0, d // 32]) - 127) for d, c in enumerate(codes[0])])
    qb, qf = rand_bf16(rng, (1, H, D))
    o, lse = run(qb, packed, [1], kv_dtype=MXFP4, e8m0=sc, e8m0_stride=18)
    assert np.array_equal(o[0], np.broadcast_to(row[:DV], (H, DV)))
    assert np.allclose(lse[0], qf[0] @ row / 24.0, rtol=1e-13, atol=1e-13)


def test_brute_force_small_mixed():
    """Secondary check: an independent numpy fp64 statement of the definition
    (dequantise, scores, stable softmax, weighted V) on tiny paged inputs."""
    rng = np.random.default_rng(14)
    lengths, ps = [3, 0, 9, 1], 2
    npages = [(n + ps - 1) // ps for n in lengths]
    pool_pages = sum(npages) + 2
    perm = rng.permutation(pool_pages)[: sum(npages)].astype(np.int32)
    kvb, kvf = rand_bf16(rng, (pool_pages * ps, D))
    qb, qf = rand_bf16(rng, (4, H, D))
    last = np.array([n - (p - 1) * ps if p else ps for n, p in zip(lengths, npages)], np.int32)
    o, lse = run(qb, kvb, lengths, page_size=ps, kv_indices=perm, last=last)
    start = 0
    for b, n in enumerate(lengths):
        pages = perm[start: start + npages[b]]
        start += npages[b]
        rows = [pages[t // ps] * ps + t % ps for t in range(n)]
        if n == 0:
            assert np.all(o[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        K = kvf[rows]
        S = qf[b] @ K.T / 24.0
        M = S.max(1, keepdims=True)
        W = np.exp(S - M)
        assert np.allclose(o[b], W @ K[:, :DV] / W.sum(1, keepdims=True), rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[b], (M + np.log(W.sum(1, keepdims=True)))[:, 0], rtol=1e-12, atol=1e-12)


# ------------------------------------------------- several query tokens

def _qlen_problem(seed=11, page_size=4, q_len=3, lengths=(0, 1, 2, 5, 40)):
    rng = np.random.default_rng(seed)
    lengths = list(lengths)
    bs = len(lengths)
    npages = [(n + page_size - 1) // page_size for n in lengths]
    total = sum(npages) + 2
    q_bits, _ = rand_bf16(rng, (bs * q_len, H, D))
    kv_bits, _ = rand_bf16(rng, (total * page_size, D))
    perm = rng.permutation(total).astype(np.int32)[: sum(npages)]
    indptr = np.zeros(bs + 1, np.int32)
    indptr[1:] = np.cumsum(npages)
    last = np.array([n - (p - 1) * page_size if p else page_size for n, p in zip(lengths, npages)],
                    np.int32)
    return dict(bs=bs, page_size=page_size, q_len=q_len, lengths=lengths, q=q_bits, kv=kv_bits,
                indptr=indptr, indices=perm, last=last)


def test_qlen_rows_are_single_token_decodes_of_causal_prefixes():
    # query token t of a request with n tokens is a one-token decode of the
    # request cut to its first n - q_len + 1 + t tokens (same pages)
    P = _qlen_problem()
    o, lse = oracle.mla_decode(bs=P["bs"], page_size=P["page_size"], q_dtype=BF16, kv_dtype=BF16,
                               q=P["q"], kv=P["kv"], kv_indptr=P["indptr"],
                               kv_indices=P["indices"], kv_last_page_len=P["last"], nthreads=4,
                               q_len=P["q_len"])
    ps, ql = P["page_size"], P["q_len"]
    assert o.shape == (P["bs"] * ql, H, DV)
    for b, n in enumerate(P["lengths"]):
        for t in range(ql):
            vis = max(0, n - ql + 1 + t)
            npg = (vis + ps - 1) // ps
            p0 = int(P["indptr"][b])
            ip = np.array([p0, p0 + npg], np.int32)
            last = np.array([vis - (npg - 1) * ps if npg else ps], np.int32)
            o1, l1 = oracle.mla_decode(bs=1, page_size=ps, q_dtype=BF16, kv_dtype=BF16,
                                       q=P["q"][b * ql + t], kv=P["kv"], kv_indptr=ip,
                                       kv_indices=P["indices"][: p0 + npg] if npg else P["indices"],
                                       kv_last_page_len=last, nthreads=1)
            r = b * ql + t
            np.testing.assert_array_equal(o[r], o1[0])
            np.testing.assert_array_equal(lse[r], l1[0])


def test_qlen_token_without_visible_kv_is_empty_and_last_sees_all():
    P = _qlen_problem(lengths=(1, 2, 7), q_len=4)
    o, lse = oracle.mla_decode(bs=P["bs"], page_size=P["page_size"], q_dtype=BF16, kv_dtype=BF16,
                               q=P["q"], kv=P["kv"], kv_indptr=P["indptr"],
                               kv_indices=P["indices"], kv_last_page_len=P["last"], nthreads=4,
                               q_len=4)
    for b, n in enumerate(P["lengths"]):
        for t in range(4):
            r = b * 4 + t
            if n - 4 + 1 + t <= 0:
                assert np.all(o[r] == 0) and np.all(np.isneginf(lse[r]))
            else:
                assert np.all(np.isfinite(lse[r]))
    # the last query token of each request attends to every token: with its q
    # row, that is the plain one-token decode of the whole request
    q_last = P["q"].reshape(P["bs"], 4, H, D)[:, 3]
    o1, l1 = oracle.mla_decode(bs=P["bs"], page_size=P["page_size"], q_dtype=BF16, kv_dtype=BF16,
                               q=q_last, kv=P["kv"], kv_indptr=P["indptr"],
                               kv_indices=P["indices"], kv_last_page_len=P["last"], nthreads=4)
    np.testing.assert_array_equal(o[3::4], o1)
    np.testing.assert_array_equal(lse[3::4], l1)


def test_qlen_split_merge_invariance():
    P = _qlen_problem(lengths=(3, 40, 17), q_len=2)
    kw = dict(bs=P["bs"], page_size=P["page_size"], q_dtype=BF16, kv_dtype=BF16, q=P["q"],
              kv=P["kv"], kv_indptr=P["indptr"], kv_indices=P["indices"],
              kv_last_page_len=P["last"], nthreads=4, q_len=2)
    o, lse = oracle.mla_decode(**kw)
    o3, l3 = oracle.mla_decode(num_splits=3, **kw)
    assert np.allclose(o3, o, atol=1e-13, rtol=0) and np.allclose(l3, lse, atol=1e-12, rtol=0)
