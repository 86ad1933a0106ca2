// mla_oracle.cpp -- plain fp64 CPU definition of single-token MLA decode.
//
// TEST INFRASTRUCTURE ONLY.  This file is the oracle the CUDA path is checked
// against.  Only the test suite, the smoke check and the benchmark's CPU
// baseline may load it; the library under test never calls it and shares no
// code, header, table or helper with it.
//
// What it computes follows the kernelindex.com pages of the amd-mixed-mla
// leaderboard submissions:
//   * submission 695854, "chunked torch attention fallback": dequantise the
//     KV (bf16 / fp8 * kv_scale / MXFP4), softmax((q * sm_scale) . kv^T) over
//     all 576 dims, multiply by the first 512 dims of kv;
//   * submission 600081 (old version), "BMM bf16 for tiny batches": the same
//     bmm -> softmax -> bmm statement;
//   * submission 668813 (v0092a), header constants: 16 query heads, one KV
//     head, 512 latent + 64 rope dims, V = first 512 dims,
//     SM_SCALE = 1/sqrt(576);
//   * submission 668813, e2m1 lookup table and e8m0 decode 2^(e-127) of the
//     MXFP4 stage-1 kernel; scale byte j covers elements 32j..32j+31 and
//     packed byte i holds element 2i in its low nibble (same kernel, and the
//     even/odd de-interleave of its log2-domain stage-2 kernel);
//   * submission 668813, "log2-domain stage-2": the split/merge algebra
//     (only used here to test that splitting does not change the result).
//
// Readings taken where the pages are silent:
//   fp8 is OCP e4m3fn (bias 7, max 448, 0x7F/0xFF are NaN, subnormals);
//   e8m0 0xFF decodes to NaN; an empty request gives o = 0, lse = -inf;
//   lse is the natural log-sum-exp of the scaled scores.
//
// Several query tokens per request (q_len > 1): the pages run one query
// token per request (max_seqlen_qo = 1 in the metadata calls of submission
// 668813, whose causal flag is set) and name four query tokens only in the
// route selection of submission 695854.  The reading taken: the q_len query
// tokens are the last q_len positions of the sequence, already in the KV
// cache, and attend causally, so that query token i of a request with n
// tokens sees tokens [0, n - q_len + 1 + i); a query token that sees no
// token gives o = 0, lse = -inf.  q and the outputs are laid out
// [request][query token][head].
//
// Everything is fp64.  Inputs are decoded exactly (every bf16 / e4m3 / e2m1 x
// e8m0 value is exactly representable in a double).  No blocking, no fusion:
// scores, max, exponentials, sum and the weighted sum of V rows are computed
// one after the other as the definition states.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <atomic>

namespace {

constexpr int kHeads = 16;      // query heads (one latent KV head)
constexpr int kQkDim = 576;     // 512 latent + 64 rope
constexpr int kVDim = 512;      // V = first 512 dims of the latent row
constexpr int kMxBlock = 32;    // MXFP4: one e8m0 scale per 32 elements

enum { DT_BF16 = 0, DT_FP8_E4M3 = 1, DT_MXFP4 = 2 };

const double kNaN = std::numeric_limits<double>::quiet_NaN();
const double kNegInf = -std::numeric_limits<double>::infinity();

// bf16: the upper 16 bits of an IEEE binary32.
double dec_bf16(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// OCP e4m3fn: s eeee mmm, bias 7, no infinities, S.1111.111 is NaN.
double dec_e4m3(uint8_t c) {
  const int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
  double mag;
  if (e == 0xF && m == 7) return kNaN;
  if (e == 0)
    mag = std::ldexp(static_cast<double>(m), -9);       // m/8 * 2^(1-7)
  else
    mag = std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// e2m1 (4-bit): s ee m, bias 1, no inf/NaN.
double dec_e2m1(uint8_t nib) {
  const int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

// e8m0: 2^(e-127); 0xFF is NaN.
double dec_e8m0(uint8_t e) {
  if (e == 0xFF) return kNaN;
  return std::ldexp(1.0, static_cast<int>(e) - 127);
}

struct Problem {
  int bs, page_size, q_dtype, kv_dtype;
  const void* q;            // [bs, 16, 576] bf16 bits or e4m3 bytes
  double q_scale;           // used when q is e4m3
  const void* kv;           // rows of 576 bf16 / 576 e4m3 / 288 packed bytes
  double kv_scale;          // used when kv is e4m3
  const uint8_t* e8m0;      // MXFP4 scales, one row per KV row
  int64_t e8m0_stride;      // bytes between scale rows (>= 18)
  const int32_t* kv_indptr; // [bs+1], in pages
  const int32_t* kv_indices;// page ids, or null for the identity table
  const int32_t* last_len;  // [bs] tokens used in the last page, or null
};

// Element d of head h of q row `qr` (row = request * q_len + query token).
double q_value(const Problem& P, int64_t qr, int h, int d) {
  const int64_t i = (qr * kHeads + h) * kQkDim + d;
  if (P.q_dtype == DT_BF16) return dec_bf16(static_cast<const uint16_t*>(P.q)[i]);
  return dec_e4m3(static_cast<const uint8_t*>(P.q)[i]) * P.q_scale;
}

// Dequantised element d of KV row `row`.
double kv_value(const Problem& P, int64_t row, int d) {
  switch (P.kv_dtype) {
    case DT_BF16:
      return dec_bf16(static_cast<const uint16_t*>(P.kv)[row * kQkDim + d]);
    case DT_FP8_E4M3:
      return dec_e4m3(static_cast<const uint8_t*>(P.kv)[row * kQkDim + d]) * P.kv_scale;
    default: {
      const uint8_t byte = static_cast<const uint8_t*>(P.kv)[row * (kQkDim / 2) + d / 2];
      const uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      const uint8_t sc = P.e8m0[row * P.e8m0_stride + d / kMxBlock];
      return dec_e2m1(nib) * dec_e8m0(sc);
    }
  }
}

// KV row ids of request b's tokens, in token order, through the page table.
std::vector<int64_t> token_rows(const Problem& P, int b) {
  std::vector<int64_t> rows;
  const int32_t p0 = P.kv_indptr[b], p1 = P.kv_indptr[b + 1];
  const int npages = p1 - p0;
  if (npages <= 0) return rows;
  int64_t ntok = static_cast<int64_t>(npages) * P.page_size;
  if (P.last_len) ntok -= P.page_size - P.last_len[b];
  for (int64_t t = 0; t < ntok; ++t) {
    const int64_t slot = p0 + t / P.page_size;
    const int64_t page = P.kv_indices ? P.kv_indices[slot] : slot;
    rows.push_back(page * P.page_size + t % P.page_size);
  }
  return rows;
}

// One (q row, head) over a token sub-range [t0, t1): the definition.
//   s_j = (1/sqrt(576)) * sum_{d<576} q[h,d] k_j[d]
//   M = max_j s_j ; w_j = exp(s_j - M) ; l = sum_j w_j
//   o = sum_j w_j v_j / l  (v_j = first 512 dims of k_j) ; lse = M + ln l
void attend(const Problem& P, int64_t qr, int h, const std::vector<int64_t>& rows,
            int64_t t0, int64_t t1, double* o, double* lse) {
  for (int d = 0; d < kVDim; ++d) o[d] = 0.0;
  if (t1 <= t0) { *lse = kNegInf; return; }
  const double sm_scale = 1.0 / std::sqrt(static_cast<double>(kQkDim));
  double q[kQkDim];
  for (int d = 0; d < kQkDim; ++d) q[d] = q_value(P, qr, h, d);
  std::vector<double> s(t1 - t0);
  for (int64_t j = t0; j < t1; ++j) {
    double acc = 0.0;
    for (int d = 0; d < kQkDim; ++d) acc += q[d] * kv_value(P, rows[j], d);
    s[j - t0] = sm_scale * acc;
  }
  double M = kNegInf;
  for (double v : s) M = std::fmax(M, v);
  double l = 0.0;
  for (int64_t j = t0; j < t1; ++j) {
    const double w = std::exp(s[j - t0] - M);
    l += w;
    for (int d = 0; d < kVDim; ++d) o[d] += w * kv_value(P, rows[j], d);
  }
  for (int d = 0; d < kVDim; ++d) o[d] /= l;
  *lse = M + std::log(l);
}

// Split mode: cut the request into S contiguous ranges of ceil(n/S) tokens
// (the split rule of the MXFP4 stage-1 kernel of submission 668813), attend
// each, then merge with the log-sum-exp weights of its stage-2 kernel
// (written here in natural log):  L = max_s lse_s,
//   o = sum_s exp(lse_s - L) o_s / sum_s exp(lse_s - L),  lse = L + ln(sum).
void attend_split(const Problem& P, int64_t qr, int h, const std::vector<int64_t>& rows,
                  int64_t n, int S, double* o, double* lse) {
  const int64_t per = (n + S - 1) / S;
  std::vector<double> os(static_cast<size_t>(S) * kVDim), ls(S);
  for (int s = 0; s < S; ++s) {
    const int64_t a = std::min<int64_t>(per * s, n), e = std::min<int64_t>(per * s + per, n);
    attend(P, qr, h, rows, a, e, &os[static_cast<size_t>(s) * kVDim], &ls[s]);
  }
  double L = kNegInf;
  for (int s = 0; s < S; ++s) L = std::fmax(L, ls[s]);
  for (int d = 0; d < kVDim; ++d) o[d] = 0.0;
  if (L == kNegInf) { *lse = kNegInf; return; }
  double wsum = 0.0;
  for (int s = 0; s < S; ++s) {
    const double w = std::exp(ls[s] - L);   // exp(-inf) = 0 for empty splits
    wsum += w;
    for (int d = 0; d < kVDim; ++d) o[d] += w * os[static_cast<size_t>(s) * kVDim + d];
  }
  for (int d = 0; d < kVDim; ++d) o[d] /= wsum;
  *lse = L + std::log(wsum);
}

}  // namespace

extern "C" {

// Format decoders, exposed so the tests can pin them to the format tables.
void oracle_decode_bf16(const uint16_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = dec_bf16(in[i]);
}
void oracle_decode_e4m3(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = dec_e4m3(in[i]);
}
void oracle_decode_e2m1(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = dec_e2m1(in[i] & 0xF);
}
void oracle_decode_e8m0(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = dec_e8m0(in[i]);
}

// Dequantise KV rows [row0, row0+nrows) into out[nrows, 576].
int oracle_dequant_kv(int kv_dtype, const void* kv, double kv_scale,
                      const uint8_t* e8m0, int64_t e8m0_stride,
                      int64_t row0, int64_t nrows, double* out) {
  if (kv_dtype < 0 || kv_dtype > 2) return 1;
  Problem P{};
  P.kv_dtype = kv_dtype; P.kv = kv; P.kv_scale = kv_scale;
  P.e8m0 = e8m0; P.e8m0_stride = e8m0_stride;
  for (int64_t r = 0; r < nrows; ++r)
    for (int d = 0; d < kQkDim; ++d) out[r * kQkDim + d] = kv_value(P, row0 + r, d);
  return 0;
}

// Full decode with q_len query tokens per request.  For each selected
// request (all of them when `select` is null) and each of its query tokens
// writes o[(i * q_len + t), 16, 512] and lse[(i * q_len + t), 16] in fp64.
// num_splits <= 1 computes the definition directly; num_splits > 1 uses the
// split/merge mode over each query token's visible tokens.
// Returns 0, or 1 on bad arguments.
int oracle_mla_decode_q(int bs, int q_len, int page_size, int q_dtype, int kv_dtype,
                        const void* q, double q_scale,
                        const void* kv, double kv_scale,
                        const uint8_t* e8m0, int64_t e8m0_stride,
                        const int32_t* kv_indptr, const int32_t* kv_indices,
                        const int32_t* last_page_len,
                        int num_splits, const int32_t* select, int nselect,
                        int nthreads, double* o, double* lse) {
  if (bs < 0 || q_len < 1 || page_size < 1 || q_dtype < 0 || q_dtype > 1 || kv_dtype < 0 ||
      kv_dtype > 2)
    return 1;
  if (kv_dtype == DT_MXFP4 && (e8m0 == nullptr || e8m0_stride < kQkDim / kMxBlock)) return 1;
  Problem P{bs, page_size, q_dtype, kv_dtype, q, q_scale, kv, kv_scale,
            e8m0, e8m0_stride, kv_indptr, kv_indices, last_page_len};
  const int nreq = select ? nselect : bs;
  if (select)
    for (int i = 0; i < nselect; ++i)
      if (select[i] < 0 || select[i] >= bs) return 1;
  const int64_t units = static_cast<int64_t>(nreq) * q_len * kHeads;
  std::atomic<int64_t> next(0);
  auto worker = [&]() {
    for (;;) {
      const int64_t u = next.fetch_add(1);
      if (u >= units) break;
      const int64_t row = u / kHeads;                      // output row i * q_len + t
      const int i = static_cast<int>(row / q_len), t = static_cast<int>(row % q_len);
      const int h = static_cast<int>(u % kHeads);
      const int b = select ? select[i] : i;
      const std::vector<int64_t> rows = token_rows(P, b);
      const int64_t n = static_cast<int64_t>(rows.size());
      // query token t sees the first n - q_len + 1 + t tokens
      const int64_t vis = std::max<int64_t>(0, std::min<int64_t>(n, n - q_len + 1 + t));
      const int64_t qr = static_cast<int64_t>(b) * q_len + t;
      double* oo = o + u * kVDim;
      if (num_splits > 1)
        attend_split(P, qr, h, rows, vis, num_splits, oo, lse + u);
      else
        attend(P, qr, h, rows, 0, vis, oo, lse + u);
    }
  };
  if (nthreads < 1) nthreads = 1;
  std::vector<std::thread> pool;
  for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return 0;
}

// One query token per request: o[i, 16, 512], lse[i, 16].
int oracle_mla_decode(int bs, int page_size, int q_dtype, int kv_dtype,
                      const void* q, double q_scale,
                      const void* kv, double kv_scale,
                      const uint8_t* e8m0, int64_t e8m0_stride,
                      const int32_t* kv_indptr, const int32_t* kv_indices,
                      const int32_t* last_page_len,
                      int num_splits, const int32_t* select, int nselect,
                      int nthreads, double* o, double* lse) {
  return oracle_mla_decode_q(bs, 1, page_size, q_dtype, kv_dtype, q, q_scale, kv, kv_scale,
                             e8m0, e8m0_stride, kv_indptr, kv_indices, last_page_len,
                             num_splits, select, nselect, nthreads, o, lse);
}

}  // extern "C"
