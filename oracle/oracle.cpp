// oracle.cpp — plain CPU reference of the block-quantized GEMV and the sparse
// MoE layer.  TEST INFRASTRUCTURE: only the tests, the smoke check and the
// benchmark's CPU-baseline leg load this library; the product path never does.
// It shares no code with the CUDA library (no common header, table or helper).
//
// Style: plain loops that follow the definitions one to one, everything in
// double, each result rounded to its output type once.  No blocking, no
// vector intrinsics, no reordering beyond a row/token split across threads.
//
// Formats (the pages name them; the byte layouts are the GGUF/llama.cpp
// reading, written out again in the decoders below):
//   [Titan Engine, §激进量化策略] Q4_K; [KTransformers, §支持的量化格式]
//   Q4_K_M, Q6_K, Q8_0; [NTransformer (Show HN), §量化支持] Q8_0, Q6_K.
// MoE structure: [Titan Engine, §MoE 专家流式加载] (a few of E experts per
// token); [KTransformers, §技术原理] (sparse MoE matrices).  Router = softmax
// top-k renormalised, lowest index first on ties; expert FFN = SwiGLU.

#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---- scalar conversions -------------------------------------------------

// IEEE binary16 -> double, exact (every half is a double).
double half_to_f64(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int exp = (h >> 10) & 31;
  const int man = h & 1023;
  double v;
  if (exp == 0) {
    v = std::ldexp((double)man, -24);                 // subnormal: man * 2^-24
  } else if (exp == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = std::ldexp((double)(1024 + man), exp - 25);   // (1 + man/1024) * 2^(exp-15)
  }
  return sign ? -v : v;
}

// bfloat16 -> double, exact: the upper 16 bits of an fp32.
double bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

double act_elem(int dtype, const void* x, int64_t i) {
  switch (dtype) {
    case OR_F32: return (double)((const float*)x)[i];
    case OR_F16: return half_to_f64(((const uint16_t*)x)[i]);
    default: return bf16_to_f64(((const uint16_t*)x)[i]);
  }
}

// ---- block decoders ------------------------------------------------------
// Each writes the QK weights of one block as doubles.  Every product below is
// exact in double; the value is then the exact closed form.

// Q4_K: d, dmin fp16; 12 bytes of eight 6-bit (sc, m) pairs; 128 bytes of
// 4-bit quants in four 32-byte groups (low nibbles: sub-block 2c, high
// nibbles: sub-block 2c+1).  w = d*sc_j*q - dmin*m_j.
void q4k_scale_min(int j, const uint8_t* s, int* sc, int* m) {
  if (j < 4) {
    *sc = s[j] & 63;
    *m = s[j + 4] & 63;
  } else {
    *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
    *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
}

void decode_q4k(const uint8_t* b, double* w) {
  const double d = half_to_f64(rd16(b));
  const double dmin = half_to_f64(rd16(b + 2));
  const uint8_t* s = b + 4;
  const uint8_t* qs = b + 16;
  for (int c = 0; c < 4; ++c) {
    int sc_lo, m_lo, sc_hi, m_hi;
    q4k_scale_min(2 * c, s, &sc_lo, &m_lo);
    q4k_scale_min(2 * c + 1, s, &sc_hi, &m_hi);
    for (int l = 0; l < 32; ++l) {
      const int q_lo = qs[32 * c + l] & 15;
      const int q_hi = qs[32 * c + l] >> 4;
      w[64 * c + l] = d * sc_lo * q_lo - dmin * m_lo;
      w[64 * c + 32 + l] = d * sc_hi * q_hi - dmin * m_hi;
    }
  }
}

// Q6_K: ql[128], qh[64], int8 scales[16], fp16 d.  Two halves of 128.
// w = d * scales[i/16] * (q - 32), q = 4 low bits (ql) | 2 high bits (qh).
void decode_q6k(const uint8_t* b, double* w) {
  const uint8_t* ql = b;
  const uint8_t* qh = b + 128;
  const int8_t* sc = (const int8_t*)(b + 192);
  const double d = half_to_f64(rd16(b + 208));
  for (int h = 0; h < 2; ++h) {
    const uint8_t* L = ql + 64 * h;
    const uint8_t* Hh = qh + 32 * h;
    for (int l = 0; l < 32; ++l) {
      const int q1 = (L[l] & 15) | (((Hh[l] >> 0) & 3) << 4);
      const int q2 = (L[l + 32] & 15) | (((Hh[l] >> 2) & 3) << 4);
      const int q3 = (L[l] >> 4) | (((Hh[l] >> 4) & 3) << 4);
      const int q4 = (L[l + 32] >> 4) | (((Hh[l] >> 6) & 3) << 4);
      const int i1 = 128 * h + l, i2 = i1 + 32, i3 = i1 + 64, i4 = i1 + 96;
      w[i1] = d * sc[i1 / 16] * (q1 - 32);
      w[i2] = d * sc[i2 / 16] * (q2 - 32);
      w[i3] = d * sc[i3 / 16] * (q3 - 32);
      w[i4] = d * sc[i4 / 16] * (q4 - 32);
    }
  }
}

// Q8_0: fp16 d, int8 qs[32]; w = d*q.
void decode_q80(const uint8_t* b, double* w) {
  const double d = half_to_f64(rd16(b));
  const int8_t* q = (const int8_t*)(b + 2);
  for (int i = 0; i < 32; ++i) w[i] = d * q[i];
}

// Q4_0: fp16 d, 16 bytes of 4-bit quants; byte j holds weight j (low nibble)
// and weight j+16 (high nibble).  w = d*(q - 8).
void decode_q40(const uint8_t* b, double* w) {
  const double d = half_to_f64(rd16(b));
  const uint8_t* qs = b + 2;
  for (int j = 0; j < 16; ++j) {
    w[j] = d * ((qs[j] & 15) - 8);
    w[j + 16] = d * ((qs[j] >> 4) - 8);
  }
}

// Q5_K: d, dmin fp16; 12 bytes of eight 6-bit (sc, m) pairs packed as in
// Q4_K; 32 bytes qh of fifth bits; 128 bytes of low 4-bit quants in four
// 32-byte groups.  Group c: weight 64c+l takes the low nibble of qs[32c+l] and
// bit 2c of qh[l]; weight 64c+32+l the high nibble and bit 2c+1.
// q in [0, 31]; w = d*sc_j*q - dmin*m_j.
void decode_q5k(const uint8_t* b, double* w) {
  const double d = half_to_f64(rd16(b));
  const double dmin = half_to_f64(rd16(b + 2));
  const uint8_t* s = b + 4;
  const uint8_t* qh = b + 16;
  const uint8_t* qs = b + 48;
  for (int c = 0; c < 4; ++c) {
    int sc_lo, m_lo, sc_hi, m_hi;
    q4k_scale_min(2 * c, s, &sc_lo, &m_lo);
    q4k_scale_min(2 * c + 1, s, &sc_hi, &m_hi);
    for (int l = 0; l < 32; ++l) {
      const int q_lo = (qs[32 * c + l] & 15) | (((qh[l] >> (2 * c)) & 1) << 4);
      const int q_hi = (qs[32 * c + l] >> 4) | (((qh[l] >> (2 * c + 1)) & 1) << 4);
      w[64 * c + l] = d * sc_lo * q_lo - dmin * m_lo;
      w[64 * c + 32 + l] = d * sc_hi * q_hi - dmin * m_hi;
    }
  }
}

// Q2_K: 16 bytes of (scale | min << 4) for the sixteen 16-weight sub-blocks,
// 64 bytes of 2-bit quants, fp16 d, fp16 dmin (84 bytes).  Weight
// 128h + 32r + l (h = 0..1, r = 0..3, l = 0..31) takes bits 2r..2r+1 of
// qs[32h + l]; sub-block j = weight / 16.  w = d*(sc_j & 15)*q - dmin*(sc_j >> 4).
void decode_q2k(const uint8_t* b, double* w) {
  const uint8_t* sc = b;
  const uint8_t* qs = b + 16;
  const double d = half_to_f64(rd16(b + 80));
  const double dmin = half_to_f64(rd16(b + 82));
  for (int h = 0; h < 2; ++h)
    for (int r = 0; r < 4; ++r)
      for (int l = 0; l < 32; ++l) {
        const int i = 128 * h + 32 * r + l;
        const int q = (qs[32 * h + l] >> (2 * r)) & 3;
        const int j = i / 16;
        w[i] = d * (sc[j] & 15) * q - dmin * (sc[j] >> 4);
      }
}

// Q3_K: hmask[32] (high bits), 64 bytes of 2-bit low quants, 12 bytes of
// sixteen 6-bit scales, fp16 d (110 bytes).  Weight 128h + 32r + l: low bits
// 2r..2r+1 of qs[32h + l], high bit = bit 4h + r of hmask[l];
// q = low - (high ? 0 : 4), in [-4, 3].  Scale j: low 4 bits = nibble j / 8 of
// scales[j % 8], high 2 bits = bits 2(j / 4)..2(j / 4)+1 of scales[8 + j % 4];
// w = d*(s_j - 32)*q, sub-block j = weight / 16.
void decode_q3k(const uint8_t* b, double* w) {
  const uint8_t* hm = b;
  const uint8_t* qs = b + 32;
  const uint8_t* s = b + 96;
  const double d = half_to_f64(rd16(b + 108));
  int sc[16];
  for (int j = 0; j < 16; ++j)
    sc[j] = (((s[j % 8] >> (4 * (j / 8))) & 15) | (((s[8 + j % 4] >> (2 * (j / 4))) & 3) << 4)) - 32;
  for (int h = 0; h < 2; ++h)
    for (int r = 0; r < 4; ++r)
      for (int l = 0; l < 32; ++l) {
        const int i = 128 * h + 32 * r + l;
        const int low = (qs[32 * h + l] >> (2 * r)) & 3;
        const int high = (hm[l] >> (4 * h + r)) & 1;
        w[i] = d * sc[i / 16] * (low - (high ? 0 : 4));
      }
}

// E2M1 (FP4): sign, 2-bit exponent (bias 1), 1-bit mantissa; exponent 0 is
// subnormal (0 or 0.5).  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
double e2m1_to_f64(int c) {
  const int e = (c >> 1) & 3, m = c & 1;
  const double mag = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return (c & 8) ? -mag : mag;
}

// E4M3 (FP8): sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0 is
// subnormal (m/8 * 2^-6); S.1111.111 is NaN, there is no infinity.
double e4m3_to_f64(int b) {
  const int e = (b >> 3) & 15, m = b & 7;
  double mag;
  if (e == 15 && m == 7) mag = NAN;
  else if (e == 0) mag = std::ldexp((double)m, -9);
  else mag = std::ldexp(1.0 + m / 8.0, e - 7);
  return (b & 128) ? -mag : mag;
}

// NVFP4 super-block (this library's layout: the pages name the format but
// print no layout): 256 weights in 144 bytes, bytes 0-15 the E4M3 scales of
// the sixteen 16-weight blocks, bytes 16-143 the E2M1 codes, two per byte,
// weight 2i in the low nibble of byte 16+i and 2i+1 in the high nibble.
// w = e2m1(code) * e4m3(scale[i/16]); a per-tensor scale is the caller's.
void decode_nvfp4(const uint8_t* b, double* w) {
  for (int i = 0; i < 256; ++i) {
    const int code = (b[16 + i / 2] >> (4 * (i & 1))) & 15;
    w[i] = e2m1_to_f64(code) * e4m3_to_f64(b[i / 16]);
  }
}

bool geometry(int fmt, int* qk, int* bytes) {
  switch (fmt) {
    case OR_Q4_K: *qk = 256; *bytes = 144; return true;
    case OR_Q6_K: *qk = 256; *bytes = 210; return true;
    case OR_Q8_0: *qk = 32; *bytes = 34; return true;
    case OR_Q4_0: *qk = 32; *bytes = 18; return true;
    case OR_Q5_K: *qk = 256; *bytes = 176; return true;
    case OR_NVFP4: *qk = 256; *bytes = 144; return true;
    case OR_Q2_K: *qk = 256; *bytes = 84; return true;
    case OR_Q3_K: *qk = 256; *bytes = 110; return true;
    default: return false;
  }
}

void decode_block(int fmt, const uint8_t* b, double* w) {
  if (fmt == OR_Q4_K) decode_q4k(b, w);
  else if (fmt == OR_Q6_K) decode_q6k(b, w);
  else if (fmt == OR_Q8_0) decode_q80(b, w);
  else if (fmt == OR_Q4_0) decode_q40(b, w);
  else if (fmt == OR_Q5_K) decode_q5k(b, w);
  else if (fmt == OR_Q2_K) decode_q2k(b, w);
  else if (fmt == OR_Q3_K) decode_q3k(b, w);
  else decode_nvfp4(b, w);
}

// Split [0, n) into nthreads contiguous ranges and run fn(lo, hi) on each.
template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
  if (nthreads <= 1 || n <= 1) {
    fn((int64_t)0, n);
    return;
  }
  const int nt = (int)std::min<int64_t>(nthreads, n);
  std::vector<std::thread> th;
  for (int i = 0; i < nt; ++i) {
    const int64_t lo = n * i / nt, hi = n * (i + 1) / nt;
    th.emplace_back([=] { fn(lo, hi); });
  }
  for (auto& t : th) t.join();
}

// acc[b] = sum_k W[row][k] * xs[b][k] for one quantized row, in double.
void row_dot(int fmt, const uint8_t* row, int64_t K, const double* xs,
             int batch, double* acc) {
  int qk, bytes;
  geometry(fmt, &qk, &bytes);
  std::vector<double> w(qk);
  for (int b = 0; b < batch; ++b) acc[b] = 0.0;
  for (int64_t blk = 0; blk < K / qk; ++blk) {
    decode_block(fmt, row + blk * bytes, w.data());
    for (int b = 0; b < batch; ++b) {
      const double* xb = xs + (int64_t)b * K + blk * qk;
      double s = 0.0;
      for (int i = 0; i < qk; ++i) s += w[i] * xb[i];
      acc[b] += s;
    }
  }
}

// Matrix-vector product with a quantized [rows][cols] matrix, double in/out.
void qmatvec(int fmt, const uint8_t* W, int rows, int cols, const double* v,
             double* out) {
  int qk, bytes;
  geometry(fmt, &qk, &bytes);
  const int64_t row_bytes = (int64_t)(cols / qk) * bytes;
  for (int r = 0; r < rows; ++r) row_dot(fmt, W + r * row_bytes, cols, v, 1, &out[r]);
}

}  // namespace

extern "C" {

int or_geometry(int fmt, int* qk, int* bytes) {
  if (!qk || !bytes) return -1;
  return geometry(fmt, qk, bytes) ? 0 : -1;
}

int or_dequant(int fmt, const uint8_t* blocks, int64_t n, float* out) {
  int qk, bytes;
  if (!blocks || !out || !geometry(fmt, &qk, &bytes) || n <= 0 || n % qk) return -1;
  std::vector<double> w(qk);
  for (int64_t blk = 0; blk < n / qk; ++blk) {
    decode_block(fmt, blocks + blk * bytes, w.data());
    // One rounding: the double value is the exact closed form (all products
    // are exact; for Q4_K the difference is rounded to fp32 here only).
    for (int i = 0; i < qk; ++i) out[blk * qk + i] = (float)w[i];
  }
  return 0;
}

int or_act_to_f64(int dtype, const void* x, int64_t n, double* out) {
  if (!x || !out || n < 0 || dtype < OR_F32 || dtype > OR_BF16) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = act_elem(dtype, x, i);
  return 0;
}

int or_qgemv(int fmt, const uint8_t* W, int64_t N, int64_t K, const void* x,
             int xdt, int batch, const int64_t* rows, int64_t nrows, float* y,
             int nthreads) {
  int qk, bytes;
  if (!W || !x || !y || !geometry(fmt, &qk, &bytes) || N <= 0 || K <= 0 ||
      K % qk || batch < 1 || xdt < OR_F32 || xdt > OR_BF16)
    return -1;
  const int64_t nr = rows ? nrows : N;
  if (nr <= 0) return -1;
  if (rows)
    for (int64_t i = 0; i < nr; ++i)
      if (rows[i] < 0 || rows[i] >= N) return -1;
  std::vector<double> xs((size_t)batch * K);
  for (int64_t i = 0; i < (int64_t)batch * K; ++i) xs[i] = act_elem(xdt, x, i);
  const int64_t row_bytes = (K / qk) * bytes;
  parallel_for(nr, nthreads, [&](int64_t lo, int64_t hi) {
    std::vector<double> acc(batch);
    for (int64_t i = lo; i < hi; ++i) {
      const int64_t r = rows ? rows[i] : i;
      row_dot(fmt, W + r * row_bytes, K, xs.data(), batch, acc.data());
      for (int b = 0; b < batch; ++b) y[(int64_t)b * nr + i] = (float)acc[b];
    }
  });
  return 0;
}

int or_router_logits(const float* Wr, int E, int H, const void* x, int xdt,
                     int T, double* logits, int nthreads) {
  if (!Wr || !x || !logits || E <= 0 || H <= 0 || T <= 0) return -1;
  parallel_for(T, nthreads, [&](int64_t lo, int64_t hi) {
    for (int64_t t = lo; t < hi; ++t)
      for (int e = 0; e < E; ++e) {
        double s = 0.0;
        for (int h = 0; h < H; ++h)
          s += (double)Wr[(int64_t)e * H + h] * act_elem(xdt, x, t * H + h);
        logits[t * E + e] = s;
      }
  });
  return 0;
}

int or_topk(const double* logits, int T, int E, int k, int32_t* idx,
            double* gate) {
  if (!logits || !idx || T <= 0 || E <= 0 || k < 1 || k > E) return -1;
  std::vector<int> order(E);
  for (int t = 0; t < T; ++t) {
    const double* l = logits + (int64_t)t * E;
    for (int e = 0; e < E; ++e) order[e] = e;
    // Full stable sort by descending logit: equal logits keep index order,
    // so the lowest index comes first on ties.
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return l[a] > l[b]; });
    for (int i = 0; i < k; ++i) idx[(int64_t)t * k + i] = order[i];
    if (gate) {
      // softmax over all E renormalised over the selection
      //   = exp(l_i - l_max) / sum_{j in sel} exp(l_j - l_max)
      const double lmax = l[order[0]];
      double z = 0.0;
      for (int i = 0; i < k; ++i) z += std::exp(l[order[i]] - lmax);
      for (int i = 0; i < k; ++i)
        gate[(int64_t)t * k + i] = std::exp(l[order[i]] - lmax) / z;
    }
  }
  return 0;
}

int or_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
               int32_t* offsets, int32_t* sorted) {
  if (!idx || !counts || !offsets || !sorted || T <= 0 || k <= 0 || E <= 0) return -1;
  const int64_t P = (int64_t)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t p = 0; p < P; ++p) {
    if (idx[p] < 0 || idx[p] >= E) return -1;
    counts[idx[p]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> fill(offsets, offsets + E);
  // visiting pairs in increasing p keeps the order stable within an expert
  for (int64_t p = 0; p < P; ++p) sorted[fill[idx[p]]++] = (int32_t)p;
  return 0;
}

double or_silu(double g) { return g / (1.0 + std::exp(-g)); }

int or_expert_ffn(int fmt, const uint8_t* Wg, const uint8_t* Wu,
                  const uint8_t* Wd, int H, int F, const double* v,
                  double* out) {
  int qk, bytes;
  if (!Wg || !Wu || !Wd || !v || !out || !geometry(fmt, &qk, &bytes) ||
      H <= 0 || F <= 0 || H % qk || F % qk)
    return -1;
  std::vector<double> g(F), u(F), h(F);
  qmatvec(fmt, Wg, F, H, v, g.data());
  qmatvec(fmt, Wu, F, H, v, u.data());
  for (int j = 0; j < F; ++j) h[j] = or_silu(g[j]) * u[j];
  qmatvec(fmt, Wd, H, F, h.data(), out);
  return 0;
}

int or_moe_forward(int fmt, int E, int k, int H, int F, int n_shared,
                   const float* Wr, const uint8_t* w_gate,
                   const uint8_t* w_up, const uint8_t* w_down,
                   const uint8_t* sh_gate, const uint8_t* sh_up,
                   const uint8_t* sh_down, const void* x, int xdt, int T,
                   const int32_t* tokens, int ntokens, float* y, int32_t* idx,
                   double* gate, double* logits, int nthreads) {
  int qk, bytes;
  if (!Wr || !w_gate || !w_up || !w_down || !x || !geometry(fmt, &qk, &bytes) ||
      E <= 0 || k < 1 || k > E || H <= 0 || F <= 0 || H % qk || F % qk ||
      T <= 0 || n_shared < 0 || (n_shared > 0 && (!sh_gate || !sh_up || !sh_down)))
    return -1;
  const int nt = tokens ? ntokens : T;
  if (nt > 0 && !y) return -1;
  if (tokens)
    for (int i = 0; i < nt; ++i)
      if (tokens[i] < 0 || tokens[i] >= T) return -1;

  std::vector<double> L((size_t)T * E);
  or_router_logits(Wr, E, H, x, xdt, T, L.data(), nthreads);
  std::vector<int32_t> I((size_t)T * k);
  std::vector<double> G((size_t)T * k);
  or_topk(L.data(), T, E, k, I.data(), G.data());
  if (logits) std::copy(L.begin(), L.end(), logits);
  if (idx) std::copy(I.begin(), I.end(), idx);
  if (gate) std::copy(G.begin(), G.end(), gate);

  // bytes of one stacked expert matrix: gate/up are [F][H], down is [H][F]
  const int64_t gu_bytes = (int64_t)F * (H / qk) * bytes;
  const int64_t dn_bytes = (int64_t)H * (F / qk) * bytes;

  parallel_for(nt, nthreads, [&](int64_t lo, int64_t hi) {
    std::vector<double> v(H), o(H), acc(H);
    for (int64_t i = lo; i < hi; ++i) {
      const int t = tokens ? tokens[i] : (int)i;
      for (int h = 0; h < H; ++h) v[h] = act_elem(xdt, x, (int64_t)t * H + h);
      for (int h = 0; h < H; ++h) acc[h] = 0.0;
      for (int s = 0; s < k; ++s) {
        const int e = I[(int64_t)t * k + s];
        const double g = G[(int64_t)t * k + s];
        or_expert_ffn(fmt, w_gate + e * gu_bytes, w_up + e * gu_bytes,
                      w_down + e * dn_bytes, H, F, v.data(), o.data());
        for (int h = 0; h < H; ++h) acc[h] += g * o[h];
      }
      for (int s = 0; s < n_shared; ++s) {
        or_expert_ffn(fmt, sh_gate + s * gu_bytes, sh_up + s * gu_bytes,
                      sh_down + s * dn_bytes, H, F, v.data(), o.data());
        for (int h = 0; h < H; ++h) acc[h] += o[h];
      }
      for (int h = 0; h < H; ++h) y[i * H + h] = (float)acc[h];
    }
  });
  return 0;
}

}  // extern "C"
