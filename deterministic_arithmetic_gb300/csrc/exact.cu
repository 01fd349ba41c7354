// exact.cu -- the exact mode of the weight gradients (page "det-train"
// (bitwise-deterministic training arithmetic), section "Method": a Kulisch long
// accumulator per output, composed by adding digit arrays, rounded once).
//
//   dA[r][k] = rn32( sum_m du[m][r] * x[m][k] )      exact sum, rounded once
//   dB[n][r] = rn32( sum_m dv[m][n] * u[m][r] ),  dv = bf16(fp32(dy * alpha))
//
// Every finite BF16 value is m * 2^s with an integer m in [-255, 255] and s in
// [-133, 120], so every product is m1 m2 2^(s1 + s2), |m1 m2| < 2^16, at bit
// position pos = s1 + s2 + 266 in [0, 506] counted from 2^-266. Each output owns
// kDigits signed 64-bit digits in radix 2^32 (digit i weighs 2^(32 i - 266)) and
// three counters of +inf, -inf and NaN products (inf * 0 and NaN factors count
// as NaN). Integer addition is associative, so the digits of any partition of
// the rows add up to the digits of the whole; written out they are first
// normalised (digits 0 .. kDigits-2 in [0, 2^32), the top one signed), which makes
// the digit arrays themselves, not only their values, independent of the
// partition. The FP32 result is the digit sum rounded to nearest even, once:
// NaN if a NaN product or both infinities occurred, else the infinity, else the
// rounded sum (an exact zero sum is +0).
//
// exact_digits_kernel: persistent CTAs (two per SM) over work units, a unit being
// 64 rows of one 16 x 64 output tile (units numbered tile by tile); CTA c takes
// the units [c U / G, (c + 1) U / G) and handles each run of them that lies in
// one tile as a segment, numbered c + t (t the tile). The rows are decoded 64 at
// a time into (m, s) pairs in shared memory. Each thread owns two outputs and
// keeps, for each, a window accumulator in registers: a signed 64-bit sum of
// m1 m2 2^(pos - anc) over the products whose position lies in [anc, anc + 30]
// (one IMAD.WIDE per product; at most 2^16 rows per window keep it below
// 2^62, so a longer segment adds its window to the digits every 2^16 rows).
// Before each 64 rows the window is anchored (or moved up, after adding it to the
// digits) so that the largest product the rows can hold -- at the position of
// the sum of the column maxima of s -- lies 24 bits above the anchor; the
// products below the window (none for data of ordinary range), and the
// infinite and NaN ones,
// and the infinite and NaN ones, are added straight into the output's digit
// array of the segment in global memory (owned by the thread; zeroed at its
// first use). Each segment leaves one record per output: the window (acc, anc)
// and whether its digit array was used.
// exact_reduce_kernel adds, per output, the windows and digit arrays of the
// segments of its tile, and writes the normalised digits or rounds them.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

constexpr int kTP = 16, kTQ = 64;                      // output tile [p][q]
constexpr int kRows = 64;                              // rows decoded per step
constexpr int kThreads = 512;                          // two outputs (p, p + 1) per thread
// Exponent codes s of the factors that are not finite non-zero values, and the ranges of e = s1 + s2
// they give: finite * finite in [-266, 240]; finite * 0 in [-20133, -19880]; 0 * 0 = -40000;
// inf * finite in [867, 1120]; inf * 0 = -19000; inf * inf = 2000; NaN * finite in [3867, 4120];
// NaN * 0 = -16000; NaN * inf = 5000; NaN * NaN = 8000.
constexpr int kZero = -20000, kInf = 1000, kNaN = 4000;
constexpr int kWindow = 30;                            // highest position above the anchor
constexpr int kBelowTop = 24;                          // anchor = the largest possible product's position - this
constexpr int kNone = -100000;                         // column maximum of a column with no non-zero finite value
constexpr int kNoneMin = 100000;                       // its column minimum
constexpr int kUnset = -100000;                        // window offset before its anchor is set
constexpr int kFlushBlocks = (1 << 16) / kRows;         // window headroom: 2^16 products below 2^46 each
constexpr int kOut = kTP * kTQ;                        // outputs per tile

// BF16 -> (m, s), value = m * 2^s; zero: (0, kZero); inf: (+-1, kInf); NaN: (0, kNaN)
__device__ __forceinline__ int2 decode_bf16(uint32_t h) {
  const int e = int(h >> 7) & 0xFF, f = int(h) & 0x7F;
  const bool neg = (h & 0x8000u) != 0u;
  if (e == 0xFF) return f ? make_int2(0, kNaN) : make_int2(neg ? -1 : 1, kInf);
  const int mag = e ? (f | 0x80) : f;
  return make_int2(neg ? -mag : mag, mag ? (e ? e : 1) - 134 : kZero);
}

__device__ __forceinline__ bool special_product(int e) { return e > 600 || (e > -19500 && e < -1000); }

// 2^sh for sh in [0, 31), 0 for sh < 0 or sh >= 32 (PTX clamps the shift amount, read unsigned)
__device__ __forceinline__ int pow2_or_zero(int sh) {
  int r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(1), "r"(sh));
  return r;
}

// The window of one output: acc * 2^(anc - 266), anc = 266 - off (off = kUnset: no anchor yet),
// and whether the output's digit array for the segment has been used.
struct Win {
  long long acc;
  int off;
  int used;
};

// The digit array of one output for one segment: dig[slot * kOut] (global memory, owned by
// one thread), zeroed at its first use.
__device__ __forceinline__ void touch(long long* dig, int& used) {
  if (!used) {
    for (int s = 0; s < kExactSlots; ++s) dig[s * kOut] = 0;
    used = 1;
  }
}

// the window's value into the digit array (the window keeps its anchor, emptied)
__device__ __forceinline__ void spill_window(Win& w, long long* dig) {
  if (w.off == kUnset || w.acc == 0) return;
  touch(dig, w.used);
  const int anc = 266 - w.off, d = anc >> 5, sa = anc & 31;
  const unsigned long long lo = (unsigned long long)w.acc << sa;
  const long long hi = sa ? (w.acc >> (64 - sa)) : (w.acc >> 63);   // acc * 2^sa = hi * 2^64 + lo
  dig[d * kOut] += (long long)(lo & 0xFFFFFFFFull);
  dig[(d + 1) * kOut] += (long long)(lo >> 32);
  dig[(d + 2) * kOut] += hi;
  w.acc = 0;
}

// a product the window did not take: mm * 2^e (e = s1 + s2); returns the new window
__device__ __forceinline__ Win slow_product(Win w, long long* dig, int mm, int e) {
  if (special_product(e)) {   // an infinite or NaN factor
    touch(dig, w.used);
    const bool nan = e > 3000 || e < 0;   // a NaN factor, or inf * 0
    dig[(nan ? kDigits + 2 : (mm < 0 ? kDigits + 1 : kDigits)) * kOut] += 1;
    return w;
  }
  if (e < -1000) return w;                             // a zero factor
  const int pos = e + 266;                             // in [0, 506]; mm != 0
  if (w.off != kUnset && pos < 266 - w.off) {          // below the window: straight into the digits
    touch(dig, w.used);
    const long long v = (long long)mm << (pos & 31);   // |v| < 2^47
    const int d = pos >> 5;
    dig[d * kOut] += (long long)(uint32_t)v;           // low word, unsigned
    dig[(d + 1) * kOut] += v >> 32;                    // the rest, signed
    return w;
  }
  // above the window, or no window yet: not reached when the window is anchored under the
  // rows' largest possible product, but kept exact all the same -- a new window, this
  // product near its top
  spill_window(w, dig);
  const int anc = max(pos - kBelowTop, 0);
  w.off = 266 - anc;
  w.acc = (long long)mm << (pos - anc);
  return w;
}

__device__ __forceinline__ long long record_tag(const Win& w) {
  return (long long)(uint32_t)(w.off == kUnset ? -1 : 266 - w.off) | ((long long)w.used << 32);
}

// How the rows' products are checked: kFree -- every non-zero product lies in the window (known
// from the column extremes): no check; kBelow -- finite values, some products may lie below the
// window; kSpecial -- infinite or NaN values among the rows.
enum RowMode { kFree, kBelow, kSpecial };

// The products of rows [0, nr) of the decoded tile for this thread's two outputs (2 pg, q) and
// (2 pg + 1, q): each adds m1 m2 2^sh to the window when sh = e + off is in [0, 30] (and 0
// otherwise: below the window, or a zero, infinite or NaN factor, whose e lies far outside),
// and the ones the window does not take go to slow_product.
template <int MODE>
__device__ __forceinline__ void window_rows(const int4 (*lft)[kTP / 2], const int2 (*rgt)[kTQ], int nr, int q, int pg,
                                            Win& wa, Win& wb, long long* dig_a, long long* dig_b) {
  for (int r0 = 0; r0 < nr; r0 += 4) {
    int2 rv[4];
    int4 lv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      rv[j] = rgt[r0 + j][q];
      lv[j] = lft[r0 + j][pg];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int mm0 = lv[j].x * rv[j].x, mm1 = lv[j].z * rv[j].x;
      const int sh0 = lv[j].y + rv[j].y + wa.off, sh1 = lv[j].w + rv[j].y + wb.off;
      wa.acc += (long long)mm0 * pow2_or_zero(sh0);
      wb.acc += (long long)mm1 * pow2_or_zero(sh1);
      if (MODE != kFree) {
        const int e0 = lv[j].y + rv[j].y, e1 = lv[j].w + rv[j].y;
        const bool out0 = MODE == kBelow ? (sh0 < 0 && e0 > -1000)
                                         : (special_product(e0) || (e0 > -1000 && unsigned(sh0) > unsigned(kWindow)));
        const bool out1 = MODE == kBelow ? (sh1 < 0 && e1 > -1000)
                                         : (special_product(e1) || (e1 > -1000 && unsigned(sh1) > unsigned(kWindow)));
        if (out0 | out1) {
          if (out0) wa = slow_product(wa, dig_a, mm0, e0);
          if (out1) wb = slow_product(wb, dig_b, mm1, e1);
        }
      }
    }
  }
}

// CTA of unit u when U units are split among G CTAs as [c U / G, (c + 1) U / G)
__host__ __device__ __forceinline__ int cta_of_unit(int64_t u, int64_t U, int G) {
  return int(((u + 1) * G - 1) / U);
}

// DV: the right operand is dV = bf16(fp32(dy * alpha)), formed from dY.
// Tiles: t = tp * n_tq + tq (16 rows of P by 64 columns of Q); B row blocks of 64 per tile.
// rec[seg][o]: (window acc, anchor (-1: none) | digits-used << 32); spill[seg][slot][o],
// o = (p - p0) * 64 + (q - q0), seg = c + t.
template <bool DV>
__global__ void __launch_bounds__(kThreads, 2)
    exact_digits_kernel(const uint16_t* __restrict__ left, int ldl, const uint16_t* __restrict__ right, int ldr,
                        int M, int P, int Q, int n_tq, int B, int64_t U, float alpha, longlong2* __restrict__ rec,
                        long long* __restrict__ spill) {
  grid_dependency_wait();
  grid_dependents_launch();
  __shared__ int4 lft[kRows][kTP / 2];   // (m, s) of left columns 2i and 2i + 1
  __shared__ int2 rgt[kRows][kTQ];
  __shared__ int2 wl[kRows / 2][kTP], wr[kRows / 8][kTQ];   // column (max, min) of s per staging thread
  __shared__ int2 ext_l[kTP], ext_r[kTQ];                     // column (max, min) of s over the 64 rows
  const int tid = threadIdx.x, q = tid % kTQ, pg = tid / kTQ;   // outputs (2 pg, q) and (2 pg + 1, q)
  const int oa = 2 * pg * kTQ + q, ob = oa + kTQ;               // their indexes in the tile
  const int G = gridDim.x, c = blockIdx.x;
  int2* l2 = reinterpret_cast<int2*>(&lft[0][0]);
  const int64_t u_end = (int64_t(c) + 1) * U / G;
  for (int64_t u = int64_t(c) * U / G; u < u_end;) {
    const int tile = int(u / B);
    const int64_t seg_end = std::min<int64_t>(u_end, (int64_t(tile) + 1) * B);
    const int q0 = (tile % n_tq) * kTQ, p0 = (tile / n_tq) * kTP;
    const size_t seg = size_t(c) + tile;
    long long* dig_a = spill + seg * kExactSlots * kOut + oa;
    long long* dig_b = spill + seg * kExactSlots * kOut + ob;
    Win wa{0, kUnset, 0}, wb{0, kUnset, 0};
    int blocks = 0;
    for (; u < seg_end; ++u) {
      const int m0 = int(u - int64_t(tile) * B) * kRows, m_end = min(M, m0 + kRows);
      __syncthreads();   // previous rows consumed
      // decode the rows: left column tid % 16, rows 2 (tid / 16) and the next; right column
      // tid % 64, rows 8 (tid / 64) .. + 7; zeros past M, P and Q. special: an infinite or NaN
      // value among them; the column extremes of s over non-zero finite values.
      int special = 0;
      {
        const int p = tid % kTP, rp = tid / kTP;
        int mx = kNone, mn = kNoneMin;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int r = 2 * rp + k, m = m0 + r;
          const uint32_t h = (m < m_end && p0 + p < P) ? left[size_t(m) * ldl + p0 + p] : 0u;
          special |= (h & 0x7F80u) == 0x7F80u;
          const int2 d = decode_bf16(h);
          l2[r * kTP + p] = d;
          if (d.x != 0 && d.y < 600) mx = max(mx, d.y), mn = min(mn, d.y);
        }
        wl[rp][p] = make_int2(mx, mn);
      }
      {
        const int rg = tid / kTQ;
        const bool qin = q0 + q < Q;
        int mx = kNone, mn = kNoneMin;
#pragma unroll
        for (int k = 0; k < kRows / 8; ++k) {
          const int r = 8 * rg + k, m = m0 + r;
          uint32_t h = (m < m_end && qin) ? right[size_t(m) * ldr + q0 + q] : 0u;
          if (DV) h = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__uint_as_float(h << 16), alpha)));
          special |= (h & 0x7F80u) == 0x7F80u;
          const int2 d = decode_bf16(h);
          rgt[r][q] = d;
          if (d.x != 0 && d.y < 600) mx = max(mx, d.y), mn = min(mn, d.y);
        }
        wr[rg][q] = make_int2(mx, mn);
      }
      const bool any_special = __syncthreads_or(special);
      if (tid < kTP) {
        int2 x = make_int2(kNone, kNoneMin);
        for (int i = 0; i < kRows / 2; ++i) x = make_int2(max(x.x, wl[i][tid].x), min(x.y, wl[i][tid].y));
        ext_l[tid] = x;
      } else if (tid >= 2 * kTQ && tid < 3 * kTQ) {
        int2 x = make_int2(kNone, kNoneMin);
        for (int i = 0; i < kRows / 8; ++i)
          x = make_int2(max(x.x, wr[i][tid - 2 * kTQ].x), min(x.y, wr[i][tid - 2 * kTQ].y));
        ext_r[tid - 2 * kTQ] = x;
      }
      __syncthreads();
      // windows: anchored (or moved up, after adding them to the digits) so that the largest
      // product these rows can hold sits kBelowTop bits above the anchor; free: the smallest
      // non-zero one lies in the window too
      bool free = true;
      {
        const int2 er = ext_r[q], ea = ext_l[2 * pg], eb = ext_l[2 * pg + 1];
        if (er.x != kNone && ea.x != kNone) {
          const int top = ea.x + er.x + 266;
          if (wa.off == kUnset || top > 266 - wa.off + kWindow) {
            spill_window(wa, dig_a);
            wa.off = 266 - max(top - kBelowTop, 0);
          }
          free = free && ea.y + er.y + wa.off >= 0;
        }
        if (er.x != kNone && eb.x != kNone) {
          const int top = eb.x + er.x + 266;
          if (wb.off == kUnset || top > 266 - wb.off + kWindow) {
            spill_window(wb, dig_b);
            wb.off = 266 - max(top - kBelowTop, 0);
          }
          free = free && eb.y + er.y + wb.off >= 0;
        }
      }
      const int nr = m_end - m0;   // rows past nr hold zeros: adding them changes nothing
      if (any_special)
        window_rows<kSpecial>(lft, rgt, nr, q, pg, wa, wb, dig_a, dig_b);
      else if (__all_sync(0xFFFFFFFFu, free))
        window_rows<kFree>(lft, rgt, nr, q, pg, wa, wb, dig_a, dig_b);
      else
        window_rows<kBelow>(lft, rgt, nr, q, pg, wa, wb, dig_a, dig_b);
      if (++blocks == kFlushBlocks) {   // 2^16 rows in the window: empty it into the digits
        spill_window(wa, dig_a);
        spill_window(wb, dig_b);
        blocks = 0;
      }
    }
    rec[seg * kOut + oa] = make_longlong2(wa.acc, record_tag(wa));
    rec[seg * kOut + ob] = make_longlong2(wb.acc, record_tag(wb));
  }
}

// carry-normalise: digits 0 .. kDigits-2 into [0, 2^32), the top digit keeps the signed rest
__device__ __forceinline__ void normalise(long long (&c)[kExactSlots]) {
  long long carry = 0;
#pragma unroll
  for (int i = 0; i < kDigits - 1; ++i) {
    const long long t = c[i] + carry;
    const long long w = (long long)(uint32_t)t;
    carry = (t - w) >> 32;   // exact: t - w is a multiple of 2^32
    c[i] = w;
  }
  c[kDigits - 1] += carry;
}

// FP32 value of a normalised digit array (round to nearest even, once)
__device__ float round_digits(const long long (&c)[kExactSlots]) {
  const long long pinf = c[kDigits], ninf = c[kDigits + 1], nan = c[kDigits + 2];
  if (nan != 0 || (pinf != 0 && ninf != 0)) return __uint_as_float(0x7FC00000u);
  if (pinf != 0) return __uint_as_float(0x7F800000u);
  if (ninf != 0) return __uint_as_float(0xFF800000u);
  // 32-bit words of the two's complement value: w[0 .. kDigits-2] and the top digit (two words)
  constexpr int kW = kDigits + 1;
  uint32_t w[kW];
#pragma unroll
  for (int i = 0; i < kDigits - 1; ++i) w[i] = uint32_t(c[i]);
  w[kDigits - 1] = uint32_t(c[kDigits - 1]);
  w[kDigits] = uint32_t(c[kDigits - 1] >> 32);
  const bool neg = c[kDigits - 1] < 0;
  if (neg) {   // magnitude
    uint32_t k = 1;
#pragma unroll
    for (int i = 0; i < kW; ++i) {
      const uint64_t t = uint64_t(~w[i]) + k;
      w[i] = uint32_t(t);
      k = uint32_t(t >> 32);
    }
  }
  int h = -1;   // highest set bit, counted from 2^-266
#pragma unroll
  for (int i = kW - 1; i >= 0; --i)
    if (h < 0 && w[i] != 0u) h = 32 * i + 31 - __clz(w[i]);
  if (h < 0) return 0.0f;
  // unit of the result: 2^(h - 23), or 2^-149 (bit 117) below the normal range
  const int L = max(h - 23, 117);
  auto bits_at = [&](int b) -> uint64_t {   // the 64 bits from bit b on
    const int i = b >> 5, s = b & 31;
    uint64_t lo = 0, mid = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < kW; ++j) {
      lo = j == i ? w[j] : lo;
      mid = j == i + 1 ? w[j] : mid;
      hi = j == i + 2 ? w[j] : hi;
    }
    const uint64_t x = lo | (mid << 32);
    return s ? (x >> s) | (hi << (64 - s)) : x;
  };
  uint64_t q = bits_at(L) & ((uint64_t(1) << 25) - 1u);
  const bool half = (bits_at(L - 1) & 1u) != 0u;
  bool sticky = false;   // any of bits 0 .. L-2
#pragma unroll
  for (int i = 0; i < kW; ++i) {
    const int b0 = 32 * i, n = L - 1 - b0;   // bits of word i below bit L-1
    if (n > 0) sticky = sticky || (w[i] & (n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u))) != 0u;
  }
  if (half && (sticky || (q & 1u))) ++q;
  // q * 2^(L - 266) in FP32: q + ((L - 117) << 23) encodes it for subnormal, normal and
  // carried-out (q = 2^24) values alike; from the exponent field's top on it is infinite
  uint64_t bits = q + (uint64_t(L - 117) << 23);
  if (bits >= 0x7F800000u) bits = 0x7F800000u;
  return __uint_as_float(uint32_t(bits) | (neg ? 0x80000000u : 0u));
}

// out index of output (p, q): [p][q], or [q][p] with transpose
__device__ __forceinline__ size_t out_index(int p, int q, int P, int Q, int transpose) {
  return transpose ? size_t(q) * P + p : size_t(p) * Q + q;
}

// the windows and digit arrays of the segments of each output's tile added; written
// normalised to out_digits ([outputs][kExactSlots], outputs in out_index order) and/or
// rounded to out
__global__ void __launch_bounds__(256) exact_reduce_kernel(const longlong2* __restrict__ rec,
                                                           const long long* __restrict__ spill, int P, int Q,
                                                           int n_tq, int B, int64_t U, int G, int transpose,
                                                           long long* __restrict__ out_digits,
                                                           float* __restrict__ out) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i >= P * Q) return;
  const int p = i / Q, q = i % Q;
  const int tile = (p / kTP) * n_tq + q / kTQ, o = (p % kTP) * kTQ + q % kTQ;
  long long c[kExactSlots];
#pragma unroll
  for (int s = 0; s < kExactSlots; ++s) c[s] = 0;
  if (B > 0) {
    const int c0 = cta_of_unit(int64_t(tile) * B, U, G), c1 = cta_of_unit((int64_t(tile) + 1) * B - 1, U, G);
    for (int cta = c0; cta <= c1; ++cta) {
      const size_t seg = size_t(cta) + tile;
      const longlong2 r = rec[seg * kOut + o];
      const int anc = int(r.y & 0xFFFFFFFF);
      if (anc >= 0) {   // window acc * 2^(anc - 266): words d, d + 1 (unsigned) and d + 2 (signed)
        const int d = anc >> 5, sa = anc & 31;
        const unsigned long long lo = (unsigned long long)r.x << sa;
        const long long hi = sa ? (r.x >> (64 - sa)) : (r.x >> 63);
        const long long w0 = (long long)(lo & 0xFFFFFFFFull), w1 = (long long)(lo >> 32);
#pragma unroll
        for (int s = 0; s < kDigits; ++s) c[s] += s == d ? w0 : (s == d + 1 ? w1 : (s == d + 2 ? hi : 0));
      }
      if ((r.y >> 32) & 1) {
#pragma unroll
        for (int s = 0; s < kExactSlots; ++s) c[s] += spill[(seg * kExactSlots + s) * kOut + o];
      }
    }
  }
  normalise(c);
  const size_t oi = out_index(p, q, P, Q, transpose);
  if (out_digits) {
#pragma unroll
    for (int s = 0; s < kExactSlots; ++s) out_digits[oi * kExactSlots + s] = c[s];
  }
  if (out) out[oi] = round_digits(c);
}

// out_digits = normalised (a + b) and / or out = its FP32 value (b may be null: a alone)
// (no __restrict__: out_digits may be a or b, an in-place sum)
__global__ void __launch_bounds__(256) exact_combine_kernel(const long long* a, const long long* b, int64_t n,
                                                            long long* out_digits, float* out) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t i = int64_t(blockIdx.x) * 256 + threadIdx.x;
  if (i >= n) return;
  long long c[kExactSlots];
#pragma unroll
  for (int s = 0; s < kExactSlots; ++s) c[s] = a[i * kExactSlots + s] + (b ? b[i * kExactSlots + s] : 0);
  normalise(c);
  if (out_digits) {
#pragma unroll
    for (int s = 0; s < kExactSlots; ++s) out_digits[i * kExactSlots + s] = c[s];
  }
  if (out) out[i] = round_digits(c);
}

int64_t tiles_of(int64_t P, int64_t Q) { return ceil_div(Q, kTQ) * ceil_div(P, kTP); }

}  // namespace

// segments of the digit kernel: at most G + tiles - 1 (G <= min(kMaxExactGrid, units))
size_t exact_segments(int64_t M, int64_t P, int64_t Q) {
  const int64_t T = tiles_of(P, Q), U = T * ceil_div(M, kRows);
  return size_t(std::min<int64_t>(kMaxExactGrid, std::max<int64_t>(U, 1)) + T);
}

size_t exact_part_bytes(int64_t M, int64_t P, int64_t Q) {
  // records (16 bytes) and digit arrays (kExactSlots int64) per segment and output
  const size_t segs = exact_segments(M, P, Q);
  return segs * kOut * (sizeof(longlong2) + kExactSlots * sizeof(long long));
}

cudaError_t launch_exact(const void* left, int ldl, const void* right, int ldr, bool dv, float alpha, int M, int P, int Q,
                         long long* part, bool transpose, long long* out_digits, float* out, int nsm,
                         cudaStream_t st) {
  const int n_tq = int(ceil_div(Q, kTQ));
  const int64_t T = tiles_of(P, Q);
  const int B = int(ceil_div(M, kRows));
  const int64_t U = T * B;
  const int G = int(std::max<int64_t>(1, std::min<int64_t>({int64_t(2) * nsm, U, kMaxExactGrid})));
  const size_t segs = exact_segments(M, P, Q);
  const uint16_t* l = static_cast<const uint16_t*>(left);
  const uint16_t* r = static_cast<const uint16_t*>(right);
  longlong2* rec = reinterpret_cast<longlong2*>(part);
  long long* spill = part + segs * kOut * 2;
  if (U > 0) {
    const cudaError_t e =
        dv ? launch_pdl(exact_digits_kernel<true>, dim3(unsigned(G)), dim3(kThreads), 0, st, l, ldl, r, ldr, M, P, Q,
                        n_tq, B, U, alpha, rec, spill)
           : launch_pdl(exact_digits_kernel<false>, dim3(unsigned(G)), dim3(kThreads), 0, st, l, ldl, r, ldr, M, P,
                        Q, n_tq, B, U, alpha, rec, spill);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(exact_reduce_kernel, dim3(unsigned(ceil_div(int64_t(P) * Q, 256))), dim3(256), 0, st,
                    static_cast<const longlong2*>(rec), static_cast<const long long*>(spill), P, Q, n_tq, B, U, G,
                    transpose ? 1 : 0, out_digits, out);
}

cudaError_t launch_exact_combine(const long long* a, const long long* b, int64_t n, long long* out_digits, float* out,
                                 cudaStream_t st) {
  return launch_pdl(exact_combine_kernel, dim3(unsigned(ceil_div(n, 256))), dim3(256), 0, st, a, b, n, out_digits,
                    out);
}

cudaError_t prepare_exact() { return cudaSuccess; }

}  // namespace lora
