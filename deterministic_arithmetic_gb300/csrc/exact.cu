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
// one tile as a segment, numbered c + t (t the tile). The raw rows of the next
// unit are copied into shared memory (cp.async) while the current one computes.
//
// Per unit, every factor is written as a fixed-point integer scaled to its
// column: with E the biased exponent and C the largest E in the column over the
// 64 rows (found by warp shuffles), a normal factor +-mag 2^(E - 134) (mag the
// significand with its leading bit) becomes f = +-mag 2^(E - C + 20) -- its
// binary32 exponent field raised by 154 - C, then converted exactly to int --
// an integer below 2^28 whenever E >= C - 20. Then each product is one wide
// multiply-add, f_l f_r < 2^56, and a thread's 64-row sum S (below 2^62) of an
// output is exact at the unit position C_l + C_r - 42 (counted from 2^-266). S
// is added, shifted, into a 128-bit window in registers (anchor set 20 bits
// below the first S's position, which leaves 41 bits of room above it), or --
// out of the window's range -- straight into the output's digit array of the
// segment in global memory (owned by the thread; zeroed at its first use).
// Factors more than 20 bits below their column's largest, and subnormal ones
// ("small"; none in data of ordinary range), are written as 0 and their
// products are added exactly one by one from the raw values; so are all the
// products of 64 rows holding an infinite or NaN value (whose products go to
// the counters), or more small factors than the list of them holds. Each
// segment leaves one record per output: the window and whether its digit array
// was used.
// exact_reduce_kernel adds, per output, the windows and digit arrays of the
// segments of its tile, and writes the normalised digits or rounds them.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

constexpr int kTP = 16, kTQ = 64;                // output tile [p][q]
constexpr int kOut = kTP * kTQ;                  // outputs per tile
constexpr int kRows = 64;                        // rows per unit
constexpr int kThreads = 512;                    // two outputs (p, p + 1) per thread
constexpr int kScale = 20;                       // fixed-point bits below a column's largest exponent
constexpr int kWinBelow = 20;                    // window anchor: this far below the first step sum's position
constexpr int kWinAbove = 41;                    // highest step-sum shift the 128-bit window takes
constexpr int kMaxSmall = 256;                   // small factors listed per unit
constexpr int kFlushUnits = 1 << 16;             // a window holds 2^24 step sums below 2^103; spilled sooner

// 128-bit two's complement accumulator
struct I128 {
  unsigned long long lo;
  long long hi;
};

// v * 2^sh (0 <= sh < 64) added into a
__device__ __forceinline__ void add_shifted(I128& a, long long v, int sh) {
  const unsigned long long lo = (unsigned long long)v << sh;
  const long long hi = sh ? (v >> (64 - sh)) : (v >> 63);
  const unsigned long long s = a.lo + lo;
  a.hi += hi + (s < lo ? 1 : 0);
  a.lo = s;
}

// The digit array of one output for one segment: dig[slot * kOut] (global memory, owned by
// one thread), zeroed at its first use.
__device__ __forceinline__ void touch(long long* dig, int& used) {
  if (!used) {
    for (int s = 0; s < kExactSlots; ++s) dig[s * kOut] = 0;
    used = 1;
  }
}

// (hi : lo) * 2^(pos - 266) into the digits, pos in [0, 446] (window anchors): words d .. d + 4
// of v * 2^(pos & 31)
__device__ __forceinline__ void digits_add128(long long* dig, int& used, I128 v, int pos) {
  touch(dig, used);
  const int d = pos >> 5, sa = pos & 31;
  const unsigned long long lo = v.lo << sa;
  const unsigned long long mid = sa ? (v.lo >> (64 - sa)) | ((unsigned long long)v.hi << sa) : (unsigned long long)v.hi;
  const long long top = sa ? (v.hi >> (64 - sa)) : (v.hi >> 63);
  dig[d * kOut] += (long long)(lo & 0xFFFFFFFFull);
  dig[(d + 1) * kOut] += (long long)(lo >> 32);
  dig[(d + 2) * kOut] += (long long)(mid & 0xFFFFFFFFull);
  dig[(d + 3) * kOut] += (long long)(mid >> 32);
  dig[(d + 4) * kOut] += top;
}

// v * 2^(pos - 266) into the digits, pos <= 506 (a negative pos: v is then a multiple of
// 2^-pos, every product's unit lying at position >= 0): words d, d + 1 of v * 2^(pos & 31)
// and the signed rest in d + 2
__device__ __forceinline__ void digits_add64(long long* dig, int& used, long long v, int pos) {
  if (v == 0) return;
  if (pos < 0) {
    v >>= -pos;
    pos = 0;
  }
  touch(dig, used);
  const int d = pos >> 5, sa = pos & 31;
  const unsigned long long lo = (unsigned long long)v << sa;
  const long long hi = sa ? (v >> (64 - sa)) : (v >> 63);
  dig[d * kOut] += (long long)(lo & 0xFFFFFFFFull);
  dig[(d + 1) * kOut] += (long long)(lo >> 32);
  dig[(d + 2) * kOut] += hi;
}

// one product of raw BF16 values a * b into the digits or the special counters
__device__ __forceinline__ void digits_product(long long* dig, int& used, uint32_t a, uint32_t b) {
  const int ea = int(a >> 7) & 0xFF, eb = int(b >> 7) & 0xFF;
  const bool za = (a & 0x7FFFu) == 0u, zb = (b & 0x7FFFu) == 0u;
  const bool nega = (a & 0x8000u) != 0u, negb = (b & 0x8000u) != 0u;
  if (ea == 0xFF || eb == 0xFF) {   // inf or NaN: NaN for a NaN factor or inf * 0
    const bool nan = (ea == 0xFF && (a & 0x7Fu)) || (eb == 0xFF && (b & 0x7Fu)) || za || zb;
    touch(dig, used);
    dig[(nan ? kDigits + 2 : (nega != negb ? kDigits + 1 : kDigits)) * kOut] += 1;
    return;
  }
  if (za || zb) return;
  const int ma = (ea ? 0x80 : 0) | int(a & 0x7Fu), mb = (eb ? 0x80 : 0) | int(b & 0x7Fu);
  const long long v = (long long)(nega != negb ? -(ma * mb) : ma * mb);
  digits_add64(dig, used, v, max(ea, 1) + max(eb, 1) - 268 + 266);
}

// a * b + c with a 64-bit product and addend (one multiply-add)
__device__ __forceinline__ long long mad_wide(int a, int b, long long c) {
  long long d;
  asm("mad.wide.s32 %0, %1, %2, %3;" : "=l"(d) : "r"(a), "r"(b), "l"(c));
  return d;
}

// 16-byte asynchronous copy global -> shared; bytes = 0 fills the 16 bytes with zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(uint32_t(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// shared memory of the digit kernel (row pitches padded against bank conflicts)
constexpr int kRawLP = 24, kRawRP = 72, kFrP = 68;
struct ExactSmem {
  uint16_t raw_l[2][kRows][kRawLP];   // raw BF16 rows (dV for the right rows of dB), double-buffered
  uint16_t raw_r[2][kRows][kRawRP];
  int frT[kTQ][kFrP];                 // right fixed-point factors, column-major
  int flT[kTP / 2][kRows][2];         // left fixed-point factors, column pairs
  int cl[kTP], cr[kTQ];               // column maxima of the biased exponent over the 64 rows
  uint32_t small[kMaxSmall];          // small factors: right << 31 | row << 16 | column
  int n_small[2];                     // their count (by unit parity)
};

// Start the copies of the raw rows of unit (tile at p0, q0; row block blk) into buffer b (one
// 16-byte chunk of the right rows per thread, one of the left rows for the first 128 threads;
// zeros past M, P and Q).
__device__ __forceinline__ void fetch_unit(ExactSmem& sm, int b, int p0, int q0, int blk, const uint16_t* left,
                                           int ldl, const uint16_t* right, int ldr, int M, int P, int Q) {
  const int m0 = blk * kRows;
  const int tid = threadIdx.x;
  {
    const int r = tid / (kTQ / 8), c8 = (tid % (kTQ / 8)) * 8;   // 512 chunks: 64 rows x 8
    const bool ok = m0 + r < M && q0 + c8 < Q;
    cp_async16(&sm.raw_r[b][r][c8], ok ? right + size_t(m0 + r) * ldr + q0 + c8 : right, ok ? 16 : 0);
  }
  if (tid < kRows * (kTP / 8)) {
    const int r = tid / (kTP / 8), c8 = (tid % (kTP / 8)) * 8;   // 128 chunks: 64 rows x 2
    const bool ok = m0 + r < M && p0 + c8 < P;
    cp_async16(&sm.raw_l[b][r][c8], ok ? left + size_t(m0 + r) * ldl + p0 + c8 : left, ok ? 16 : 0);
  }
}

// The fixed-point factor +-mag 2^(E - c + kScale) of a BF16 value h (E its biased exponent,
// mag its significand with the leading bit) in a column whose largest E is c: adding
// (154 - c) << 23 to the exponent field of h as binary32 gives exactly that integer (below
// 2^28) whenever E >= max(c - kScale, 1), and the conversion to int is then exact. Otherwise
// the factor is 0, and small is set when h is non-zero (a subnormal, or more than kScale bits
// below c). Not for inf or NaN (rows holding one take another path).
struct ColScale {
  uint32_t adj;   // (154 - c) << 23
  int lo;         // max(c - kScale, 1)
};
__device__ __forceinline__ ColScale col_scale(int c) { return ColScale{uint32_t(154 - c) << 23, max(c - kScale, 1)}; }
__device__ __forceinline__ int fixed_factor(uint32_t h, ColScale cs, bool& small) {
  const uint32_t x = h << 16;
  const int e = int(x >> 23) & 0xFF;
  const bool ok = e >= cs.lo;
  small = !ok && (x & 0x7FFF0000u) != 0u;
  return ok ? __float2int_rz(__uint_as_float(x + cs.adj)) : 0;
}

// The window of one output: a 128-bit sum at anchor anc (-1: none yet) and whether the
// output's digit array for the segment has been used.
struct Win {
  I128 acc;
  int anc;
  int used;
};

// the 64-row sum s at unit position pos added to the window (or, outside its range, to the digits)
__device__ __forceinline__ void window_fold(Win& w, long long* dig, long long s, int pos) {
  if (s == 0) return;
  if (w.anc < 0) w.anc = max(pos - kWinBelow, 0);
  const int sh = pos - w.anc;
  if (sh >= 0 && sh <= kWinAbove) add_shifted(w.acc, s, sh);
  else digits_add64(dig, w.used, s, pos);
}

__device__ __forceinline__ void window_spill(Win& w, long long* dig) {
  if (w.anc >= 0 && (w.acc.lo != 0 || w.acc.hi != 0)) digits_add128(dig, w.used, w.acc, w.anc);
  w.acc = I128{0, 0};
}

// CTA of unit u when U units are split among G CTAs as [c U / G, (c + 1) U / G)
__host__ __device__ __forceinline__ int cta_of_unit(int64_t u, int64_t U, int G) {
  return int(((u + 1) * G - 1) / U);
}

// Segment record of one output: the window (lo, hi) and anc | used << 32 (anc = -1: none)
struct ExactRec {
  unsigned long long lo;
  long long hi;
  long long tag;
  long long pad;
};

// DV: the right operand is dV = bf16(fp32(dy * alpha)), formed from dY.
// Tiles: t = tp * n_tq + tq (16 rows of P by 64 columns of Q); B row blocks of 64 per tile.
// rec[seg][o], spill[seg][slot][o] with o = (p - p0) * 64 + (q - q0), seg = c + t.
// Left and right rows are 16-byte aligned (P, Q, ldl, ldr multiples of 8).
template <bool DV>
__global__ void __launch_bounds__(kThreads, 2)
    exact_digits_kernel(const uint16_t* __restrict__ left, int ldl, const uint16_t* __restrict__ right, int ldr,
                        int M, int P, int Q, int n_tq, int B, int64_t U, float alpha, ExactRec* __restrict__ rec,
                        long long* __restrict__ spill) {
  grid_dependency_wait();
  grid_dependents_launch();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ExactSmem& sm = *reinterpret_cast<ExactSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int q = tid % kTQ, pg = tid / kTQ;            // outputs (2 pg, q) and (2 pg + 1, q)
  const int oa = 2 * pg * kTQ + q, ob = oa + kTQ;     // their indexes in the tile
  const int dr_c = tid / 8, dr_i = tid % 8;           // decoding: right column, rows dr_i + 8 k
  const int G = gridDim.x, c = blockIdx.x;
  const int64_t u_begin = int64_t(c) * U / G, u_end = (int64_t(c) + 1) * U / G;
  if (tid < 2) sm.n_small[tid] = 0;
  // the unit (tile, row block) now and next, advanced without divisions; the next tile's corner
  int tile = u_begin < u_end ? int(u_begin / B) : 0, blk = int(u_begin - int64_t(tile) * B);
  int next_tile = tile, next_blk = blk, next_q0 = (tile % n_tq) * kTQ, next_p0 = (tile / n_tq) * kTP;
  if (u_begin < u_end) fetch_unit(sm, 0, next_p0, next_q0, blk, left, ldl, right, ldr, M, P, Q);
  cp_async_commit();
  int units = 0;
  size_t seg = 0;
  long long *dig_a = spill, *dig_b = spill;
  Win wa{{0, 0}, -1, 0}, wb{{0, 0}, -1, 0};
  for (int64_t u = u_begin; u < u_end; ++u) {
    const int buf = int((u - u_begin) & 1);
    tile = next_tile;
    blk = next_blk;
    if (++next_blk == B) {
      next_blk = 0;
      ++next_tile;
      if ((next_q0 += kTQ) >= n_tq * kTQ) {
        next_q0 = 0;
        next_p0 += kTP;
      }
    }
    if (u == u_begin || blk == 0) {   // a new segment
      seg = size_t(c) + tile;
      dig_a = spill + seg * kExactSlots * kOut + oa;
      dig_b = spill + seg * kExactSlots * kOut + ob;
      wa = Win{{0, 0}, -1, 0};
      wb = Win{{0, 0}, -1, 0};
      units = 0;
    }
    cp_async_wait_all();   // this thread's copies of unit u have landed
    __syncthreads();       // everyone's; the previous unit consumed; buffer buf ^ 1 free
    if (u + 1 < u_end) fetch_unit(sm, buf ^ 1, next_p0, next_q0, next_blk, left, ldl, right, ldr, M, P, Q);
    cp_async_commit();
    if (tid == 0) sm.n_small[buf ^ 1] = 0;
    // decode: each group of 8 lanes takes one right column (rows dr_i + 8 k), each warp one left
    // column (rows lane and lane + 32); the column's largest E' by shuffles, then the fixed-point
    // factors; small ones listed; inf / NaN noted
    int special = 0;
    {
      uint32_t h[8];
      int mx = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        h[k] = sm.raw_r[buf][dr_i + 8 * k][dr_c];
        if (DV) {
          h[k] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__uint_as_float(h[k] << 16), alpha)));
          sm.raw_r[buf][dr_i + 8 * k][dr_c] = uint16_t(h[k]);
        }
        mx = max(mx, int(h[k] >> 7) & 0xFF);
      }
#pragma unroll
      for (int s = 1; s < 8; s <<= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, s));
      special |= mx == 0xFF;
      if (dr_i == 0) sm.cr[dr_c] = mx;
      const ColScale cs = col_scale(mx);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        bool s = false;
        sm.frT[dr_c][dr_i + 8 * k] = fixed_factor(h[k], cs, s);
        if (s) {
          const int i = atomicAdd(&sm.n_small[buf], 1);
          if (i < kMaxSmall) sm.small[i] = 0x80000000u | uint32_t((dr_i + 8 * k) << 16 | dr_c);
        }
      }
    }
    {
      const uint32_t h0 = sm.raw_l[buf][lane][warp], h1 = sm.raw_l[buf][lane + 32][warp];
      int mx = max(int(h0 >> 7) & 0xFF, int(h1 >> 7) & 0xFF);
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, s));
      special |= mx == 0xFF;
      if (lane == 0) sm.cl[warp] = mx;
      const ColScale cs = col_scale(mx);
      bool s0 = false, s1 = false;
      sm.flT[warp / 2][lane][warp % 2] = fixed_factor(h0, cs, s0);
      sm.flT[warp / 2][lane + 32][warp % 2] = fixed_factor(h1, cs, s1);
      if (s0) {
        const int i = atomicAdd(&sm.n_small[buf], 1);
        if (i < kMaxSmall) sm.small[i] = uint32_t(lane << 16 | warp);
      }
      if (s1) {
        const int i = atomicAdd(&sm.n_small[buf], 1);
        if (i < kMaxSmall) sm.small[i] = uint32_t((lane + 32) << 16 | warp);
      }
    }
    const bool any_special = __syncthreads_or(special);
    const int n_small = sm.n_small[buf];
    if (any_special || n_small > kMaxSmall) {
      // every product of these rows, one by one from the raw values
      for (int r = 0; r < kRows; ++r) {
        const uint32_t hr = sm.raw_r[buf][r][q];
        digits_product(dig_a, wa.used, sm.raw_l[buf][r][2 * pg], hr);
        digits_product(dig_b, wb.used, sm.raw_l[buf][r][2 * pg + 1], hr);
      }
    } else {
      long long sa = 0, sb = 0;
#pragma unroll 4
      for (int r = 0; r < kRows; r += 4) {
        const int4 fr = *reinterpret_cast<const int4*>(&sm.frT[q][r]);
        const int4 f01 = *reinterpret_cast<const int4*>(&sm.flT[pg][r][0]);      // rows r, r + 1
        const int4 f23 = *reinterpret_cast<const int4*>(&sm.flT[pg][r + 2][0]);  // rows r + 2, r + 3
        sa = mad_wide(f01.x, fr.x, sa);
        sb = mad_wide(f01.y, fr.x, sb);
        sa = mad_wide(f01.z, fr.y, sa);
        sb = mad_wide(f01.w, fr.y, sb);
        sa = mad_wide(f23.x, fr.z, sa);
        sb = mad_wide(f23.y, fr.z, sb);
        sa = mad_wide(f23.z, fr.w, sa);
        sb = mad_wide(f23.w, fr.w, sb);
      }
      const int crq = sm.cr[q];
      window_fold(wa, dig_a, sa, sm.cl[2 * pg] + crq - 2 * kScale - 2);
      window_fold(wb, dig_b, sb, sm.cl[2 * pg + 1] + crq - 2 * kScale - 2);
      // the small factors' products, exactly (a product of two small factors once: with the
      // left one's entry)
      for (int i = 0; i < n_small; ++i) {
        const uint32_t e = sm.small[i];
        const int r = int(e >> 16) & 0x7FFF, col = int(e & 0xFFFFu);
        if (e >> 31) {   // right factor (r, col): with every left factor of row r that is not small
          if (col != q) continue;
          const uint32_t hr = sm.raw_r[buf][r][q];
          if (sm.flT[pg][r][0] != 0) digits_product(dig_a, wa.used, sm.raw_l[buf][r][2 * pg], hr);
          if (sm.flT[pg][r][1] != 0) digits_product(dig_b, wb.used, sm.raw_l[buf][r][2 * pg + 1], hr);
        } else {         // left factor (r, col): with every right factor of row r
          if ((col >> 1) != pg) continue;
          if (col & 1) digits_product(dig_b, wb.used, sm.raw_l[buf][r][col], sm.raw_r[buf][r][q]);
          else digits_product(dig_a, wa.used, sm.raw_l[buf][r][col], sm.raw_r[buf][r][q]);
        }
      }
    }
    if (++units == kFlushUnits) {   // window headroom
      window_spill(wa, dig_a);
      window_spill(wb, dig_b);
      units = 0;
    }
    if (u + 1 == u_end || next_tile != tile) {   // the segment ends: its records
      rec[seg * kOut + oa] = ExactRec{wa.acc.lo, wa.acc.hi, (long long)(uint32_t)wa.anc | ((long long)wa.used << 32), 0};
      rec[seg * kOut + ob] = ExactRec{wb.acc.lo, wb.acc.hi, (long long)(uint32_t)wb.anc | ((long long)wb.used << 32), 0};
    }
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
__global__ void __launch_bounds__(256) exact_reduce_kernel(const ExactRec* __restrict__ rec,
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
      const ExactRec r = rec[seg * kOut + o];
      const int anc = int(r.tag & 0xFFFFFFFF);
      if (anc >= 0) {   // window (hi : lo) * 2^(anc - 266): words d .. d + 4 of it * 2^(anc & 31)
        const int d = anc >> 5, sa = anc & 31;
        const unsigned long long lo = r.lo << sa;
        const unsigned long long mid = sa ? (r.lo >> (64 - sa)) | ((unsigned long long)r.hi << sa) : (unsigned long long)r.hi;
        const long long top = sa ? (r.hi >> (64 - sa)) : (r.hi >> 63);
        const long long w[5] = {(long long)(lo & 0xFFFFFFFFull), (long long)(lo >> 32), (long long)(mid & 0xFFFFFFFFull),
                                (long long)(mid >> 32), top};
#pragma unroll
        for (int s = 0; s < kDigits; ++s) {
          long long v = 0;
#pragma unroll
          for (int j = 0; j < 5; ++j) v = s == d + j ? w[j] : v;
          c[s] += v;
        }
      }
      if ((r.tag >> 32) & 1) {
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
  // records and digit arrays (kExactSlots int64) per segment and output
  const size_t segs = exact_segments(M, P, Q);
  return segs * kOut * (sizeof(ExactRec) + kExactSlots * sizeof(long long));
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
  ExactRec* rec = reinterpret_cast<ExactRec*>(part);
  long long* spill = part + segs * kOut * (sizeof(ExactRec) / sizeof(long long));
  if (U > 0) {
    const cudaError_t e =
        dv ? launch_pdl(exact_digits_kernel<true>, dim3(unsigned(G)), dim3(kThreads), sizeof(ExactSmem), st, l, ldl, r, ldr, M, P, Q,
                        n_tq, B, U, alpha, rec, spill)
           : launch_pdl(exact_digits_kernel<false>, dim3(unsigned(G)), dim3(kThreads), sizeof(ExactSmem), st, l, ldl, r, ldr, M, P,
                        Q, n_tq, B, U, alpha, rec, spill);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(exact_reduce_kernel, dim3(unsigned(ceil_div(int64_t(P) * Q, 256))), dim3(256), 0, st,
                    static_cast<const ExactRec*>(rec), static_cast<const long long*>(spill), P, Q, n_tq, B, U, G,
                    transpose ? 1 : 0, out_digits, out);
}

cudaError_t launch_exact_combine(const long long* a, const long long* b, int64_t n, long long* out_digits, float* out,
                                 cudaStream_t st) {
  return launch_pdl(exact_combine_kernel, dim3(unsigned(ceil_div(n, 256))), dim3(256), 0, st, a, b, n, out_digits,
                    out);
}

// The ceiling of the digit kernel's product step, measured: independent chains of 32-bit wide
// multiply-adds (one per product of an exact sum) in the digit kernel's launch shape (two CTAs of
// kThreads threads per SM). Each thread runs kProbeChains chains for `iters` rounds; the right
// factor changes every round, so every product is a new one, and the chains' sum goes to
// sink[thread] so that none of the work can be dropped.
constexpr int kProbeChains = 8;
__global__ void __launch_bounds__(kThreads, 2) exact_rate_probe_kernel(int iters, long long* sink) {
  int a[kProbeChains];
  long long acc[kProbeChains];
#pragma unroll
  for (int j = 0; j < kProbeChains; ++j) {
    a[j] = int(threadIdx.x) * kProbeChains + j + 1;
    acc[j] = j;
  }
  const int b0 = int(blockIdx.x) | 1;
  for (int i = 0; i < iters; ++i) {
    const int b = b0 + i;
#pragma unroll
    for (int j = 0; j < kProbeChains; ++j) asm volatile("mad.wide.s32 %0, %1, %2, %0;" : "+l"(acc[j]) : "r"(a[j]), "r"(b));
  }
  long long t = 0;
#pragma unroll
  for (int j = 0; j < kProbeChains; ++j) t += acc[j];
  sink[size_t(blockIdx.x) * blockDim.x + threadIdx.x] = t;
}

size_t exact_probe_sink_bytes(int nsm) { return size_t(2) * nsm * kThreads * sizeof(long long); }

cudaError_t launch_exact_rate_probe(int iters, long long* sink, int nsm, int64_t* products, cudaStream_t st) {
  *products = int64_t(2) * nsm * kThreads * kProbeChains * int64_t(iters);
  exact_rate_probe_kernel<<<dim3(unsigned(2 * nsm)), dim3(kThreads), 0, st>>>(iters, sink);
  return cudaGetLastError();
}

cudaError_t prepare_exact() {
  cudaError_t e = cudaFuncSetAttribute(exact_digits_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(sizeof(ExactSmem)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(exact_digits_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(sizeof(ExactSmem)));
}

}  // namespace lora
