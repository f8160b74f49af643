// Low-bit group quantiser and hybrid-cache construction.
//
// Quant_B(.; G) of Algorithm 4 ("HyQuant: Hybrid-Precision Quantization for
// LLM Attention", Appendix A.4) with B = B_K for keys and B_V for values (4 or
// 8 bits) and G = 32 along head_dim, and the
// Freeze re-organisation of the cache into a 4-bit stream, vertical-line rows
// and a BF16 tail (§4.3 Eq. 8).
//
// A CTA builds one 64-row block of the 4-bit stream: the BF16 rows are staged
// in shared memory with each group's min / max, one thread per group derives
// the FP16 step and zero point, and each thread then assembles whole 32-bit
// code words in the tensor-core fragment order documented in hyq.h and
// stores them directly (no atomics, no float64).
#include <type_traits>

#include "hyq_common.cuh"
#include "hyq_f2.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = HYQ_QBLOCK_ROWS;  // 64 stream rows per block
constexpr int kChunks = HYQ_D / 8;      // 16 chunks of 8 elements per row

// Shared image of one 64-row block being built.
struct BuildSmem {
  __nv_bfloat16 x[2][kRows][HYQ_D];  // K and V rows (zero for padding / kept rows)
  float mn[2][kRows][4], mx[2][kRows][4];
  float z[2][kRows][4], r[2][kRows][4], s[2][kRows][4];
  int32_t pos[kRows];      // source row of each slot, -1 for none
  uint8_t keep[kRows];     // slot already holds a stream row (append)
  uint8_t nan[2][kRows][4];
  uint8_t fast[2][kRows][4];  // every code of the group needs no clamp
};

// Rounding by addition: for |t| < 2^22, fl32(t + 1.5 * 2^23) is
// 1.5 * 2^23 + rint(t) (the sum's ulp is 1, ties to even), so its bit
// pattern is kMagicBits + rint(t).
constexpr float kMagic = 12582912.f;
constexpr uint32_t kMagicBits = 0x4B400000u;
__host__ __device__ constexpr uint32_t magic_sum8() {
  uint32_t s = 0;
  for (int p = 0; p < 8; ++p) s += kMagicBits << (4 * p);
  return s;
}
constexpr uint32_t kMagicSum = magic_sum8();

__device__ __forceinline__ uint32_t lo32(uint64_t v) { return (uint32_t)v; }
__device__ __forceinline__ uint32_t hi32(uint64_t v) { return (uint32_t)(v >> 32); }

// The code is the grid point z + c s nearest to x, ties to the even c.  It is
// found from t = fl32(fl32(x - z) * r), r = RN(1/s), whose relative error is
// at most about 3 * 2^-24 (|t| < 2^8 where it matters: under 5e-5), so
// rint(t) is the exact answer unless t lies within kNearTie of a half
// integer; those elements are decided exactly (exact_code).
constexpr float kNearTie = 0.5f - 0.000244140625f;  // 1/2 - 2^-12

// Step of a group: the smallest FP16 value s with qmax s >= mx - mn (the
// subtraction, the division and the FP16 conversion all round up, which gives
// exactly that value: qmax h is exact in FP32 for every FP16 h).
__device__ __forceinline__ __half group_step(float mn, float mx, float qmax) {
  return __float2half_ru(__fdiv_ru(__fsub_ru(mx, mn), qmax));
}

// Exact decision near the midpoint k + 1/2, k = floor(t): in float64 the
// midpoint z + (k + 1/2) s is exact (s and z are FP16 values: a multiple of
// 2^-25 below 2^25 in magnitude) and the sign of x minus it is exact.
__device__ __forceinline__ float exact_code(float x, float z, float s, float t) {
  const float k = floorf(t);
  const double d = (double)x - ((double)z + ((double)k + 0.5) * (double)s);
  if (d > 0.0) return k + 1.f;
  if (d < 0.0) return k;
  return (__float2int_rz(k) & 1) ? k + 1.f : k;  // a tie: the even one
}

// Bit patterns kMagicBits + code of the two BF16 elements of w (x: low half),
// for a group whose (x - z) * r all lie in (-0.5, 15.5): there the clamp of
// the code decision is the identity and the added magic rounds exactly as
// rint does.  nz2 = (-z, -z), r2 = (r, r).  The magic add is a scalar
// __fadd_rn, which is never contracted with the product into a fused
// multiply-add (that would round the unrounded product).  `near` is set when
// either element lies within kNearTie of a midpoint (the caller then takes
// the exact path for the whole word).
__device__ __forceinline__ uint2 code_bits2(uint32_t w, uint64_t nz2, uint64_t r2, bool& near) {
  const uint64_t x2 = (uint64_t)(w << 16) | ((uint64_t)(w & 0xffff0000u) << 32);
  const uint64_t t2 = f2_mul(f2_add(x2, nz2), r2);
  const float t0 = __uint_as_float(lo32(t2)), t1 = __uint_as_float(hi32(t2));
  const float b0 = __fadd_rn(t0, kMagic), b1 = __fadd_rn(t1, kMagic);
  near |= fabsf(__fsub_rn(t0, __fsub_rn(b0, kMagic))) > kNearTie ||
          fabsf(__fsub_rn(t1, __fsub_rn(b1, kMagic))) > kNearTie;
  return make_uint2(__float_as_uint(b0), __float_as_uint(b1));
}

// Code word from b[p] = kMagicBits + code of nibble p: the shift-add chain
// sums b[p] << 4p modulo 2^32, which is the word plus sum_p kMagicBits << 4p.
__device__ __forceinline__ uint32_t pack_nibbles(const uint32_t (&b)[8]) {
  uint32_t w = b[7];
#pragma unroll
  for (int p = 6; p >= 0; --p) w = (w << 4) + b[p];
  return w - kMagicSum;
}

// r = 1 / s rounded, and 0 exactly when the step s is 0; qmax = 2^B - 1.
__device__ __forceinline__ uint32_t code_of(float x, float z, float r, float s, float qmax = 15.f) {
  if (r == 0.f) return 0u;
  const float t = __fmul_rn(__fsub_rn(x, z), r);
  float c = rintf(t);
  if (fabsf(__fsub_rn(t, c)) > kNearTie) c = exact_code(x, z, s, t);
  c = fminf(fmaxf(c, 0.f), qmax);
  return (uint32_t)c;
}

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Pass 3 of an 8-bit code region (tensor T: 0 = K, 1 = V): one 32-bit word
// (four codes of the byte order in hyq.h) per job; rows with keep = 1 keep
// their bytes.
template <int T, int kTileBytes, int kOff>
__device__ void pack_codes8(const BuildSmem& sm, uint8_t* dst, bool any_keep) {
  for (int j = threadIdx.x; j < 4 * 32 * 16; j += kThreads) {
    const int tile = j >> 9, lane = (j >> 4) & 31, u = j & 15;
    const int g = lane >> 2, t = lane & 3;
    uint8_t* wp = dst + tile * kTileBytes + kOff + 512 * (u >> 2) + 16 * lane + 4 * (u & 3);
    const uint32_t old = any_keep ? *reinterpret_cast<const uint32_t*>(wp) : 0u;
    uint32_t w = 0;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      // K: row g + 8(u%2), element 16(u/2) + 4t + (0, 2, 1, 3)[jj];
      // V: row 2t + (0, 8, 1, 9)[jj], element 32(u/4) + 4g + 2((u/2)%2) + u%2
      const int row = T == 0 ? 16 * tile + g + 8 * (u & 1) : 16 * tile + 2 * t + 8 * (jj & 1) + (jj >> 1);
      const int e = T == 0 ? 16 * (u >> 1) + 4 * t + 2 * (jj & 1) + (jj >> 1)
                           : 32 * (u >> 2) + 4 * g + 2 * ((u >> 1) & 1) + (u & 1);
      const int q = e >> 5;
      const uint32_t c = sm.keep[row] ? (old >> (8 * jj)) & 0xFFu
                                      : code_of(__bfloat162float(sm.x[T][row][e]), sm.z[T][row][q], sm.r[T][row][q],
                                                sm.s[T][row][q], 255.f);
      w |= c << (8 * jj);
    }
    *reinterpret_cast<uint32_t*>(wp) = w;
  }
}

// Build one 64-row block of the quantised stream at `dst` (global), keys with
// BK-bit and values with BV-bit codes.  sm.pos / sm.keep must be set.  Rows
// with keep = 1 keep their existing codes and metadata; rows with pos < 0
// become zero padding.
template <int BK, int BV>
__device__ void build_block(BuildSmem& sm, const __nv_bfloat16* kbase, const __nv_bfloat16* vbase,
                            uint8_t* dst, bool any_keep, int32_t* err) {
  using F = QFmt<BK, BV>;
  const int tid = threadIdx.x;
  // Pass 1: load the rows (all of a thread's loads first), per-group min /
  // max (4 chunks of 8 per group are on 4 consecutive lanes).
  constexpr int kPer = 2 * kRows * kChunks / kThreads;
  uint4 vin[kPer];
#pragma unroll
  for (int it = 0; it < kPer; ++it) {
    const int f = tid + it * kThreads;
    const int T = f >> 10, row = (f >> 4) & (kRows - 1), c = f & (kChunks - 1);
    const int32_t p = sm.pos[row];
    vin[it] = make_uint4(0, 0, 0, 0);
    if (p >= 0 && !sm.keep[row])
      vin[it] = __ldg(reinterpret_cast<const uint4*>((T ? vbase : kbase) + (size_t)p * HYQ_D + 8 * c));
  }
#pragma unroll
  for (int it = 0; it < kPer; ++it) {
    const int f = tid + it * kThreads;
    const int T = f >> 10, row = (f >> 4) & (kRows - 1), c = f & (kChunks - 1);
    const uint4 v = vin[it];
    *reinterpret_cast<uint4*>(&sm.x[T][row][8 * c]) = v;
    // BF16 pairs: min / max are exact in BF16, and the _nan forms carry a
    // NaN through, so one test at the end finds any NaN of the group.
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
    __nv_bfloat162 mn2 = __hmin2_nan(__hmin2_nan(p2[0], p2[1]), __hmin2_nan(p2[2], p2[3]));
    __nv_bfloat162 mx2 = __hmax2_nan(__hmax2_nan(p2[0], p2[1]), __hmax2_nan(p2[2], p2[3]));
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      mn2 = __hmin2_nan(mn2, __shfl_xor_sync(0xffffffffu, mn2, o));
      mx2 = __hmax2_nan(mx2, __shfl_xor_sync(0xffffffffu, mx2, o));
    }
    if ((c & 3) == 0) {
      const float2 fm = __bfloat1622float2(mn2), fx = __bfloat1622float2(mx2);
      sm.mn[T][row][c >> 2] = fminf(fm.x, fm.y);
      sm.mx[T][row][c >> 2] = fmaxf(fx.x, fx.y);
      sm.nan[T][row][c >> 2] = (uint8_t)(isnan(fm.x) || isnan(fm.y));
    }
  }
  __syncthreads();
  // Pass 2: one thread per group: step s = smallest FP16 with qmax s >= mx - mn
  // (the subtraction, the division and the FP16 conversion all round up,
  // which gives exactly that value: qmax h is exact in FP32 for every FP16 h);
  // zero z = FP16(mn) to nearest.
  for (int i = tid; i < 2 * kRows * 4; i += kThreads) {
    const int T = i >> 8, row = (i >> 2) & (kRows - 1), q = i & 3;
    if (sm.keep[row]) continue;
    const float qmax = (T == 0 ? BK : BV) == 8 ? 255.f : 15.f;
    const float mn = sm.mn[T][row][q], mx = sm.mx[T][row][q];
    __half sh = group_step(mn, mx, qmax);
    __half zh = __float2half_rn(mn);
    float s32 = __half2float(sh), z32 = __half2float(zh);
    if (sm.nan[T][row][q] || isinf(s32) || isinf(z32)) {
      hyq_set_err(err, HYQ_DEVERR_QUANT_RANGE);
      sh = zh = __float2half_rn(0.f);
      s32 = z32 = 0.f;
    }
    const float r32 = s32 > 0.f ? __frcp_rn(s32) : 0.f;
    sm.z[T][row][q] = z32;
    sm.r[T][row][q] = r32;
    sm.s[T][row][q] = s32;
    // (x - z) * r is monotone in x, so the group's extremes bound every code
    // argument; a NaN extreme fails the test.
    const float tl = __fmul_rn(__fsub_rn(mn, z32), r32), th = __fmul_rn(__fsub_rn(mx, z32), r32);
    sm.fast[T][row][q] = (uint8_t)(tl > -0.5f && th < qmax + 0.5f);
    // Metadata order of hyq.h: K rows hold four scales then four zeros; V
    // rows pair up (2i, 2i + 1), scales in the first half, zeros in the second.
    uint8_t* mb = dst + (row >> 4) * F::kTile + F::kKMeta + T * 256;
    const int r = row & 15;
    const int so = T == 0 ? 16 * r + 2 * q : 16 * (r >> 1) + 4 * q + 2 * (r & 1);
    const int zo = T == 0 ? so + 8 : so + 128;
    *reinterpret_cast<uint16_t*>(mb + so) = __half_as_ushort(sh);
    *reinterpret_cast<uint16_t*>(mb + zo) = __half_as_ushort(zh);
  }
  __syncthreads();
  if (BK == 8) pack_codes8<0, F::kTile, 0>(sm, dst, any_keep);
  if (BV == 8) pack_codes8<1, F::kTile, F::kVCode>(sm, dst, any_keep);
  // Pass 3a: 4-bit K code words.  Job (tile, g, chunk cc): rows g and g+8 of
  // the tile, elements 8cc..8cc+7 -> the two words u = 2(cc/4) + {0,1} of lane 4g + cc%4.
  for (int j = tid; j < (BK == 4 ? 4 * 8 * kChunks : 0); j += kThreads) {
    const int tile = j >> 7, g = (j >> 4) & 7, cc = j & 15;
    const int q = cc >> 2, t = cc & 3;
    uint8_t* wp = dst + tile * F::kTile + 512 * (cc >> 3) + 16 * (4 * g + t) + 4 * (2 * (q & 1));
    const int rk0 = 16 * tile + g, rk1 = rk0 + 8;
    if (!any_keep && sm.fast[0][rk0][q] && sm.fast[0][rk1][q]) {
      // Row a, element 4 sub + 2 b + c -> nibble a + 2 b + 4 c of word sub.
      uint2 pb[2][4];
      bool near = false;
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int row = a ? rk1 : rk0;
        const uint4 xv = *reinterpret_cast<const uint4*>(&sm.x[0][row][8 * cc]);
        const uint64_t nz2 = f2_splat(-sm.z[0][row][q]), r2 = f2_splat(sm.r[0][row][q]);
        pb[a][0] = code_bits2(xv.x, nz2, r2, near);
        pb[a][1] = code_bits2(xv.y, nz2, r2, near);
        pb[a][2] = code_bits2(xv.z, nz2, r2, near);
        pb[a][3] = code_bits2(xv.w, nz2, r2, near);
      }
      uint32_t wf[2];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        uint32_t bb[8];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            bb[a + 2 * b] = pb[a][2 * sub + b].x;
            bb[a + 2 * b + 4] = pb[a][2 * sub + b].y;
          }
        wf[sub] = pack_nibbles(bb);
      }
      if (!near) {
        *reinterpret_cast<uint2*>(wp) = make_uint2(wf[0], wf[1]);
        continue;
      }
    }
    uint32_t w[2] = {0u, 0u};
    uint2 old = make_uint2(0, 0);
    if (any_keep) old = *reinterpret_cast<const uint2*>(wp);
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int row = 16 * tile + g + 8 * a;
      if (sm.keep[row]) {
        const uint32_t mm = 0x0F0F0F0Fu << (4 * a);  // this row's nibbles a + 2b + 4c
        w[0] |= old.x & mm;
        w[1] |= old.y & mm;
        continue;
      }
      float e[8];
      unpack8(*reinterpret_cast<const uint4*>(&sm.x[0][row][8 * cc]), e);
      const float z = sm.z[0][row][q], r = sm.r[0][row][q], sc = sm.s[0][row][q];
#pragma unroll
      for (int sub = 0; sub < 2; ++sub)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            w[sub] |= code_of(e[4 * sub + 2 * b + c], z, r, sc) << (4 * (a + 2 * b + 4 * c));
    }
    *reinterpret_cast<uint2*>(wp) = make_uint2(w[0], w[1]);
  }
  // Pass 3b: 4-bit V code words.  Job (tile, t, chunk cc): rows 2t + 8b + c,
  // elements 8cc..8cc+7 = 32q + 4g + 2s + a with q = cc/4 and g = 2(cc%4) + gl
  // -> the words (lane 4g + t, u = 2q + s) for gl, s in {0, 1}; the two s
  // words of one lane are adjacent.
  for (int j = tid; j < (BV == 4 ? 4 * 4 * kChunks : 0); j += kThreads) {
    const int tile = j >> 6, t = (j >> 4) & 3, cc = j & 15;
    const int q = cc >> 2;
    const int rv = 16 * tile + 2 * t;  // rows rv + 8 b + c
    if (!any_keep && sm.fast[1][rv][q] && sm.fast[1][rv + 1][q] && sm.fast[1][rv + 8][q] &&
        sm.fast[1][rv + 9][q]) {
      // Row (b, c), element 4 gl + 2 ss + a -> nibble a + 2 b + 4 c of word (gl, ss).
      uint2 pb[4][4];
      bool near = false;
#pragma unroll
      for (int bc = 0; bc < 4; ++bc) {
        const int row = rv + 8 * (bc & 1) + (bc >> 1);
        const uint4 xv = *reinterpret_cast<const uint4*>(&sm.x[1][row][8 * cc]);
        const uint64_t nz2 = f2_splat(-sm.z[1][row][q]), r2 = f2_splat(sm.r[1][row][q]);
        pb[bc][0] = code_bits2(xv.x, nz2, r2, near);
        pb[bc][1] = code_bits2(xv.y, nz2, r2, near);
        pb[bc][2] = code_bits2(xv.z, nz2, r2, near);
        pb[bc][3] = code_bits2(xv.w, nz2, r2, near);
      }
#pragma unroll
      for (int gl = 0; gl < 2; ++gl) {
        uint32_t wf[2];
#pragma unroll
        for (int ss = 0; ss < 2; ++ss) {
          uint32_t bb[8];
#pragma unroll
          for (int bc = 0; bc < 4; ++bc) {  // b = bc & 1, c = bc >> 1: nibbles 2 b + 4 c + a
            const int n0 = 2 * (bc & 1) + 4 * (bc >> 1);
            bb[n0] = pb[bc][2 * gl + ss].x;
            bb[n0 + 1] = pb[bc][2 * gl + ss].y;
          }
          wf[ss] = pack_nibbles(bb);
        }
        const int g = 2 * (cc & 3) + gl;
        if (!near)
          *reinterpret_cast<uint2*>(dst + tile * F::kTile + F::kVCode + 512 * (cc >> 3) + 16 * (4 * g + t) +
                                    8 * (q & 1)) = make_uint2(wf[0], wf[1]);
      }
      if (!near) continue;
    }
    uint8_t* wp[2];
    uint32_t w[2][2] = {{0u, 0u}, {0u, 0u}};
    uint2 old[2] = {make_uint2(0, 0), make_uint2(0, 0)};
#pragma unroll
    for (int gl = 0; gl < 2; ++gl) {
      const int g = 2 * (cc & 3) + gl;
      wp[gl] = dst + tile * F::kTile + F::kVCode + 512 * (cc >> 3) + 16 * (4 * g + t) + 8 * (q & 1);
      if (any_keep) old[gl] = *reinterpret_cast<const uint2*>(wp[gl]);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int row = 16 * tile + 2 * t + 8 * b + c;
        if (sm.keep[row]) {
          const uint32_t mm = 0xFFu << (4 * (2 * b + 4 * c));  // nibbles a + 2b + 4c, a = 0, 1
#pragma unroll
          for (int gl = 0; gl < 2; ++gl) {
            w[gl][0] |= old[gl].x & mm;
            w[gl][1] |= old[gl].y & mm;
          }
          continue;
        }
        float e[8];
        unpack8(*reinterpret_cast<const uint4*>(&sm.x[1][row][8 * cc]), e);
        const float z = sm.z[1][row][q], r = sm.r[1][row][q], sc = sm.s[1][row][q];
#pragma unroll
        for (int gl = 0; gl < 2; ++gl)
#pragma unroll
          for (int ss = 0; ss < 2; ++ss)
#pragma unroll
            for (int a = 0; a < 2; ++a)
              w[gl][ss] |= code_of(e[4 * gl + 2 * ss + a], z, r, sc) << (4 * (a + 2 * b + 4 * c));
      }
#pragma unroll
    for (int gl = 0; gl < 2; ++gl) *reinterpret_cast<uint2*>(wp[gl]) = make_uint2(w[gl][0], w[gl][1]);
  }
}

// The 4-bit stream holds every position that has left the BF16 tail, at
// row = position; a vertical-line position keeps its codes but its four key
// steps hold FP16 NaN, which the decode kernel reads as "skip this row".
// A rebuild therefore quantises only the positions [NQ, P) not in the stream
// yet, and moves the NaN marks from the old vertical-line set to the new one.

// Rebuild, step 1: quantise stream rows [NQ, P) from the BF16 source (rows
// already in the stream are kept: their positions and codes do not change).
// Block-row loop over the 64-row blocks from NQ / 64.  grid (n, HKV, B)
template <int BK, int BV>
__global__ void __launch_bounds__(kThreads) rebuild_rows_kernel(
    const __nv_bfloat16* __restrict__ k_src, const __nv_bfloat16* __restrict__ v_src, int32_t ld, int32_t P,
    hyq_layout lay, int32_t nblk_cap) {
  __shared__ __align__(16) BuildSmem sm;
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t nq_cnt = lay.counts[(size_t)b * HYQ_COUNTS + HYQ_CNT_NQ];
  const int32_t nq0 = min(max(nq_cnt, 0), P);
  const int32_t nblocks = (P + kRows - 1) / kRows - nq0 / kRows;
  for (int32_t i = blockIdx.x; i < nblocks; i += gridDim.x) {
    // append_body handles block nq0 / 64 + blockIdx.x; shift the source so
    // that its row (r - nq0) is position r
    BuildSmem& s2 = sm;
    const int32_t bi = nq0 / kRows + i;
    if (threadIdx.x < kRows) {
      const int32_t row = bi * kRows + threadIdx.x;
      s2.keep[threadIdx.x] = row < nq0;
      s2.pos[threadIdx.x] = (row >= nq0 && row < P) ? row - nq0 : -1;
    }
    __syncthreads();
    build_block<BK, BV>(s2, k_src + (bh * ld + nq0) * HYQ_D, v_src + (bh * ld + nq0) * HYQ_D,
                        lay.qblocks + (bh * nblk_cap + bi) * (size_t)QFmt<BK, BV>::kBlock, bi * kRows < nq0, lay.err);
    __syncthreads();
  }
}

// Rebuild, step 2: NaN key steps for the new vertical-line positions; the
// true steps (recomputed from the BF16 key row, as step 1 computes them) for
// positions of the old set that left it and stay in the stream.  grid
// (kMarkChunks, HKV, B): block c takes the c-th share of the old and of the
// new list; it reads the old set and counts before step 3 replaces them.
// The new list is staged in shared memory (dynamic, k ints; a list too long
// for it is searched in global memory).
constexpr int kMarkChunks = 8;
constexpr int kMarkSmemInts = 11776;  // 46 KB: with the static arrays under the 48 KB default

template <int BK, int BV>
__global__ void __launch_bounds__(kThreads) rebuild_marks_kernel(
    const __nv_bfloat16* __restrict__ k_src, int32_t ld, int32_t P, const int32_t* __restrict__ idx, int32_t k,
    hyq_layout lay, int32_t cap_vl, int32_t nblk_cap) {
  using F = QFmt<BK, BV>;
  extern __shared__ int32_t s_new[];
  __shared__ int32_t s_leave[kThreads];
  __shared__ int s_nleave;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  const int32_t nq_old = min(max(cnt[HYQ_CNT_NQ], 0), P), nvl_old = min(max(cnt[HYQ_CNT_NVL], 0), cap_vl);
  const int32_t* inew = idx + bh * k;
  const int32_t* iold = lay.vl_idx + bh * cap_vl;
  uint8_t* stream = lay.qblocks + bh * (size_t)nblk_cap * F::kBlock;
  auto kmeta = [&](int32_t pos) {  // the four key steps of stream row pos
    return reinterpret_cast<__half*>(stream + (pos >> 4) * F::kTile + F::kKMeta + 16 * (pos & 15));
  };
  const bool staged = k <= kMarkSmemInts;
  if (staged)
    for (int32_t i = threadIdx.x; i < k; i += kThreads) s_new[i] = __ldg(inew + i);
  if (threadIdx.x == 0) s_nleave = 0;
  __syncthreads();
  const int32_t* list = staged ? s_new : inew;
  // this block's old entries, one per thread per pass: leaving the set?
  const int32_t o0 = (int32_t)((int64_t)nvl_old * c / kMarkChunks), o1 = (int32_t)((int64_t)nvl_old * (c + 1) / kMarkChunks);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float qmax = BK == 8 ? 255.f : 15.f;
  for (int32_t base = o0; base < o1; base += kThreads) {
    const int32_t i = base + threadIdx.x;
    if (i < o1) {
      const int32_t pos = __ldg(iold + i);
      int32_t lo = 0, hi = k;
      while (lo < hi) {
        const int32_t m = (lo + hi) >> 1;
        if (list[m] < pos) lo = m + 1;
        else hi = m;
      }
      if (pos >= 0 && pos < nq_old && !(lo < k && list[lo] == pos)) s_leave[atomicAdd(&s_nleave, 1)] = pos;
    }
    __syncthreads();
    // restore the leaving rows: a warp per row, four rows' loads in flight per warp
    const int nl = s_nleave;
    for (int r0 = 4 * warp; r0 < nl; r0 += 4 * kWarps) {
      uint2 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = r0 + u < nl ? __ldg(reinterpret_cast<const uint2*>(k_src + (bh * ld + s_leave[r0 + u]) * HYQ_D) + lane)
                           : make_uint2(0, 0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // lane: elements 4 lane .. 4 lane + 3 of the key row; group lane / 8
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
        __nv_bfloat162 mn2 = __hmin2_nan(p2[0], p2[1]), mx2 = __hmax2_nan(p2[0], p2[1]);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          mn2 = __hmin2_nan(mn2, __shfl_xor_sync(0xffffffffu, mn2, o));
          mx2 = __hmax2_nan(mx2, __shfl_xor_sync(0xffffffffu, mx2, o));
        }
        if ((lane & 7) == 0 && r0 + u < nl) {
          const float2 fm = __bfloat1622float2(mn2), fx = __bfloat1622float2(mx2);
          __half sh = group_step(fminf(fm.x, fm.y), fmaxf(fx.x, fx.y), qmax);
          if (isinf(__half2float(sh)) || isnan(fm.x) || isnan(fm.y)) sh = __float2half_rn(0.f);  // as step 1 stores it
          kmeta(s_leave[r0 + u])[lane >> 3] = sh;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) s_nleave = 0;
    __syncthreads();
  }
  // this block's share of the new set: NaN steps
  const __half nanh = __ushort_as_half((unsigned short)0x7E00);
  const int32_t n0 = (int32_t)((int64_t)k * c / kMarkChunks), n1 = (int32_t)((int64_t)k * (c + 1) / kMarkChunks);
  for (int32_t i = n0 + threadIdx.x; i < n1; i += kThreads) {
    const int32_t pos = list[i];
    if (pos >= 0 && pos < P) {
      __half* m = kmeta(pos);
      m[0] = m[1] = m[2] = m[3] = nanh;
    }
  }
}

// Vertical-line gather, BF16 tail copy and counters.  One warp per row:
// lanes 0-15 copy the K row, lanes 16-31 the V row.  grid (ceil((k+ntail)/8), HKV, B)
__global__ void __launch_bounds__(kThreads) rebuild_gather_kernel(
    const __nv_bfloat16* __restrict__ k_src, const __nv_bfloat16* __restrict__ v_src, int32_t ld,
    int32_t L, int32_t P, const int32_t* __restrict__ idx, int32_t k, hyq_layout lay,
    int32_t cap_vl, int32_t cap_tail) {
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t ntail = L - P;
  const int32_t row = blockIdx.x * kWarps + warp;
  if (row < k + ntail) {
    int32_t src;
    uint4* dk;
    uint4* dv;
    if (row < k) {
      src = idx[bh * k + row];
      bool ok = src >= 0 && src < P && (row == 0 || idx[bh * k + row - 1] < src);
      if (!ok) {
        if (lane == 0) hyq_set_err(lay.err, HYQ_DEVERR_INDEX);
        src = min(max(src, 0), max(P - 1, 0));
      }
      dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.vl_k) + (bh * cap_vl + row) * HYQ_D);
      dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.vl_v) + (bh * cap_vl + row) * HYQ_D);
      if (lane == 0) lay.vl_idx[bh * cap_vl + row] = src;
    } else {
      int32_t t = row - k;
      src = P + t;
      dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_k) + (bh * cap_tail + t) * HYQ_D);
      dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_v) + (bh * cap_tail + t) * HYQ_D);
    }
    const uint4* s = reinterpret_cast<const uint4*>((lane < 16 ? k_src : v_src) + (bh * ld + src) * HYQ_D);
    (lane < 16 ? dk : dv)[lane & 15] = s[lane & 15];
  }
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {
    int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
    cnt[HYQ_CNT_NQ] = P;
    cnt[HYQ_CNT_NVL] = k;
    cnt[HYQ_CNT_NTAIL] = ntail;
    cnt[HYQ_CNT_LEN] = L;
  }
}

// Block blockIdx.x of appending rows [0, end - nq0) of kbase / vbase (row r
// at kbase + r * 128) to the quantised stream of (b, h) after its nq0 rows.
template <int BK, int BV>
__device__ void append_body(BuildSmem& sm, const __nv_bfloat16* kbase, const __nv_bfloat16* vbase, int32_t nq0,
                            int32_t end, size_t bh, const hyq_layout& lay, int32_t nblk_cap) {
  const int32_t bi = nq0 / kRows + blockIdx.x;
  if (max(bi * kRows, nq0) >= min((bi + 1) * kRows, end)) return;  // uniform across the block
  if (threadIdx.x < kRows) {
    const int32_t row = bi * kRows + threadIdx.x;
    sm.keep[threadIdx.x] = row < nq0;
    sm.pos[threadIdx.x] = (row >= nq0 && row < end) ? row - nq0 : -1;
  }
  __syncthreads();
  build_block<BK, BV>(sm, kbase, vbase, lay.qblocks + (bh * nblk_cap + bi) * (size_t)QFmt<BK, BV>::kBlock,
                      bi * kRows < nq0, lay.err);
}

// Append n rows per (b, h) after the current NQ rows.  grid (blocks touched, HKV, B)
template <int BK, int BV>
__global__ void __launch_bounds__(kThreads) append_blocks_kernel(
    const __nv_bfloat16* __restrict__ k_rows, const __nv_bfloat16* __restrict__ v_rows, int32_t n,
    hyq_layout lay, int32_t nblk_cap) {
  __shared__ __align__(16) BuildSmem sm;
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t nq0 = lay.counts[(size_t)b * HYQ_COUNTS + HYQ_CNT_NQ];
  const int32_t cap_rows = nblk_cap * kRows;
  if (nq0 < 0 || nq0 > cap_rows) {
    if (threadIdx.x == 0) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
    return;
  }
  const int32_t end = min(nq0 + n, cap_rows);
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0 && nq0 + n > cap_rows)
    hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
  append_body<BK, BV>(sm, k_rows + bh * n * HYQ_D, v_rows + bh * n * HYQ_D, nq0, end, bh, lay, nblk_cap);
}

// Rows the tail of sequence b gives up in hyq_age_tail: max(0, NTAIL - W),
// or 0 (and the layout left unchanged) when the counters are out of range or
// the stream has no room for them.
__device__ __forceinline__ int32_t age_rows(const hyq_layout& lay, int b, int32_t window, int32_t cap_rows,
                                            int32_t cap_tail) {
  const int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  const int32_t nq = cnt[HYQ_CNT_NQ], ntail = cnt[HYQ_CNT_NTAIL];
  if (nq < 0 || nq > cap_rows || ntail < 0 || ntail > cap_tail) return 0;
  const int32_t m = max(0, ntail - window);
  return nq + m <= cap_rows ? m : 0;
}

// hyq_age_tail, step 1: the oldest m tail rows of (b, h) onto the 4-bit
// stream.  grid (blocks touched, HKV, B)
template <int BK, int BV>
__global__ void __launch_bounds__(kThreads) age_blocks_kernel(hyq_layout lay, int32_t nblk_cap, int32_t window,
                                                              int32_t cap_tail) {
  __shared__ __align__(16) BuildSmem sm;
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t m = age_rows(lay, b, window, nblk_cap * kRows, cap_tail);
  if (m == 0) return;
  const int32_t nq0 = lay.counts[(size_t)b * HYQ_COUNTS + HYQ_CNT_NQ];
  append_body<BK, BV>(sm, static_cast<const __nv_bfloat16*>(lay.tail_k) + bh * cap_tail * HYQ_D,
              static_cast<const __nv_bfloat16*>(lay.tail_v) + bh * cap_tail * HYQ_D, nq0, nq0 + m, bh, lay,
              nblk_cap);
}

// hyq_age_tail, step 2: tail rows [m, NTAIL) of (b, h) move to [0, NTAIL - m).
// The destination lies below the source, so chunks taken in ascending order,
// each read whole before any of it is written, never overwrite a row still
// to be read.  grid (HKV, B)
__global__ void __launch_bounds__(kThreads) age_shift_kernel(hyq_layout lay, int32_t nblk_cap, int32_t window,
                                                             int32_t cap_tail) {
  const int h = blockIdx.x, b = blockIdx.y, HKV = gridDim.x;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t m = age_rows(lay, b, window, nblk_cap * kRows, cap_tail);
  if (m == 0) return;
  const int32_t keep = lay.counts[(size_t)b * HYQ_COUNTS + HYQ_CNT_NTAIL] - m;
  uint4* tk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_k) + bh * cap_tail * HYQ_D);
  uint4* tv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lay.tail_v) + bh * cap_tail * HYQ_D);
  constexpr int kChunkRows = kThreads / kChunks;  // 16 uint4 per row
  for (int r0 = 0; r0 < keep; r0 += kChunkRows) {
    const int r = r0 + threadIdx.x / kChunks, c = threadIdx.x % kChunks;
    uint4 a = make_uint4(0, 0, 0, 0), bv = a;
    if (r < keep) {
      a = tk[(size_t)(m + r) * kChunks + c];
      bv = tv[(size_t)(m + r) * kChunks + c];
    }
    __syncthreads();
    if (r < keep) {
      tk[(size_t)r * kChunks + c] = a;
      tv[(size_t)r * kChunks + c] = bv;
    }
    __syncthreads();
  }
}

// hyq_age_tail, step 3: NQ += m, NTAIL -= m (LEN unchanged).  grid (B)
__global__ void age_counts_kernel(hyq_layout lay, int32_t nblk_cap, int32_t window, int32_t cap_tail) {
  const int b = blockIdx.x;
  int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  const int32_t nq = cnt[HYQ_CNT_NQ], ntail = cnt[HYQ_CNT_NTAIL];
  const int32_t m = age_rows(lay, b, window, nblk_cap * kRows, cap_tail);
  if (m == 0) {
    const bool bad = nq < 0 || nq > nblk_cap * kRows || ntail < 0 || ntail > cap_tail ||
                     (ntail > window && nq + (ntail - window) > nblk_cap * kRows);
    if (bad) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
    return;
  }
  cnt[HYQ_CNT_NQ] = nq + m;
  cnt[HYQ_CNT_NTAIL] = ntail - m;
}

__global__ void append_counts_kernel(hyq_layout lay, int32_t n, int32_t cap_rows) {
  const int b = blockIdx.x;
  int32_t* cnt = lay.counts + (size_t)b * HYQ_COUNTS;
  int32_t nq0 = cnt[HYQ_CNT_NQ];
  if (nq0 < 0 || nq0 > cap_rows) return;
  int32_t add = min(n, cap_rows - nq0);
  cnt[HYQ_CNT_NQ] = nq0 + add;
  cnt[HYQ_CNT_LEN] += add;
}

// Calls f(std::integral_constant<int, BK>, std::integral_constant<int, BV>)
// for the config's code widths.
template <class Fn>
auto with_widths(const hyq_config* c, Fn f) {
  const int bk = hyq_bits_k(c), bv = hyq_bits_v(c);
  using I4 = std::integral_constant<int, 4>;
  using I8 = std::integral_constant<int, 8>;
  if (bk == 8) return bv == 8 ? f(I8{}, I8{}) : f(I8{}, I4{});
  return bv == 8 ? f(I4{}, I8{}) : f(I4{}, I4{});
}

}  // namespace

cudaError_t hyq_launch_age_tail(const hyq_config* c, const hyq_layout* lay, cudaStream_t s) {
  const int32_t nblk = hyq_nblk(c), ct = hyq_cap_tail(c);
  // at most cap_tail - W = period rows leave: that many 64-row blocks plus one
  const int32_t most = ct - c->window;
  if (most <= 0) return cudaSuccess;
  dim3 grid((most + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS + 1, c->num_kv_heads, c->batch);
  with_widths(c, [&](auto bk, auto bv) {
    age_blocks_kernel<bk.value, bv.value><<<grid, kThreads, 0, s>>>(*lay, nblk, c->window, ct);
    return 0;
  });
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  age_shift_kernel<<<dim3(c->num_kv_heads, c->batch), kThreads, 0, s>>>(*lay, nblk, c->window, ct);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  age_counts_kernel<<<c->batch, 1, 0, s>>>(*lay, nblk, c->window, ct);
  return cudaGetLastError();
}

cudaError_t hyq_launch_quantize_append(const hyq_config* c, const void* k, const void* v,
                                       int32_t n_rows, const hyq_layout* lay, cudaStream_t s) {
  int32_t nblk = hyq_nblk(c);
  dim3 grid((n_rows + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS + 1, c->num_kv_heads, c->batch);
  with_widths(c, [&](auto bk, auto bv) {
    append_blocks_kernel<bk.value, bv.value><<<grid, kThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), n_rows, *lay, nblk);
    return 0;
  });
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  append_counts_kernel<<<c->batch, 1, 0, s>>>(*lay, n_rows, nblk * HYQ_QBLOCK_ROWS);
  return cudaGetLastError();
}

cudaError_t hyq_launch_rebuild(const hyq_config* c, const void* k_src, const void* v_src,
                               int32_t ld, int32_t L, const int32_t* idx, int32_t k,
                               const hyq_layout* lay, cudaStream_t s) {
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  int32_t nblk = hyq_nblk(c);
  const __nv_bfloat16* kk = static_cast<const __nv_bfloat16*>(k_src);
  const __nv_bfloat16* vv = static_cast<const __nv_bfloat16*>(v_src);
  if (P > 0) {
    // the rows still to quantise are unknown here (the stream length is on the
    // device): a few blocks per (b, KV head) loop over them; a first rebuild
    // of a long context gets more
    const int32_t blocks = (P + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS;
    dim3 grid(blocks < 8 ? blocks : (blocks / 8 < 8 ? 8 : blocks / 8), c->num_kv_heads, c->batch);
    with_widths(c, [&](auto bk, auto bv) {
      rebuild_rows_kernel<bk.value, bv.value><<<grid, kThreads, 0, s>>>(kk, vv, ld, P, *lay, nblk);
      const size_t smem = k <= kMarkSmemInts ? (size_t)k * sizeof(int32_t) : 0;
      rebuild_marks_kernel<bk.value, bv.value><<<dim3(kMarkChunks, c->num_kv_heads, c->batch), kThreads, smem, s>>>(
          kk, ld, P, idx, k, *lay, hyq_vl_stride(c), nblk);
      return 0;
    });
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int32_t rows = k + (L - P);
  dim3 grid2(rows > 0 ? (rows + kWarps - 1) / kWarps : 1, c->num_kv_heads, c->batch);
  rebuild_gather_kernel<<<grid2, kThreads, 0, s>>>(kk, vv, ld, L, P, idx, k, *lay, hyq_vl_stride(c),
                                                   hyq_cap_tail(c));
  return cudaGetLastError();
}
