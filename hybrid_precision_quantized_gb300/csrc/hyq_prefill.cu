// Hybrid-precision prefill attention on the 5th-generation tensor cores.
//
// "HyQuant: Hybrid-Precision Quantization for LLM Attention", §4.2 Eq. 6-7
// and Appendix A.2, Algorithm 2:
//   O = softmax(a Q^ K^_Q^T || a Q K_FP^T) (V^_Q || V_FP),   a = 1/sqrt(d),
// causal.  K_FP/V_FP are the vertical-line keys and the last W keys, kept in
// BF16; K_Q/V_Q are the remaining prefix positions, quantised per tile of 64
// keys (taken in ascending position) with one symmetric scale per tile and
// tensor; Q is quantised with one scale per 128-row block of one head.
//
// Two launches:
//  1. pack_kernel (Algorithm 2 stages 1-2): the reordered key lists, their
//     per-tile scales and codes, written straight into the shared-memory
//     image the tensor cores read (128-byte swizzled K-major tiles), so the
//     main kernel moves each 128-key tile with one bulk copy.  Values are
//     stored transposed (dims x keys) for the P.V product.
//  2. prefill_kernel (stage 3): one CTA per (query block of 128 rows, query
//     head).  Warps 8 and 9 stream key and value tiles (bulk copies, one
//     ring each); warp 10 issues tcgen05.mma S = Q K^T into TMEM and warp 11
//     O_h += P_h V_h into TMEM for the two 64-key halves h of each tile;
//     warps 0-7 (one thread per query row = TMEM lane and key half) read S,
//     scale, mask, run an online softmax per half and write P as BF16 into
//     one of two TMEM buffers, where the P.V MMA takes its A operand; a
//     barrier per P buffer signals both halves' P of a tile and a commit per
//     buffer their P.V (so the softmax waits for the P.V two tiles back, the
//     last reader of the buffer, unless it rescales O), and the two halves'
//     (max, sum, O) merge once at the end.  The MMA threads
//     share schedulers with softmax warps, so their loops are kept to a few
//     instructions, and the two products are issued from two threads so
//     that neither's waits hold back the other.  The quantised segment uses e4m3 codes or e2m1 (FP4)
//     codes (kind::f8f6f4; an e2m1 operand row keeps 16 elements in each
//     16-byte chunk, packed in its first 8 bytes with element 2i in the low
//     nibble of byte i, the other 8 bytes unread, so that an MMA takes 32
//     elements from 32 bytes as with e4m3) or INT8 codes held exactly as
//     BF16 integers (kind::f16; sm_103a has no integer tensor-core MMA); the
//     full-precision segment uses BF16.  P.V runs in
//     BF16 with the value codes (exact in BF16) and the value scale folded
//     into P.
//
// Every wait is bounded; on expiry the kernel sets HYQ_DEVERR_TIMEOUT, drains
// its own copies and MMAs, frees its TMEM and returns.
#include <cuda_fp8.h>

#include <cmath>
#include <cstdint>

#include "hyq_f2.cuh"
#include "hyq_tc.cuh"

namespace {

constexpr int kRows = 128;           // query rows per CTA (MMA M)
constexpr int kKeys = 128;           // keys per MMA tile
constexpr int kScaleTile = 64;       // keys per quantisation scale (B_N)
constexpr int kRegion = 16384;       // 128 rows x 128 bytes, swizzled
constexpr int kImg16 = 2 * kRegion;  // 128 x 128 16-bit operand image
constexpr int kImg8 = kRegion;       // 128 x 128 8-bit operand image
constexpr int kSoft = 256;           // softmax threads (warps 0-7)
constexpr int kCopyWarp = 8;  // copy warps 8 (keys) and 9 (values)
constexpr int kMmaWarp = 10;  // issues S = Q K^T (and allocates TMEM)
constexpr int kPvWarp = 11;   // issues O += P V
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S (one 128-key tile, FP32), P (two tiles in flight, BF16
// pairs: 64 columns per tile, 32 per key half), one O accumulator per key half.
constexpr uint32_t kColS = 0, kColP = 128, kColO0 = 256, kColO1 = 384;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int kOffQ = 0;                   // Q, BF16 image
constexpr int kOffQc = kOffQ + kImg16;     // Q codes image (8- or 16-bit)
constexpr int kOffK = kOffQc + kImg16;     // key stages
#ifndef HYQ_PREFILL_KSTAGES
#define HYQ_PREFILL_KSTAGES 3
#endif
constexpr int kKStages = HYQ_PREFILL_KSTAGES, kVStages = 5 - HYQ_PREFILL_KSTAGES;
constexpr int kOffV = kOffK + kKStages * kImg16;  // value stages (transposed)
constexpr int kOffBar = kOffV + kVStages * kImg16;
constexpr int kNumBars = 24;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 64;
constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base

constexpr uint32_t kIdescBF16 = tc_idesc(kTcBF16, kTcBF16, kRows, kKeys);
constexpr uint32_t kIdescE4M3 = tc_idesc(kTcE4M3, kTcE4M3, kRows, kKeys);
constexpr uint32_t kTcE2M1 = 5;  // kind::f8f6f4 operand format e2m1
constexpr uint32_t kIdescE2M1 = tc_idesc(kTcE2M1, kTcE2M1, kRows, kKeys);

// Code types of the quantised segment (the HYQ_PREFILL_* values).
constexpr int kDtInt8 = HYQ_PREFILL_INT8, kDtFp8 = HYQ_PREFILL_FP8, kDtFp4 = HYQ_PREFILL_FP4;
// c_B: the largest code magnitude.
__host__ __device__ constexpr float code_max(int dt) { return dt == kDtFp8 ? 448.f : dt == kDtFp4 ? 6.f : 127.f; }

struct PackParams {
  const __nv_bfloat16* k;  // [B][HKV][ldk][128]
  const __nv_bfloat16* v;
  int64_t ldk;
  const int32_t* vl;  // [B][HKV][kvl]
  int32_t kvl;
  uint8_t* kq;  // [B][HKV][ntq] key code images
  uint8_t* vq;  // [B][HKV][ntq] value code images (BF16, transposed)
  uint8_t* kf;  // [B][HKV][ntf] BF16 key images
  uint8_t* vf;  // [B][HKV][ntf] BF16 value images (transposed)
  uint8_t* kb;  // [B][HKV][ntb] per-query band: BF16 key images of positions 128t .. 128t+127
  uint8_t* vb;  // [B][HKV][ntb] the same for values (transposed)
  int32_t* kpos;
  int32_t* fpos;
  float* sk;
  float* sv;
  int32_t* err;
  int32_t L, P, HKV, nq, nfp, ntq, ntf, ntb;
};

struct MainParams {
  const __nv_bfloat16* q;  // [B][HQ][ldq][128]
  __nv_bfloat16* out;      // [B][HQ][L][128]
  const uint8_t* kq;
  const uint8_t* vq;
  const uint8_t* kf;
  const uint8_t* vf;
  const uint8_t* kb;    // per-query band images (band mode)
  const uint8_t* vb;
  const int32_t* kpos;  // [B][HKV][ntq*128], ascending, padding INT32_MAX
  const int32_t* fpos;  // [B][HKV][ntf*128]
  const float* sk;      // [B][HKV][ntq*2]
  const float* sv;
  int32_t* err;
  int64_t ldq;
  int32_t L, HQ, HKV, ntq, ntf, ntb, W;
  float alpha_log2e;
};

// Byte offset of the 16-byte chunk `c` (of the 128-byte row `r`) in a
// 128-byte-swizzled region.
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ float bf16_at(const uint4& u, int e) {
  const uint32_t w = (&u.x)[e >> 1];
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// Codes of the exact quotient x / s (x a BF16 value, s > 0 the FP32 scale, or
// s = 0 for an all-zero tile).  t = fl32(x / s) is correctly rounded and
// monotone in x / s, so rounding t to the code grid gives the code of x / s
// except when t itself is a midpoint of that grid; then the sign of x - t s
// decides (an exact tie keeps the even code).  One fused multiply-add gives
// it: t s is formed exactly (t has at most 9 significant bits, s 24) and the
// difference is rounded once, which keeps its sign (scales below the FP32
// normal range, tiles whose maximum is under c_B 2^-126, aside).
__device__ __forceinline__ float quotient(float x, float s) { return s > 0.f ? __fdiv_rn(x, s) : 0.f; }

__device__ __forceinline__ float past_midpoint(float x, float s, float t, float below, float above, float even) {
  const float d = fmaf(-t, s, x);
  return d > 0.f ? above : d < 0.f ? below : even;
}

// INT8: the nearest integer to x / s, ties to even, clamped to +-127.
__device__ __forceinline__ float code_i8(float x, float s) {
  const float t = quotient(x, s);
  float c = rintf(t);
  const float f = floorf(t);
  if (t - f == 0.5f && fabsf(t) < 128.f) c = past_midpoint(x, s, t, f, f + 1.f, c);
  return fminf(fmaxf(c, -127.f), 127.f);
}

// e4m3: the value nearest to x / s, ties to even, saturating at +-448.  Its
// midpoints are the odd multiples of 2^-10 below 2^-6 and, above, the values
// whose FP32 fraction ends in binary 1 followed by 19 zeros; h is half the
// e4m3 spacing there.
__device__ __forceinline__ float code_f8(float x, float s) {
  const float t = quotient(x, s);
  const float c = static_cast<float>(__nv_fp8_e4m3(t));  // nearest even, saturating
  const float a = fabsf(t);
  if (a >= 448.f) return c;
  float h = 0.f;
  if (a < 0.015625f) {
    const float u = a * 1024.f;  // exact
    if (u == floorf(u) && (__float2int_rz(u) & 1)) h = 0.0009765625f;
  } else if ((__float_as_uint(a) & 0x000FFFFFu) == 0x00080000u) {
    h = __uint_as_float(__float_as_uint(a) & 0xFF800000u) * 0.0625f;  // 2^(E-4)
  }
  return h > 0.f ? past_midpoint(x, s, t, t - h, t + h, c) : c;
}

__device__ __forceinline__ uint8_t code_f8_bits(float x, float s) {
  return __nv_cvt_float_to_fp8(code_f8(x, s), __NV_SATFINITE, __NV_E4M3);  // exact: an e4m3 value
}

// INT8 fast path with r = RN(1/s): t = fl32(x r) lies within 2^-23 |x / s|
// of the exact quotient, under 2^-16 for |t| < 2^8, so rounding t gives the
// code of x / s unless its fractional part is within 2^-15 of 1/2; those
// elements take the exact path above.  (The same gate for e4m3, around the
// fraction pattern of its midpoints, measured no faster and is not used.)
__device__ __forceinline__ float recip(float s) { return s > 0.f ? __frcp_rn(s) : 0.f; }

__device__ __forceinline__ float code_i8_fast(float x, float s, float r) {
  const float t = x * r;
  if (s > 0.f && fabsf(t - floorf(t) - 0.5f) > 3.0517578125e-05f) return fminf(fmaxf(rintf(t), -127.f), 127.f);
  return code_i8(x, s);
}


// e2m1 (FP4): the value nearest to x / s among 0, 0.5, 1, 1.5, 2, 3, 4, 6
// and their negatives, ties to the even code (the value with a zero fraction
// bit), saturating at +-6.  The magnitude code is the number of midpoints
// m_k = 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 that |x| / s passes: |x| - m_k s
// is formed by one fused multiply-add from the exact product m_k s (m_k has
// at most three significant bits), so its sign is exact, and at a tie
// (zero) the code moves past m_k only toward an even code (odd k).  No
// quotient is rounded on the way.  s = 0 (an all-zero tile) gives 0.
__device__ __forceinline__ uint32_t e2m1_code(float x, float s) {
  const float a = fabsf(x);
  constexpr float kMid[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.f};
  uint32_t m = 0;
#pragma unroll
  for (int k = 0; k < 7; ++k) {
    const float d = fmaf(-kMid[k], s, a);
    m += (d > 0.f || (d == 0.f && (k & 1))) ? 1u : 0u;
  }
  if (!(s > 0.f)) m = 0;
  return (x < 0.f && m != 0 ? 8u : 0u) | m;
}

// The e2m1 value of a 4-bit pattern (sign, two exponent bits, one fraction bit).
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;
  const float v = m < 4u ? 0.5f * static_cast<float>(m) : static_cast<float>(1u << ((m >> 1) - 1u)) * (m & 1u ? 1.5f : 1.f);
  return c & 8u ? -v : v;
}

__device__ __forceinline__ float code_f4(float x, float s) { return e2m1_value(e2m1_code(x, s)); }

// Sixteen consecutive elements x[0..15] (BF16 in two uint4) as the 16-byte
// operand chunk of e2m1 codes: 8 bytes, element 2i in the low nibble of
// byte i, then 8 bytes the tensor core does not read (zeros).
__device__ __forceinline__ uint4 pack_f4x16(const uint4& lo, const uint4& hi, float s) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e) w[e >> 3] |= e2m1_code(bf16_at(e < 8 ? lo : hi, e & 7), s) << (4 * (e & 7));
  return make_uint4(w[0], w[1], 0u, 0u);
}

// Number of entries <= x in the ascending array a[0..n).
__device__ __forceinline__ int count_le(const int32_t* a, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) <= x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Warp-cooperative count of the entries <= x in the ascending a[0..n): 32
// probes per round, so a 32K-entry list takes 3-4 dependent loads.
__device__ __forceinline__ int warp_count_le(const int32_t* a, int n, int32_t x, int lane) {
  int lo = 0, hi = n;  // invariant: a[i] <= x for i < lo, a[i] > x for i >= hi
  while (lo < hi) {
    const int step = (hi - lo + 31) >> 5;
    const int idx = lo + lane * step;
    const bool le = idx < hi && __ldg(a + idx) <= x;
    const int cnt = __popc(__ballot_sync(0xffffffffu, le));
    if (cnt == 0) {
      hi = lo;
    } else {
      const int nlo = lo + (cnt - 1) * step + 1;
      hi = min(hi, lo + cnt * step);
      lo = nlo;
    }
  }
  return lo;
}

// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float block_max(float v, float* red, int nwarps) {
  v = warp_max_xor(v, 1);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float m = red[0];
  for (int i = 1; i < nwarps; ++i) m = fmaxf(m, red[i]);
  return m;
}

// ---------------------------------------------------------------------------
// Stage 1-2: key lists, scales, code images.  Grid (2 ntq + 2 ntf + 2 ntb,
// HKV, B); each block handles one 64-key scale tile of one list: the
// quantised prefix, the full-precision list, or (per-query band, ntb > 0)
// the BF16 images of all positions in order.
// ---------------------------------------------------------------------------
template <int kDt>
__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackParams p) {
  __shared__ float vs[kScaleTile][HYQ_D + 1];
  __shared__ int32_t spos[kScaleTile];
  __shared__ float red[8];
  const int tid = threadIdx.x;
  const int kh = blockIdx.y, b = blockIdx.z;
  const size_t bh = (size_t)b * p.HKV + kh;
  const int nq2 = 2 * p.ntq, nf2 = 2 * p.ntf;
  const int seg = blockIdx.x < nq2 ? 0 : (blockIdx.x < nq2 + nf2 ? 1 : 2);  // quantised, full, band
  const bool quant = seg == 0;
  const int t64 = blockIdx.x - (seg == 0 ? 0 : (seg == 1 ? nq2 : nq2 + nf2));
  const int n = seg == 0 ? p.nq : (seg == 1 ? p.nfp : p.L);
  const int32_t* vl = p.vl + bh * p.kvl;

  if (tid < kScaleTile) {
    const int i = t64 * kScaleTile + tid;
    int32_t pos = INT32_MAX;
    if (i < n) {
      if (quant) {
        // i-th position of [0, P) that is not a vertical line
        int lo = i, hi = min(p.P - 1, i + p.kvl);
        while (lo < hi) {
          int mid = (lo + hi) >> 1;
          int c = mid + 1 - count_le(vl, p.kvl, mid);
          if (c >= i + 1) hi = mid;
          else lo = mid + 1;
        }
        pos = lo;
      } else if (seg == 2) {
        pos = i;
      } else {
        if (i < p.kvl) {
          pos = __ldg(vl + i);
          if (pos < 0 || pos >= p.P || (i > 0 && __ldg(vl + i - 1) >= pos)) {
            hyq_set_err(p.err, HYQ_DEVERR_INDEX);
            pos = min(max(pos, 0), p.L - 1);
          }
        } else {
          pos = p.P + (i - p.kvl);
        }
      }
    }
    spos[tid] = pos;
    if (seg == 0) p.kpos[bh * p.ntq * kKeys + i] = pos;
    else if (seg == 1) p.fpos[bh * p.ntf * kKeys + i] = pos;
  }
  __syncthreads();

  // Each thread: 32 elements (quarter qq) of row r of K and of V.
  const int r = tid >> 2, qq = tid & 3;
  const int32_t pos = spos[r];
  const bool valid = pos != INT32_MAX;
  uint4 kr[4], vr[4];
  if (valid) {
    const uint4* ks = reinterpret_cast<const uint4*>(p.k + (bh * p.ldk + pos) * HYQ_D + 32 * qq);
    const uint4* vv = reinterpret_cast<const uint4*>(p.v + (bh * p.ldk + pos) * HYQ_D + 32 * qq);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      kr[c] = __ldg(ks + c);
      vr[c] = __ldg(vv + c);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) kr[c] = vr[c] = make_uint4(0, 0, 0, 0);
  }

  const int key = (t64 & 1) * kScaleTile + r;  // row of the 128-key MMA tile
  const int tile = t64 >> 1;
  float sk = 1.f, sv = 1.f, rk = 1.f, rv = 1.f;
  if (quant) {
    float ak = 0.f, av = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      ak = fmaxf(ak, fabsf(bf16_at(kr[e >> 3], e & 7)));
      av = fmaxf(av, fabsf(bf16_at(vr[e >> 3], e & 7)));
    }
    const float cb = code_max(kDt);
    ak = block_max(ak, red, 8);
    av = block_max(av, red, 8);
    sk = __fdiv_rn(ak, cb);
    sv = __fdiv_rn(av, cb);
    rk = recip(sk);
    rv = recip(sv);
    if (tid == 0) {
      p.sk[bh * p.ntq * 2 + t64] = sk;
      p.sv[bh * p.ntq * 2 + t64] = sv;
    }
  }

  // Key image.
  if (quant && kDt == kDtFp4) {
    // dims 32qq .. 32qq+31: chunks 2qq and 2qq+1 of the row
    uint8_t* img = p.kq + (bh * p.ntq + tile) * (size_t)kImg8;
    *reinterpret_cast<uint4*>(img + swz(key, 2 * qq)) = pack_f4x16(kr[0], kr[1], sk);
    *reinterpret_cast<uint4*>(img + swz(key, 2 * qq + 1)) = pack_f4x16(kr[2], kr[3], sk);
  } else if (quant && kDt == kDtFp8) {
    uint8_t* img = p.kq + (bh * p.ntq + tile) * (size_t)kImg8;
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // two 16-byte chunks of 16 codes
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t acc = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int el = 16 * h + 4 * u + e;
          const float x = bf16_at(kr[el >> 3], el & 7);
          acc |= static_cast<uint32_t>(code_f8_bits(x, sk)) << (8 * e);
        }
        w[u] = acc;
      }
      *reinterpret_cast<uint4*>(img + swz(key, 2 * qq + h)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    uint8_t* img = quant      ? p.kq + (bh * p.ntq + tile) * (size_t)kImg16
                   : seg == 1 ? p.kf + (bh * p.ntf + tile) * (size_t)kImg16
                              : p.kb + (bh * p.ntb + tile) * (size_t)kImg16;
    // dims 32qq .. 32qq+31 = bytes 64qq .. 64qq+63: region qq/2, chunks 4(qq&1)..+3
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 u = kr[c];
      if (quant) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = bf16_at(kr[c], 2 * e), x1 = bf16_at(kr[c], 2 * e + 1);
          w[e] = pack_bf16x2(code_i8_fast(x0, sk, rk), code_i8_fast(x1, sk, rk));
        }
        u = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(img + (qq >> 1) * kRegion + swz(key, 4 * (qq & 1) + c)) = u;
    }
  }

  // Value image, transposed: rows = dims, 128-byte rows hold 64 keys (BF16);
  // keys 0-63 of the MMA tile in region 0, 64-127 in region 1.
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float x = bf16_at(vr[e >> 3], e & 7);
    float y = x;
    if (quant) y = kDt == kDtFp8 ? code_f8(x, sv) : kDt == kDtFp4 ? code_f4(x, sv) : code_i8_fast(x, sv, rv);
    vs[r][32 * qq + e] = y;
  }
  __syncthreads();
  uint8_t* vimg = quant      ? p.vq + (bh * p.ntq + tile) * (size_t)kImg16
                  : seg == 1 ? p.vf + (bh * p.ntf + tile) * (size_t)kImg16
                             : p.vb + (bh * p.ntb + tile) * (size_t)kImg16;
  vimg += (t64 & 1) * kRegion;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int item = tid + 256 * it;
    const int dim = item & (HYQ_D - 1), kc = item >> 7;  // kc: 8-key chunk 0..7
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(vs[8 * kc + 2 * e][dim], vs[8 * kc + 2 * e + 1][dim]);
    *reinterpret_cast<uint4*>(vimg + swz(dim, kc)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------------------
// Stage 3: segmented online softmax on tcgen05.  Tiles in order: the
// quantised prefix, the full-precision list, and with kBand the band tiles
// (positions 128 tb0 .. 128 (tb0 + nbt) - 1).  Fixed window: every segment
// masks keys after the row (j <= i).  Per-query band: the quantised prefix
// and the vertical lines mask j <= i - W, the band tiles i - W < j <= i.
// ---------------------------------------------------------------------------
template <int kDt, bool kBand>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ MainParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* qready = bars + 0;
  uint64_t* kfull = bars + 18;  // [kKStages]
  uint64_t* kempty = bars + 21; // [kKStages]
  uint64_t* sfull = bars + 5;   // S of the current tile is in TMEM
  uint64_t* sfree = bars + 6;   // every softmax thread has read it
  uint64_t* pfull = bars + 7;   // [2]: both key halves' P of tile i written, on pfull[i % 2]
  uint64_t* pvdone = bars + 9;  // [2]: tile i's P.V done (both halves) on pvdone[i % 2]
  uint64_t* mmadone = bars + 11;
  uint64_t* vfull = bars + 12;  // [kVStages]
  uint64_t* vempty = bars + 15; // [kVStages]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);
  int* ntiles = reinterpret_cast<int*>(sm + kOffMisc + 8);     // [6]
  float* red = reinterpret_cast<float*>(sm + kOffMisc + 32);   // [8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, b = blockIdx.z;
  const int nqb = (p.L + kRows - 1) / kRows;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.y);  // longest blocks first
  const int r0 = qb * kRows;
  const int rlast = min(p.L, r0 + kRows) - 1;
  const int g = p.HQ / p.HKV, kh = h / g;
  const size_t bh = (size_t)b * p.HKV + kh;
  const int32_t* kpos = p.kpos + bh * p.ntq * kKeys;
  const int32_t* fpos = p.fpos + bh * p.ntf * kKeys;
  constexpr bool kF8F6F4 = kDt != kDtInt8;  // quantised S on kind::f8f6f4
  constexpr int kKImg = kF8F6F4 ? kImg8 : kImg16;

  if (tid == 0) {
    mbar_init(qready, kSoft);
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(vfull + i, 1);
      mbar_init(vempty + i, 1);
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(kfull + i, 1);
      mbar_init(kempty + i, 1);
    }
    mbar_init(pfull, kSoft);
    mbar_init(pfull + 1, kSoft);
    mbar_init(pvdone, 1);
    mbar_init(pvdone + 1, 1);
    mbar_init(mmadone, 2);  // one commit from each MMA-issuing thread
    mbar_init(sfull, 1);
    mbar_init(sfree, kSoft);
    mbar_fence_init();
    *abort_flag = 0;
  }
  if (warp == kCopyWarp) {
    // last key position any row of the block may see in the listed segments
    const int32_t hi = kBand ? rlast - p.W : rlast, lo = kBand ? r0 - p.W : r0;
    const int cq1 = warp_count_le(kpos, p.ntq * kKeys, hi, lane);
    const int cf1 = warp_count_le(fpos, p.ntf * kKeys, hi, lane);
    const int cq0 = warp_count_le(kpos, p.ntq * kKeys, lo, lane);
    const int cf0 = warp_count_le(fpos, p.ntf * kKeys, lo, lane);
    if (lane == 0) {
      ntiles[0] = (cq1 + kKeys - 1) / kKeys;
      ntiles[1] = (cf1 + kKeys - 1) / kKeys;
      // tiles before these hold only keys every row of the block sees
      ntiles[2] = cq0 / kKeys;
      ntiles[3] = cf0 / kKeys;
      // band tiles: positions r0 - W + 1 .. rlast
      const int tb0 = max(0, r0 - p.W + 1) / kKeys;
      ntiles[4] = tb0;
      ntiles[5] = (kBand && p.W > 0) ? rlast / kKeys - tb0 + 1 : 0;
    }
  }
  if (warp == kMmaWarp) tc_alloc(tslot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int nqt = ntiles[0], nlt = ntiles[0] + ntiles[1], nt = nlt + ntiles[5];
  const int mask_q = ntiles[2], mask_f = ntiles[3], tb0 = ntiles[4];

  if (tid < kSoft) {
    // ---------------- softmax / epilogue warps --------------------------
    // Thread = (query row, key half): warps 0-3 take keys 0-63 of every
    // tile, warps 4-7 keys 64-127, each half with its own online-softmax
    // state and its own O accumulator in TMEM; the halves merge at the end.
    const int hf = tid >> 7;           // key half
    const int rr = tid & (kRows - 1);  // row in the block = TMEM lane
    const int row = r0 + rr;
    const bool rvalid = row <= rlast;
    auto fail = [&]() {
      *abort_flag = 1;
      hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
    };
    // Query row (dims 64hf .. 64hf+63) -> BF16 image and code image.
    uint4 qv[8];
    const uint4* qrow = reinterpret_cast<const uint4*>(
        p.q + (((size_t)b * p.HQ + h) * p.ldq + (rvalid ? row : 0)) * HYQ_D + 64 * hf);
#pragma unroll
    for (int c = 0; c < 8; ++c) qv[c] = rvalid ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(bf16_at(qv[c], e)));
      *reinterpret_cast<uint4*>(sm + kOffQ + hf * kRegion + swz(rr, c)) = qv[c];
    }
    amax = warp_max_xor(amax, 1);
    if (lane == 0) red[warp] = amax;
    asm volatile("bar.sync 1, 256;\n" ::: "memory");
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    const float sq = __fdiv_rn(amax, code_max(kDt)), rq = recip(sq);
    if (kDt == kDtFp4) {
      // dims 64hf .. 64hf+63: chunks 4hf .. 4hf+3
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(sm + kOffQc + swz(rr, 4 * hf + c)) = pack_f4x16(qv[2 * c], qv[2 * c + 1], sq);
    } else if (kDt == kDtFp8) {
#pragma unroll
      for (int c16 = 0; c16 < 4; ++c16) {  // 16 codes per chunk: chunks 4hf .. 4hf+3
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t acc = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int el = 16 * c16 + 4 * u + e;
            const float x = bf16_at(qv[el >> 3], el & 7);
            acc |= static_cast<uint32_t>(code_f8_bits(x, sq)) << (8 * e);
          }
          w[u] = acc;
        }
        *reinterpret_cast<uint4*>(sm + kOffQc + swz(rr, 4 * hf + c16)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = bf16_at(qv[c], 2 * e), x1 = bf16_at(qv[c], 2 * e + 1);
          w[e] = pack_bf16x2(code_i8_fast(x0, sq, rq), code_i8_fast(x1, sq, rq));
        }
        *reinterpret_cast<uint4*>(sm + kOffQc + hf * kRegion + swz(rr, c)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(qready);

    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tbase + lane_off + (hf ? kColO1 : kColO0);
    const float* skp = p.sk + bh * p.ntq * 2 + hf;
    const float* svp = p.sv + bh * p.ntq * 2 + hf;
    const float qfac = p.alpha_log2e * sq;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    // this half's scales for the current tile, loaded a tile ahead
    float2 sc = nqt > 0 ? make_float2(__ldg(skp), __ldg(svp)) : make_float2(0.f, 1.f);
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      const bool quant = j < nqt;
      if (!mbar_wait_or_abort(sfull, j & 1, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      float x[64];
      {
        uint32_t ra[32], rb[32];
        const uint32_t ts = tbase + lane_off + kColS + 64 * hf;
        tc_ld32(ts, ra);
        tc_ld32(ts + 32, rb);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(ra[i]);
          x[32 + i] = __uint_as_float(rb[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(sfree);  // the MMA warp may compute the next tile's S now

      // A scale is 0 only when every code it multiplies is 0; keeping it
      // positive changes no score and makes masked (-inf) keys give 0.
      const float cs = quant ? fmaxf(qfac * sc.x, 1.17549435e-38f) : p.alpha_log2e;
      // log2 of the value scale, added to the exponent (2^(t + log2 vf) =
      // vf 2^t); a scale below 2^-60 only multiplies codes whose values are
      // below 2^-51, so raising it to 2^-60 changes no output.
      const float lvf = quant ? fast_log2(fmaxf(sc.y, 8.67361738e-19f)) : 0.f;
      if (j + 1 < nqt) sc = make_float2(__ldg(skp + 2 * j + 2), __ldg(svp + 2 * j + 2));
      // some key of the tile is hidden from some row of the block
      const bool masked = quant ? j >= mask_q : (j < nlt ? j - nqt >= mask_f : true);
      if (masked) {
        const int lim = kBand ? row - p.W : row;  // last visible position of a listed segment
        if (!kBand || j < nlt) {
          const int4* pp =
              reinterpret_cast<const int4*>((quant ? kpos + j * kKeys : fpos + (j - nqt) * kKeys) + 64 * hf);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int4 q4 = __ldg(pp + c);
            if (q4.x > lim) x[4 * c] = -INFINITY;
            if (q4.y > lim) x[4 * c + 1] = -INFINITY;
            if (q4.z > lim) x[4 * c + 2] = -INFINITY;
            if (q4.w > lim) x[4 * c + 3] = -INFINITY;
          }
        } else {
          // band tile: key i of this half is position base + i, visible
          // when lim < base + i <= row
          const int base = kKeys * (tb0 + j - nlt) + 64 * hf, ilo = lim - base, ihi = row - base;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i <= ilo || i > ihi) x[i] = -INFINITY;
        }
      }
      // P_h as BF16 pairs with the value scale folded in (the A operand of
      // P.V), built with the exponentials; stored once the P buffer is free.
      float rs;
      uint32_t pw[32];
      auto exps = [&](float mb) {
        // Pairs: scale and shift (by m - log2 vf, so that 2^t comes out
        // multiplied by vf), sum, pack (masked keys are -inf here and give 0);
        // the sum is taken back to the unscaled terms once per tile.
        const uint64_t cs2 = f2_splat(cs), nmb2 = f2_splat(lvf - mb);
        uint64_t ps2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int w = 0; w < 32; ++w) {
          uint64_t e2 = f2_fma(f2_pack(x[2 * w], x[2 * w + 1]), cs2, nmb2);
          e2 = f2_pack(fast_exp2(f2_lo(e2)), fast_exp2(f2_hi(e2)));
          ps2[w & 3] = f2_add(ps2[w & 3], e2);
          pw[w] = pack_bf16x2(f2_lo(e2), f2_hi(e2));
        }
        const uint64_t r2 = f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3]));
        rs = (f2_lo(r2) + f2_hi(r2)) * fast_exp2(-lvf);
      };
      // Lazy maximum.  Once a row has a running maximum, the tile's terms
      // are formed against it without a row maximum: their sum bounds each
      // of them, so a sum up to 2^16 means no term exceeds 2^16 and nothing
      // needs rescaling (all of them are far inside the FP32 and BF16
      // range).  A warp with a row whose sum is larger (or not finite), or
      // with a row that has no maximum yet, takes the row maximum and
      // rescales the rows where it grew by more than 2^8.
      float fac = 1.f;
      bool full = __any_sync(0xffffffffu, m_used == -INFINITY);
      if (!full) {
        exps(m_used);
        full = __any_sync(0xffffffffu, !(rs <= 65536.f));
      }
      if (full) {
        float a[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) a[u] = x[u];
#pragma unroll
        for (int i = 8; i < 64; i += 2) a[(i >> 1) & 7] = fmax3(a[(i >> 1) & 7], x[i], x[i + 1]);
        const float hmax = fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
        const float tmax = hmax == -INFINITY ? -INFINITY : hmax * cs;
        const bool grow = tmax > m_used + 8.f;
        const float m_new = grow ? tmax : m_used;
        fac = grow ? fast_exp2(m_used - m_new) : 1.f;
        m_used = m_new;
        exps(m_new == -INFINITY ? 0.f : m_new);
      }
      l_sum = l_sum * fac + rs;

      // A rescale of O needs every earlier P.V finished (the previous
      // tile's); otherwise only the P.V that last read this tile's P buffer
      // (two tiles back) has to be.
      const bool resc = j > 0 && __any_sync(0xffffffffu, fac != 1.f);
      if (resc || j > 1) {
        const int jw = resc ? j - 1 : j - 2;
        if (!mbar_wait_or_abort(pvdone + (jw & 1), (jw >> 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (resc) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tc_ld32(tO + 32 * c, o);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * fac);
            tc_st32(tO + 32 * c, o);
          }
          tc_wait_st();
        }
      }
      // P buffer j % 2: the P.V that last read it is done
      tc_st32(tbase + lane_off + kColP + 64 * s + 32 * hf, pw);
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(pfull + s);
    }
    // Merge the two halves.  Each half waits for the last P.V, leaves
    // (m, l) in its own region of key stage 0 (no copy or MMA touches it any
    // more: every MMA before that last P.V has finished), and the named barrier
    // makes both halves' accumulators and (m, l) visible to every thread;
    // each thread then writes dims 64hf .. 64hf+63 of its row.
    bool done = ok && nt > 0;
    if (done && !mbar_wait_or_abort(pvdone + ((nt - 1) & 1), ((nt - 1) >> 1) & 1, abort_flag)) {
      fail();
      done = false;
    }
    float* xch_own = reinterpret_cast<float*>(sm + kOffK + hf * kRegion);
    const float* xch_oth = reinterpret_cast<const float*>(sm + kOffK + (hf ^ 1) * kRegion);
    if (done) {
      xch_own[rr] = m_used;
      xch_own[kRows + rr] = l_sum;
    }
    tc_fence_before();
    asm volatile("bar.sync 1, 256;\n" ::: "memory");
    if (done && !*abort_flag) {
      tc_fence_after();
      const float ma = hf ? xch_oth[rr] : m_used, la = hf ? xch_oth[kRows + rr] : l_sum;
      const float mb2 = hf ? m_used : xch_oth[rr], lb = hf ? l_sum : xch_oth[kRows + rr];
      const float m = fmaxf(ma, mb2);
      const float wa = ma == -INFINITY ? 0.f : fast_exp2(ma - m);
      const float wb = mb2 == -INFINITY ? 0.f : fast_exp2(mb2 - m);
      const float l = la * wa + lb * wb;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float fa = wa * inv, fb = wb * inv;
      uint4* orow = reinterpret_cast<uint4*>(p.out + (((size_t)b * p.HQ + h) * p.L + row) * HYQ_D + 64 * hf);
      const uint32_t ta = tbase + lane_off + kColO0 + 64 * hf, tb = tbase + lane_off + kColO1 + 64 * hf;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t oa[32], ob[32];
        tc_ld32(ta + 32 * c, oa);
        tc_ld32(tb + 32 * c, ob);
        tc_wait_ld();
        if (rvalid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              f[e] = __uint_as_float(oa[8 * u + e]) * fa + __uint_as_float(ob[8 * u + e]) * fb;
            orow[4 * c + u] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                         pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
          }
        }
      }
    }
  } else if (warp == kCopyWarp || warp == kCopyWarp + 1) {
    // ---------------- copy warps: keys (8) and values (9), each its own
    // ring, so that key tiles are not held back by value tiles.  A tile
    // image goes as four quarter copies from the four lanes of its stage:
    // the bulk copies one thread issues complete one after another, so
    // separate lanes per stage keep every stage's copies in flight. -------
    const bool is_v = warp != kCopyWarp;
    uint64_t* full = is_v ? vfull : kfull;
    uint64_t* empty = is_v ? vempty : kempty;
    const int qimg = is_v ? kImg16 : kKImg;
    const uint8_t* qsrc = is_v ? p.vq + bh * p.ntq * (size_t)kImg16 : p.kq + bh * p.ntq * (size_t)kKImg;
    const uint8_t* fsrc = (is_v ? p.vf : p.kf) + bh * p.ntf * (size_t)kImg16;
    const uint8_t* bsrc = (is_v ? p.vb : p.kb) + bh * p.ntb * (size_t)kImg16;
    uint8_t* dst = sm + (is_v ? kOffV : kOffK);
    const int nst = is_v ? kVStages : kKStages;  // ring stages
    int last_j = -1;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int s = j % nst;
      if (j >= nst) {
        bool got = true;
        if (lane == 0) got = mbar_wait_or_abort(empty + s, ((j / nst) & 1) ^ 1, abort_flag);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
      }
      const bool quant = j < nqt;
      const uint32_t bytes = quant ? qimg : kImg16, part = bytes / 4;
      const uint8_t* src = quant     ? qsrc + (size_t)j * qimg
                           : j < nlt ? fsrc + (size_t)(j - nqt) * kImg16
                                     : bsrc + (size_t)(tb0 + j - nlt) * kImg16;
      if (lane == 0) mbar_arrive_expect_tx(full + s, bytes);
      __syncwarp();
      // stage s is always filled by lanes 4s .. 4s+3, so the stages' copies
      // are in flight together
      const int qt = lane - 4 * s;
      if (qt >= 0 && qt < 4) bulk_g2s(dst + s * kImg16 + qt * part, src + qt * part, part, full + s);
      last_j = j;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
      // let the copies in flight (the last stages' tiles) land before the
      // CTA's shared memory goes away
      for (int j = max(0, last_j - nst + 1); j <= last_j; ++j) mbar_wait(full + j % nst, (j / nst) & 1);
    }
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ---------------- MMA warps ----------------------------------------
    if (lane == 0) {
      const uint32_t aQ = smem_u32(sm + kOffQ), aQc = smem_u32(sm + kOffQc);
      bool ok = mbar_wait_or_abort(qready, 0, abort_flag);
      tc_fence_after();
      // Each MMA thread shares its scheduler with two softmax warps, so its
      // own instructions are few: descriptors are built once and advanced by
      // adding offsets (the start-address field counts 16-byte units), ring
      // stages and phases are tracked incrementally.
      const uint64_t dQc = tc_desc_sw128(aQc), dQ = tc_desc_sw128(aQ);
      const uint64_t dK0 = tc_desc_sw128(smem_u32(sm + kOffK)), dV0 = tc_desc_sw128(smem_u32(sm + kOffV));
      constexpr uint64_t kStageStep = kImg16 >> 4, kRegionStep = kRegion >> 4;
      const uint32_t tS = tbase + kColS;
      int sk = 0, sv = 0;
      uint32_t kph = 0, vph = 0;
      // Two issuing threads: warp 10 the S = Q K^T products, warp 11 the
      // O += P V products.  A commit tracks the MMAs of the thread that
      // issues it, and the two streams write disjoint TMEM (S; O, reading P
      // from its own buffers), so each waits only on its own inputs.
      if (warp == kMmaWarp) {
        for (int j = 0; ok && j < nt; ++j) {
          ok = mbar_wait_or_abort(kfull + sk, kph, abort_flag);
          // the softmax has read S of the previous tile
          if (ok && j >= 1) ok = mbar_wait_or_abort(sfree, (j - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dK = dK0 + sk * kStageStep;
          if (kDt == kDtFp8 && j < nqt) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc_mma_f8(tS, dQc + 2 * ks, dK + 2 * ks, kIdescE4M3, ks > 0);
          } else if (kDt == kDtFp4 && j < nqt) {  // 32 elements (two 16-byte chunks) per MMA
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) tc_mma_f8(tS, dQc + 2 * ks, dK + 2 * ks, kIdescE2M1, ks > 0);
          } else {
            const uint64_t dA = j < nqt ? dQc : dQ;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t off = (ks >> 2) * kRegionStep + (ks & 3) * 2;
              tc_mma_f16(tS, dA + off, dK + off, kIdescBF16, ks > 0);
            }
          }
          tc_commit(sfull);
          tc_commit(kempty + sk);
          if (++sk == kKStages) {
            sk = 0;
            kph ^= 1;
          }
        }
      } else {
        for (int i = 0; ok && i < nt; ++i) {  // O_h += P_h V_h for the two key halves h
          const uint32_t tP = tbase + kColP + 64 * (i & 1);
          ok = mbar_wait_or_abort(vfull + sv, vph, abort_flag);
          const uint64_t dV = dV0 + sv * kStageStep;
          if (ok) ok = mbar_wait_or_abort(pfull + (i & 1), (i >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t tO = tbase + (hf ? kColO1 : kColO0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_f16_ts(tO, tP + 32 * hf + 8 * ks, dV + hf * kRegionStep + 2 * ks, kIdescBF16,
                            (i > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(pvdone + (i & 1));
          tc_commit(vempty + sv);
          if (++sv == kVStages) {
            sv = 0;
            vph ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
      }
      tc_commit(mmadone);  // every MMA this thread issued has finished once both arrive
      mbar_wait(mmadone, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tc_dealloc(tbase, kTmemCols);
  }
}

size_t align_up(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

struct WsLayout {
  size_t kq, vq, kf, vf, kb, vb, kpos, fpos, sk, sv, total;
};

WsLayout ws_layout(const hyq_config* c, bool k8, int32_t ntq, int32_t ntf, int32_t ntb) {
  const size_t bh = (size_t)c->batch * c->num_kv_heads;
  WsLayout w{};
  size_t off = 0;
  w.kq = off;
  off = align_up(off + bh * ntq * (size_t)(k8 ? kImg8 : kImg16));
  w.vq = off;
  off = align_up(off + bh * ntq * (size_t)kImg16);
  w.kf = off;
  off = align_up(off + bh * ntf * (size_t)kImg16);
  w.vf = off;
  off = align_up(off + bh * ntf * (size_t)kImg16);
  w.kb = off;
  off = align_up(off + bh * ntb * (size_t)kImg16);
  w.vb = off;
  off = align_up(off + bh * ntb * (size_t)kImg16);
  w.kpos = off;
  off = align_up(off + bh * ntq * (size_t)kKeys * 4);
  w.fpos = off;
  off = align_up(off + bh * ntf * (size_t)kKeys * 4);
  w.sk = off;
  off = align_up(off + bh * ntq * 2 * sizeof(float));
  w.sv = off;
  off = align_up(off + bh * ntq * 2 * sizeof(float));
  w.total = off;
  return w;
}

template <int kDt, bool kBand>
cudaError_t launch_main(const MainParams& mp, dim3 grid, cudaStream_t s) {
  static std::atomic<uint64_t> done{0};
  const cudaError_t e = hyq_once_per_device(done, [] {
    return cudaFuncSetAttribute(prefill_kernel<kDt, kBand>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  prefill_kernel<kDt, kBand><<<grid, kThreads, kSmemBytes, s>>>(mp);
  return cudaGetLastError();
}

int32_t tiles_of(int32_t n) { return (n + kKeys - 1) / kKeys; }

}  // namespace

// Full-precision list: the vertical lines, plus the last W positions for the
// fixed window; the band mode adds BF16 images of all L positions instead.
size_t hyq_prefill_ws_bytes(const hyq_config* c, int dtype, int32_t L, int32_t kvl, bool band) {
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const int32_t nq = P - kvl, nfp = band ? kvl : kvl + (L - P);
  return ws_layout(c, dtype != HYQ_PREFILL_INT8, tiles_of(nq), tiles_of(nfp), band ? tiles_of(L) : 0).total;
}

size_t hyq_prefill_ws_bytes_hint(const hyq_config* c, int32_t L, bool band) {
  // Worst case over the calls with context length <= L: every prefix position
  // quantised (kvl = 0) for the code images, the configured vertical-line
  // count (plus the window) for the BF16 images; 16-bit key codes.
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const int32_t nfp = hyq_vl_count(c, P) + (band ? 0 : L - P);
  return ws_layout(c, false, tiles_of(P), tiles_of(nfp), band ? tiles_of(L) : 0).total;
}

cudaError_t hyq_launch_prefill(const hyq_config* c, int dtype, const void* q, int64_t ldq, const void* k,
                               const void* v, int64_t ldk, int32_t L, const int32_t* vl, int32_t kvl, void* out,
                               void* ws, int32_t* err, cudaStream_t s, bool band) {
  const bool k8 = dtype != HYQ_PREFILL_INT8;  // 8-bit key images (e4m3, or packed e2m1)
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const int32_t nq = P - kvl, nfp = band ? kvl : kvl + (L - P);
  const int32_t ntq = tiles_of(nq), ntf = tiles_of(nfp), ntb = band ? tiles_of(L) : 0;
  const WsLayout w = ws_layout(c, k8, ntq, ntf, ntb);
  uint8_t* base = static_cast<uint8_t*>(ws);

  PackParams pp{};
  pp.k = static_cast<const __nv_bfloat16*>(k);
  pp.v = static_cast<const __nv_bfloat16*>(v);
  pp.ldk = ldk;
  pp.vl = vl;
  pp.kvl = kvl;
  pp.kq = base + w.kq;
  pp.vq = base + w.vq;
  pp.kf = base + w.kf;
  pp.vf = base + w.vf;
  pp.kb = base + w.kb;
  pp.vb = base + w.vb;
  pp.kpos = reinterpret_cast<int32_t*>(base + w.kpos);
  pp.fpos = reinterpret_cast<int32_t*>(base + w.fpos);
  pp.sk = reinterpret_cast<float*>(base + w.sk);
  pp.sv = reinterpret_cast<float*>(base + w.sv);
  pp.err = err;
  pp.L = L;
  pp.P = P;
  pp.HKV = c->num_kv_heads;
  pp.nq = nq;
  pp.nfp = nfp;
  pp.ntq = ntq;
  pp.ntf = ntf;
  pp.ntb = ntb;
  dim3 g1(2 * ntq + 2 * ntf + 2 * ntb, c->num_kv_heads, c->batch);
  if (dtype == HYQ_PREFILL_FP8) pack_kernel<kDtFp8><<<g1, 256, 0, s>>>(pp);
  else if (dtype == HYQ_PREFILL_FP4) pack_kernel<kDtFp4><<<g1, 256, 0, s>>>(pp);
  else pack_kernel<kDtInt8><<<g1, 256, 0, s>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  MainParams mp{};
  mp.q = static_cast<const __nv_bfloat16*>(q);
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.kq = pp.kq;
  mp.vq = pp.vq;
  mp.kf = pp.kf;
  mp.vf = pp.vf;
  mp.kb = pp.kb;
  mp.vb = pp.vb;
  mp.kpos = pp.kpos;
  mp.fpos = pp.fpos;
  mp.sk = pp.sk;
  mp.sv = pp.sv;
  mp.err = err;
  mp.ldq = ldq;
  mp.L = L;
  mp.HQ = c->num_q_heads;
  mp.HKV = c->num_kv_heads;
  mp.ntq = ntq;
  mp.ntf = ntf;
  mp.ntb = ntb;
  mp.W = c->window;
  mp.alpha_log2e = kLog2e / sqrtf(static_cast<float>(HYQ_D));
  dim3 g2(c->num_q_heads, (L + kRows - 1) / kRows, c->batch);
  if (dtype == HYQ_PREFILL_FP8)
    return band ? launch_main<kDtFp8, true>(mp, g2, s) : launch_main<kDtFp8, false>(mp, g2, s);
  if (dtype == HYQ_PREFILL_FP4)
    return band ? launch_main<kDtFp4, true>(mp, g2, s) : launch_main<kDtFp4, false>(mp, g2, s);
  return band ? launch_main<kDtInt8, true>(mp, g2, s) : launch_main<kDtInt8, false>(mp, g2, s);
}
