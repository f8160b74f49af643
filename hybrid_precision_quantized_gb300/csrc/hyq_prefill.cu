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
//     head).  Warp 4 streams key/value tiles (bulk copies, 2-stage rings);
//     warp 5 issues tcgen05.mma: S = Q K^T into TMEM (double buffer), then
//     O += P V into TMEM; warps 0-3 (one thread per query row = TMEM lane)
//     read S, scale, mask, run the online softmax and write P back to shared
//     memory.  The quantised segment uses e4m3 codes (kind::f8f6f4) or INT8
//     codes held exactly as BF16 integers (kind::f16; sm_103a has no integer
//     tensor-core MMA); the full-precision segment uses BF16.  P.V runs in
//     BF16 with the value codes (exact in BF16) and the value scale folded
//     into P.
//
// Every wait is bounded; on expiry the kernel sets HYQ_DEVERR_TIMEOUT, drains
// its own copies and MMAs, frees its TMEM and returns.
#include <cuda_fp8.h>

#include <cmath>
#include <cstdint>

#include "hyq_tc.cuh"

namespace {

constexpr int kRows = 128;           // query rows per CTA (MMA M)
constexpr int kKeys = 128;           // keys per MMA tile
constexpr int kScaleTile = 64;       // keys per quantisation scale (B_N)
constexpr int kRegion = 16384;       // 128 rows x 128 bytes, swizzled
constexpr int kImg16 = 2 * kRegion;  // 128 x 128 16-bit operand image
constexpr int kImg8 = kRegion;       // 128 x 128 8-bit operand image
constexpr int kSoft = 128;           // softmax threads (warps 0-3)
constexpr int kThreads = 192;        // + copy warp (4) + MMA warp (5)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr int kOffQ = 0;                   // Q, BF16 image
constexpr int kOffQc = kOffQ + kImg16;     // Q codes image (8- or 16-bit)
constexpr int kOffK = kOffQc + kImg16;     // 2 key stages
constexpr int kOffV = kOffK + 2 * kImg16;  // 2 value stages (transposed)
constexpr int kOffP = kOffV + 2 * kImg16;  // probabilities, BF16 image
constexpr int kOffBar = kOffP + kImg16;
constexpr int kNumBars = 16;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 64;
constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base

constexpr uint32_t kIdescBF16 = tc_idesc(kTcBF16, kTcBF16, kRows, kKeys);
constexpr uint32_t kIdescE4M3 = tc_idesc(kTcE4M3, kTcE4M3, kRows, kKeys);

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
  int32_t* kpos;
  int32_t* fpos;
  float* sk;
  float* sv;
  int32_t* err;
  int32_t L, P, HKV, nq, nfp, ntq, ntf;
};

struct MainParams {
  const __nv_bfloat16* q;  // [B][HQ][ldq][128]
  __nv_bfloat16* out;      // [B][HQ][L][128]
  const uint8_t* kq;
  const uint8_t* vq;
  const uint8_t* kf;
  const uint8_t* vf;
  const int32_t* kpos;  // [B][HKV][ntq*128], ascending, padding INT32_MAX
  const int32_t* fpos;  // [B][HKV][ntf*128]
  const float* sk;      // [B][HKV][ntq*2]
  const float* sv;
  int32_t* err;
  int64_t ldq;
  int32_t L, HQ, HKV, ntq, ntf;
  float alpha_log2e;
};

// Byte offset of the 16-byte chunk `c` (of the 128-byte row `r`) in a
// 128-byte-swizzled region.
__device__ __forceinline__ int swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ float bf16_at(const uint4& u, int e) {
  const uint32_t w = (&u.x)[e >> 1];
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// INT8 code of t (rint, ties to even, clamped to +-127).
__device__ __forceinline__ float code_i8(float t) { return fminf(fmaxf(rintf(t), -127.f), 127.f); }

// e4m3 code of t (nearest, ties to even, saturating) as its float value.
__device__ __forceinline__ float code_f8(float t) {
  __nv_fp8_e4m3 c(t);  // round to nearest even, saturate to finite
  return static_cast<float>(c);
}

__device__ __forceinline__ uint8_t code_f8_bits(float t) {
  return __nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
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
// Stage 1-2: key lists, scales, code images.  Grid (2 ntq + 2 ntf, HKV, B);
// each block handles one 64-key scale tile of one list.
// ---------------------------------------------------------------------------
template <bool kFp8>
__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackParams p) {
  __shared__ float vs[kScaleTile][HYQ_D + 1];
  __shared__ int32_t spos[kScaleTile];
  __shared__ float red[8];
  const int tid = threadIdx.x;
  const int kh = blockIdx.y, b = blockIdx.z;
  const size_t bh = (size_t)b * p.HKV + kh;
  const bool quant = blockIdx.x < 2 * p.ntq;
  const int t64 = quant ? blockIdx.x : blockIdx.x - 2 * p.ntq;
  const int n = quant ? p.nq : p.nfp;
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
    if (quant) p.kpos[bh * p.ntq * kKeys + i] = pos;
    else p.fpos[bh * p.ntf * kKeys + i] = pos;
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
  float sk = 1.f, sv = 1.f;
  if (quant) {
    float ak = 0.f, av = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      ak = fmaxf(ak, fabsf(bf16_at(kr[e >> 3], e & 7)));
      av = fmaxf(av, fabsf(bf16_at(vr[e >> 3], e & 7)));
    }
    const float cb = kFp8 ? 448.f : 127.f;
    ak = block_max(ak, red, 8);
    av = block_max(av, red, 8);
    sk = __fdiv_rn(ak, cb);
    sv = __fdiv_rn(av, cb);
    if (tid == 0) {
      p.sk[bh * p.ntq * 2 + t64] = sk;
      p.sv[bh * p.ntq * 2 + t64] = sv;
    }
  }

  // Key image.
  if (quant && kFp8) {
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
          const float t = sk > 0.f ? __fdiv_rn(x, sk) : 0.f;
          acc |= static_cast<uint32_t>(code_f8_bits(t)) << (8 * e);
        }
        w[u] = acc;
      }
      *reinterpret_cast<uint4*>(img + swz(key, 2 * qq + h)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    uint8_t* img = quant ? p.kq + (bh * p.ntq + tile) * (size_t)kImg16
                         : p.kf + (bh * p.ntf + tile) * (size_t)kImg16;
    // dims 32qq .. 32qq+31 = bytes 64qq .. 64qq+63: region qq/2, chunks 4(qq&1)..+3
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 u = kr[c];
      if (quant) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = bf16_at(kr[c], 2 * e), x1 = bf16_at(kr[c], 2 * e + 1);
          const float t0 = sk > 0.f ? __fdiv_rn(x0, sk) : 0.f;
          const float t1 = sk > 0.f ? __fdiv_rn(x1, sk) : 0.f;
          w[e] = pack_bf16x2(code_i8(t0), code_i8(t1));
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
    if (quant) {
      const float t = sv > 0.f ? __fdiv_rn(x, sv) : 0.f;
      y = kFp8 ? code_f8(t) : code_i8(t);
    }
    vs[r][32 * qq + e] = y;
  }
  __syncthreads();
  uint8_t* vimg = quant ? p.vq + (bh * p.ntq + tile) * (size_t)kImg16
                        : p.vf + (bh * p.ntf + tile) * (size_t)kImg16;
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
// Stage 3: segmented online softmax on tcgen05.
// ---------------------------------------------------------------------------
template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ MainParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* qready = bars + 0;
  uint64_t* kfull = bars + 1;   // [2]
  uint64_t* kempty = bars + 3;  // [2]
  uint64_t* vfull = bars + 5;   // [2]
  uint64_t* vempty = bars + 7;  // [2]
  uint64_t* sfull = bars + 9;   // [2]
  uint64_t* sfree = bars + 11;  // [2]
  uint64_t* pfull = bars + 13;
  uint64_t* pvdone = bars + 14;
  uint64_t* mmadone = bars + 15;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);
  int* ntiles = reinterpret_cast<int*>(sm + kOffMisc + 8);  // [2]
  float* red = reinterpret_cast<float*>(sm + kOffMisc + 32);  // [4]

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
  constexpr int kKImg = kFp8 ? kImg8 : kImg16;

  if (tid == 0) {
    mbar_init(qready, kSoft);
    for (int i = 0; i < 2; ++i) {
      mbar_init(kfull + i, 1);
      mbar_init(kempty + i, 1);
      mbar_init(vfull + i, 1);
      mbar_init(vempty + i, 1);
      mbar_init(sfull + i, 1);
      mbar_init(sfree + i, kSoft);
    }
    mbar_init(pfull, kSoft);
    mbar_init(pvdone, 1);
    mbar_init(mmadone, 1);
    mbar_fence_init();
    *abort_flag = 0;
    ntiles[0] = (count_le(kpos, p.ntq * kKeys, rlast) + kKeys - 1) / kKeys;
    ntiles[1] = (count_le(fpos, p.ntf * kKeys, rlast) + kKeys - 1) / kKeys;
  }
  if (warp == 5) tc_alloc(tslot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int nqt = ntiles[0], nt = ntiles[0] + ntiles[1];

  if (tid < kSoft) {
    // ---------------- softmax / epilogue warps --------------------------
    const int row = r0 + tid;
    const bool rvalid = row <= rlast;
    auto fail = [&]() {
      *abort_flag = 1;
      hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
    };
    // Query row -> BF16 image and code image.
    uint4 qv[16];
    const uint4* qrow =
        reinterpret_cast<const uint4*>(p.q + (((size_t)b * p.HQ + h) * p.ldq + (rvalid ? row : 0)) * HYQ_D);
#pragma unroll
    for (int c = 0; c < 16; ++c) qv[c] = rvalid ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(bf16_at(qv[c], e)));
      *reinterpret_cast<uint4*>(sm + kOffQ + (c >> 3) * kRegion + swz(tid, c & 7)) = qv[c];
    }
    amax = warp_max_xor(amax, 1);
    if (lane == 0) red[warp] = amax;
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float sq = __fdiv_rn(amax, kFp8 ? 448.f : 127.f);
    if (kFp8) {
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t acc = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int el = 16 * c16 + 4 * u + e;
            const float x = bf16_at(qv[el >> 3], el & 7);
            const float t = sq > 0.f ? __fdiv_rn(x, sq) : 0.f;
            acc |= static_cast<uint32_t>(code_f8_bits(t)) << (8 * e);
          }
          w[u] = acc;
        }
        *reinterpret_cast<uint4*>(sm + kOffQc + swz(tid, c16)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = bf16_at(qv[c], 2 * e), x1 = bf16_at(qv[c], 2 * e + 1);
          const float t0 = sq > 0.f ? __fdiv_rn(x0, sq) : 0.f;
          const float t1 = sq > 0.f ? __fdiv_rn(x1, sq) : 0.f;
          w[e] = pack_bf16x2(code_i8(t0), code_i8(t1));
        }
        *reinterpret_cast<uint4*>(sm + kOffQc + (c >> 3) * kRegion + swz(tid, c & 7)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(qready);

    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float* skp = p.sk + bh * p.ntq * 2;
    const float* svp = p.sv + bh * p.ntq * 2;
    const float qfac = p.alpha_log2e * sq;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      const bool quant = j < nqt;
      if (!mbar_wait_or_abort(sfull + s, (j >> 1) & 1, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      float x[128];
      {
        uint32_t r0v[32], r1v[32], r2v[32], r3v[32];
        const uint32_t ts = tbase + lane_off + (s ? kColS1 : kColS0);
        tc_ld32(ts + 0, r0v);
        tc_ld32(ts + 32, r1v);
        tc_ld32(ts + 64, r2v);
        tc_ld32(ts + 96, r3v);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(r0v[i]);
          x[32 + i] = __uint_as_float(r1v[i]);
          x[64 + i] = __uint_as_float(r2v[i]);
          x[96 + i] = __uint_as_float(r3v[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(sfree + s);

      const int32_t* tpos = quant ? kpos + j * kKeys : fpos + (j - nqt) * kKeys;
      float cs0, cs1, vf0, vf1;
      if (quant) {
        cs0 = qfac * __ldg(skp + 2 * j);
        cs1 = qfac * __ldg(skp + 2 * j + 1);
        vf0 = __ldg(svp + 2 * j);
        vf1 = __ldg(svp + 2 * j + 1);
      } else {
        cs0 = cs1 = p.alpha_log2e;
        vf0 = vf1 = 1.f;
      }
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        x[i] *= cs0;
        x[64 + i] *= cs1;
      }
      if (__ldg(tpos + kKeys - 1) > r0) {  // some key of this tile is after some row
        const int4* pp = reinterpret_cast<const int4*>(tpos);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int4 q4 = __ldg(pp + c);
          if (q4.x > row) x[4 * c] = -INFINITY;
          if (q4.y > row) x[4 * c + 1] = -INFINITY;
          if (q4.z > row) x[4 * c + 2] = -INFINITY;
          if (q4.w > row) x[4 * c + 3] = -INFINITY;
        }
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) tmax = fmaxf(tmax, x[i]);
      // Lazy maximum: rescale only when the row maximum grew by more than 2^8.
      const bool grow = tmax > m_used + 8.f;
      const float m_new = grow ? tmax : m_used;
      const float fac = grow ? exp2f(m_used - m_new) : 1.f;
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;
      float rs = 0.f;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        x[i] = exp2f(x[i] - mb);
        rs += x[i];
      }
      l_sum = l_sum * fac + rs;
      m_used = m_new;

      if (j > 0) {  // P.V of the previous tile done: O stable, P buffer free
        if (!mbar_wait_or_abort(pvdone, (j - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, fac != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            const uint32_t to = tbase + lane_off + kColO + 32 * c;
            tc_ld32(to, o);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * fac);
            tc_st32(to, o);
          }
          tc_wait_st();
        }
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float f = c < 8 ? vf0 : vf1;
        const uint4 u = make_uint4(pack_bf16x2(x[8 * c] * f, x[8 * c + 1] * f),
                                   pack_bf16x2(x[8 * c + 2] * f, x[8 * c + 3] * f),
                                   pack_bf16x2(x[8 * c + 4] * f, x[8 * c + 5] * f),
                                   pack_bf16x2(x[8 * c + 6] * f, x[8 * c + 7] * f));
        *reinterpret_cast<uint4*>(sm + kOffP + (c >> 3) * kRegion + swz(tid, c & 7)) = u;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(pfull);
    }
    if (ok && nt > 0) {
      if (!mbar_wait_or_abort(pvdone, (nt - 1) & 1, abort_flag)) {
        fail();
      } else {
        tc_fence_after();
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        uint4* orow = reinterpret_cast<uint4*>(p.out + (((size_t)b * p.HQ + h) * p.L + row) * HYQ_D);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc_ld32(tbase + lane_off + kColO + 32 * c, o);
          tc_wait_ld();
          if (rvalid) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float* f = reinterpret_cast<const float*>(o) + 8 * u;
              orow[4 * c + u] = make_uint4(pack_bf16x2(f[0] * inv, f[1] * inv), pack_bf16x2(f[2] * inv, f[3] * inv),
                                           pack_bf16x2(f[4] * inv, f[5] * inv), pack_bf16x2(f[6] * inv, f[7] * inv));
            }
          }
        }
      }
    }
  } else if (warp == 4) {
    // ---------------- copy warp ----------------------------------------
    if (lane == 0) {
      const uint8_t* kq = p.kq + bh * p.ntq * (size_t)kKImg;
      const uint8_t* vq = p.vq + bh * p.ntq * (size_t)kImg16;
      const uint8_t* kf = p.kf + bh * p.ntf * (size_t)kImg16;
      const uint8_t* vf = p.vf + bh * p.ntf * (size_t)kImg16;
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      bool ok = true;
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1;
        const uint32_t prev = ((j >> 1) & 1) ^ 1;
        const bool quant = j < nqt;
        if (j >= 2 && !mbar_wait_or_abort(kempty + s, prev, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t kb = quant ? kKImg : kImg16;
        mbar_arrive_expect_tx(kfull + s, kb);
        bulk_g2s(sm + kOffK + s * kImg16, quant ? kq + (size_t)j * kKImg : kf + (size_t)(j - nqt) * kImg16, kb,
                 kfull + s);
        last_k[s] = j;
        if (j >= 2 && !mbar_wait_or_abort(vempty + s, prev, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(vfull + s, kImg16);
        bulk_g2s(sm + kOffV + s * kImg16, quant ? vq + (size_t)j * kImg16 : vf + (size_t)(j - nqt) * kImg16,
                 kImg16, vfull + s);
        last_v[s] = j;
      }
      if (!ok) {
        *abort_flag = 1;
        hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
        // let the copies in flight land before the CTA's shared memory goes away
        for (int s = 0; s < 2; ++s) {
          if (last_k[s] >= 0) mbar_wait(kfull + s, (last_k[s] >> 1) & 1);
          if (last_v[s] >= 0) mbar_wait(vfull + s, (last_v[s] >> 1) & 1);
        }
      }
    }
  } else {
    // ---------------- MMA warp -----------------------------------------
    if (lane == 0) {
      const uint32_t tS[2] = {tbase + kColS0, tbase + kColS1};
      const uint32_t tO = tbase + kColO;
      const uint32_t aQ = smem_u32(sm + kOffQ), aQc = smem_u32(sm + kOffQc), aP = smem_u32(sm + kOffP);
      bool ok = mbar_wait_or_abort(qready, 0, abort_flag);
      tc_fence_after();
      for (int j = 0; ok && j <= nt; ++j) {
        if (j < nt) {
          const int s = j & 1;
          ok = mbar_wait_or_abort(kfull + s, (j >> 1) & 1, abort_flag);
          if (ok && j >= 2) ok = mbar_wait_or_abort(sfree + s, ((j >> 1) & 1) ^ 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t aK = smem_u32(sm + kOffK + s * kImg16);
          if (kFp8 && j < nqt) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_f8(tS[s], tc_desc_sw128(aQc + 32 * ks), tc_desc_sw128(aK + 32 * ks), kIdescE4M3, ks > 0);
          } else {
            const uint32_t aA = j < nqt ? aQc : aQ;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = (ks >> 2) * kRegion + (ks & 3) * 32;
              tc_mma_f16(tS[s], tc_desc_sw128(aA + off), tc_desc_sw128(aK + off), kIdescBF16, ks > 0);
            }
          }
          tc_commit(sfull + s);
          tc_commit(kempty + s);
        }
        if (j >= 1) {  // O += P V for tile i = j - 1
          const int i = j - 1, s = i & 1;
          ok = mbar_wait_or_abort(pfull, i & 1, abort_flag);
          if (ok) ok = mbar_wait_or_abort(vfull + s, (i >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t aV = smem_u32(sm + kOffV + s * kImg16);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kRegion + (ks & 3) * 32;
            tc_mma_f16(tO, tc_desc_sw128(aP + off), tc_desc_sw128(aV + off), kIdescBF16, (i > 0 || ks > 0) ? 1u : 0u);
          }
          tc_commit(pvdone);
          tc_commit(vempty + s);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        hyq_set_err(p.err, HYQ_DEVERR_TIMEOUT);
      }
      tc_commit(mmadone);  // every MMA issued above has finished once this arrives
      mbar_wait(mmadone, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tc_dealloc(tbase, kTmemCols);
  }
}

size_t align_up(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

struct WsLayout {
  size_t kq, vq, kf, vf, kpos, fpos, sk, sv, total;
};

WsLayout ws_layout(const hyq_config* c, bool fp8, int32_t ntq, int32_t ntf) {
  const size_t bh = (size_t)c->batch * c->num_kv_heads;
  WsLayout w{};
  size_t off = 0;
  w.kq = off;
  off = align_up(off + bh * ntq * (size_t)(fp8 ? kImg8 : kImg16));
  w.vq = off;
  off = align_up(off + bh * ntq * (size_t)kImg16);
  w.kf = off;
  off = align_up(off + bh * ntf * (size_t)kImg16);
  w.vf = off;
  off = align_up(off + bh * ntf * (size_t)kImg16);
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

template <bool kFp8>
cudaError_t set_attrs() {
  static bool done = false;
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess) done = true;
  return e;
}

}  // namespace

size_t hyq_prefill_ws_bytes(const hyq_config* c, int dtype, int32_t L, int32_t kvl) {
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const int32_t nq = P - kvl, nfp = kvl + (L - P);
  return ws_layout(c, dtype == HYQ_PREFILL_FP8, (nq + kKeys - 1) / kKeys, (nfp + kKeys - 1) / kKeys).total;
}

size_t hyq_prefill_ws_bytes_hint(const hyq_config* c, int32_t L) {
  // Worst case over the calls with context length <= L: every prefix position
  // quantised (kvl = 0) for the code images, the configured vertical-line
  // count plus the window for the BF16 images; 16-bit key codes.
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const int32_t nfp = hyq_vl_count(c, P) + (L - P);
  return ws_layout(c, false, (P + kKeys - 1) / kKeys, (nfp + kKeys - 1) / kKeys).total;
}

cudaError_t hyq_launch_prefill(const hyq_config* c, int dtype, const void* q, int64_t ldq, const void* k,
                               const void* v, int64_t ldk, int32_t L, const int32_t* vl, int32_t kvl, void* out,
                               void* ws, int32_t* err, cudaStream_t s) {
  const bool fp8 = dtype == HYQ_PREFILL_FP8;
  const int32_t P = L - c->window > 0 ? L - c->window : 0;
  const int32_t nq = P - kvl, nfp = kvl + (L - P);
  const int32_t ntq = (nq + kKeys - 1) / kKeys, ntf = (nfp + kKeys - 1) / kKeys;
  const WsLayout w = ws_layout(c, fp8, ntq, ntf);
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
  dim3 g1(2 * ntq + 2 * ntf, c->num_kv_heads, c->batch);
  if (fp8) pack_kernel<true><<<g1, 256, 0, s>>>(pp);
  else pack_kernel<false><<<g1, 256, 0, s>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  MainParams mp{};
  mp.q = static_cast<const __nv_bfloat16*>(q);
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.kq = pp.kq;
  mp.vq = pp.vq;
  mp.kf = pp.kf;
  mp.vf = pp.vf;
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
  mp.alpha_log2e = kLog2e / sqrtf(static_cast<float>(HYQ_D));
  dim3 g2(c->num_q_heads, (L + kRows - 1) / kRows, c->batch);
  if (fp8) {
    if ((e = set_attrs<true>()) != cudaSuccess) return e;
    prefill_kernel<true><<<g2, kThreads, kSmemBytes, s>>>(mp);
  } else {
    if ((e = set_attrs<false>()) != cudaSuccess) return e;
    prefill_kernel<false><<<g2, kThreads, kSmemBytes, s>>>(mp);
  }
  return cudaGetLastError();
}
