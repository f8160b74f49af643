// 4-bit group quantiser and hybrid-cache construction.
//
// Quant_B(.; G) of Algorithm 4 ("HyQuant: Hybrid-Precision Quantization for
// LLM Attention", Appendix A.4) with B = 4 and G = 32 along head_dim, and the
// Freeze re-organisation of the cache into a 4-bit stream, vertical-line rows
// and a BF16 tail (§4.3 Eq. 8).
//
// A CTA builds one 64-row block image of the 4-bit stream in shared memory
// (codes placed directly in the tensor-core fragment order documented in
// hyq.h) and writes it out with 16-byte stores.  One warp quantises one
// 128-element row: lane l holds elements 4l..4l+3, lanes 8q..8q+7 form group q.
#include "hyq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Position of the nibble of (row tt of a 16-row tile, element e) in the K tile.
__device__ __forceinline__ void k_nibble(int tt, int e, int& word, int& shift) {
  int ks = e >> 4, c = e & 15;
  int ch = c >> 3, t = (c & 7) >> 1, lo_hi = c & 1;
  int g = tt & 7, rh = tt >> 3;
  int n = rh + 2 * ch + 4 * lo_hi;
  int lane = 4 * g + t;
  word = (512 * (ks >> 2) + 16 * lane + 4 * (ks & 3)) >> 2;
  shift = 4 * n;
}

// Same for the V tile (rows of the tensor-core A operand are elements).
__device__ __forceinline__ void v_nibble(int tt, int e, int& word, int& shift) {
  int mt = e >> 4, rr = e & 15;
  int g = rr & 7, rh = rr >> 3;
  int ch = tt >> 3, t = (tt & 7) >> 1, lo_hi = tt & 1;
  int n = rh + 2 * ch + 4 * lo_hi;
  int lane = 4 * g + t;
  word = (512 * (mt >> 2) + 16 * lane + 4 * (mt & 3)) >> 2;
  shift = 4 * n;
}

// Quantise one row held by a warp; returns this lane's 4 codes and the
// (scale, zero) of its group as an FP16 pair (scale in the low half).
__device__ __forceinline__ void quant_row(const float x[4], uint32_t c[4], uint32_t& sz,
                                          bool& bad) {
  float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  int nan = isnan(x[0]) | isnan(x[1]) | isnan(x[2]) | isnan(x[3]);
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    nan |= __shfl_xor_sync(0xffffffffu, nan, o);
  }
  // s = (mx - mn) / 15 in float64, rounded up to FP16 (float64 -> float32 ->
  // FP16, both rounding up, which equals one rounding up); z = FP16(mn), RN.
  double q = ((double)mx - (double)mn) / 15.0;
  __half s = __float2half_ru(__double2float_ru(q));
  __half z = __float2half_rn(mn);
  float s32 = __half2float(s), z32 = __half2float(z);
  bad = nan || isinf(s32) || isinf(z32);
  if (bad) {
    s32 = 0.f;
    s = __float2half_rn(0.f);
    z = s;
  }
  if (s32 == 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = 0;
  } else {
    float r = __frcp_rn(s32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float t = rintf(__fmul_rn(__fsub_rn(x[i], z32), r));
      t = fminf(fmaxf(t, 0.f), 15.f);
      c[i] = (uint32_t)t;
    }
  }
  sz = (uint32_t)__half_as_ushort(s) | ((uint32_t)__half_as_ushort(z) << 16);
}

// Quantise K and V row `src_row` (or a zero padding row when src is null)
// into slot `tau` (0..63) of the shared block image `img`.
__device__ __forceinline__ void quant_into_block(uint32_t* img, int tau, const __nv_bfloat16* srck,
                                                 const __nv_bfloat16* srcv, int lane, int32_t* err) {
#pragma unroll
  for (int tensor = 0; tensor < 2; ++tensor) {
    const __nv_bfloat16* src = tensor ? srcv : srck;
    uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
    __nv_bfloat162 p0 = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
    __nv_bfloat162 p1 = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
    float x[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
    uint32_t c[4], sz;
    bool bad;
    quant_row(x, c, sz, bad);
    if (bad && (lane & 7) == 0) hyq_set_err(err, HYQ_DEVERR_QUANT_RANGE);
    int tile = tau >> 4, tt = tau & 15;
    uint32_t* codes = img + ((tensor ? HYQ_VCODE_OFF : 0) + tile * HYQ_TILE_BYTES) / 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int w, sh;
      if (tensor) v_nibble(tt, 4 * lane + i, w, sh);
      else k_nibble(tt, 4 * lane + i, w, sh);
      if (c[i]) atomicOr(codes + w, c[i] << sh);
    }
    if ((lane & 7) == 0) {
      uint32_t* meta = img + ((tensor ? HYQ_VMETA_OFF : HYQ_KMETA_OFF) + tau * 16) / 4;
      meta[lane >> 3] = sz;
    }
  }
}

__device__ __forceinline__ void store_block(uint8_t* dst, const uint32_t* img) {
  const uint4* s = reinterpret_cast<const uint4*>(img);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < HYQ_QBLOCK_BYTES / 16; i += kThreads) d[i] = s[i];
}

// Source position of stream row r: the r-th position of [0, P) not in idx
// (idx strictly ascending).  With f(i) = idx[i] - i non-decreasing, the
// number of idx entries before that position is #{i : f(i) <= r}.
__device__ __forceinline__ int32_t stream_pos(int32_t r, const int32_t* idx, int32_t k) {
  int32_t lo = 0, hi = k;
  while (lo < hi) {
    int32_t mid = (lo + hi) >> 1;
    if (idx[mid] - mid <= r) lo = mid + 1;
    else hi = mid;
  }
  return r + lo;
}

// grid (nblocks of the new stream, HKV, B)
__global__ void __launch_bounds__(kThreads) rebuild_blocks_kernel(
    const __nv_bfloat16* __restrict__ k_src, const __nv_bfloat16* __restrict__ v_src, int32_t ld,
    int32_t P, const int32_t* __restrict__ idx, int32_t k, uint8_t* __restrict__ qblocks,
    int32_t nblk_cap, int32_t* err) {
  __shared__ __align__(16) uint32_t img[HYQ_QBLOCK_BYTES / 4];
  __shared__ int32_t pos[HYQ_QBLOCK_ROWS];
  const int bi = blockIdx.x, h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t nq = P - k;
  const int32_t* idx_bh = idx ? idx + bh * k : nullptr;
  for (int i = threadIdx.x; i < HYQ_QBLOCK_BYTES / 4; i += kThreads) img[i] = 0;
  if (threadIdx.x < HYQ_QBLOCK_ROWS) {
    int32_t r = bi * HYQ_QBLOCK_ROWS + threadIdx.x;
    int32_t p = -1;
    if (r < nq) {
      p = k > 0 ? stream_pos(r, idx_bh, k) : r;
      if (p < 0 || p >= P) {  // only possible for an invalid idx list
        hyq_set_err(err, HYQ_DEVERR_INDEX);
        p = min(max(p, 0), P - 1);
      }
    }
    pos[threadIdx.x] = p;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* kb = k_src + bh * ld * HYQ_D;
  const __nv_bfloat16* vb = v_src + bh * ld * HYQ_D;
  for (int tau = warp; tau < HYQ_QBLOCK_ROWS; tau += kWarps) {
    int32_t p = pos[tau];
    if (p < 0) continue;  // padding row: zero codes, zero metadata
    quant_into_block(img, tau, kb + (size_t)p * HYQ_D, vb + (size_t)p * HYQ_D, lane, err);
  }
  __syncthreads();
  store_block(qblocks + (bh * nblk_cap + bi) * HYQ_QBLOCK_BYTES, img);
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
    cnt[HYQ_CNT_NQ] = P - k;
    cnt[HYQ_CNT_NVL] = k;
    cnt[HYQ_CNT_NTAIL] = ntail;
    cnt[HYQ_CNT_LEN] = L;
  }
}

// Append n rows per (b, h) after the current NQ rows.  grid (blocks touched, HKV, B)
__global__ void __launch_bounds__(kThreads) append_blocks_kernel(
    const __nv_bfloat16* __restrict__ k_rows, const __nv_bfloat16* __restrict__ v_rows, int32_t n,
    hyq_layout lay, int32_t nblk_cap) {
  __shared__ __align__(16) uint32_t img[HYQ_QBLOCK_BYTES / 4];
  const int h = blockIdx.y, b = blockIdx.z, HKV = gridDim.y;
  const size_t bh = (size_t)b * HKV + h;
  const int32_t nq0 = lay.counts[(size_t)b * HYQ_COUNTS + HYQ_CNT_NQ];
  const int32_t cap_rows = nblk_cap * HYQ_QBLOCK_ROWS;
  if (nq0 < 0 || nq0 > cap_rows) {
    if (threadIdx.x == 0) hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
    return;
  }
  const int32_t end = min(nq0 + n, cap_rows);
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0 && nq0 + n > cap_rows)
    hyq_set_err(lay.err, HYQ_DEVERR_COUNT);
  const int32_t bi = nq0 / HYQ_QBLOCK_ROWS + blockIdx.x;
  const int32_t r0 = max(bi * HYQ_QBLOCK_ROWS, nq0);
  const int32_t r1 = min((bi + 1) * HYQ_QBLOCK_ROWS, end);
  if (r0 >= r1) return;
  uint8_t* dst = lay.qblocks + (bh * nblk_cap + bi) * HYQ_QBLOCK_BYTES;
  if (bi * HYQ_QBLOCK_ROWS < nq0) {
    const uint4* s = reinterpret_cast<const uint4*>(dst);
    uint4* d = reinterpret_cast<uint4*>(img);
    for (int i = threadIdx.x; i < HYQ_QBLOCK_BYTES / 16; i += kThreads) d[i] = s[i];
  } else {
    for (int i = threadIdx.x; i < HYQ_QBLOCK_BYTES / 4; i += kThreads) img[i] = 0;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int32_t r = r0 + warp; r < r1; r += kWarps) {
    size_t src = (bh * n + (r - nq0)) * HYQ_D;
    quant_into_block(img, r - bi * HYQ_QBLOCK_ROWS, k_rows + src, v_rows + src, lane, lay.err);
  }
  __syncthreads();
  store_block(dst, img);
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

}  // namespace

cudaError_t hyq_launch_quantize_append(const hyq_config* c, const void* k, const void* v,
                                       int32_t n_rows, const hyq_layout* lay, cudaStream_t s) {
  int32_t nblk = hyq_nblk(c);
  dim3 grid((n_rows + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS + 1, c->num_kv_heads, c->batch);
  append_blocks_kernel<<<grid, kThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(k),
                                                 static_cast<const __nv_bfloat16*>(v), n_rows,
                                                 *lay, nblk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  append_counts_kernel<<<c->batch, 1, 0, s>>>(*lay, n_rows, nblk * HYQ_QBLOCK_ROWS);
  return cudaGetLastError();
}

cudaError_t hyq_launch_rebuild(const hyq_config* c, const void* k_src, const void* v_src,
                               int32_t ld, int32_t L, const int32_t* idx, int32_t k,
                               const hyq_layout* lay, cudaStream_t s) {
  int32_t P = L - c->window > 0 ? L - c->window : 0;
  int32_t nq = P - k;
  int32_t nblk = hyq_nblk(c);
  const __nv_bfloat16* kk = static_cast<const __nv_bfloat16*>(k_src);
  const __nv_bfloat16* vv = static_cast<const __nv_bfloat16*>(v_src);
  if (nq > 0) {
    dim3 grid((nq + HYQ_QBLOCK_ROWS - 1) / HYQ_QBLOCK_ROWS, c->num_kv_heads, c->batch);
    rebuild_blocks_kernel<<<grid, kThreads, 0, s>>>(kk, vv, ld, P, idx, k, lay->qblocks, nblk, lay->err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int32_t rows = k + (L - P);
  dim3 grid2(rows > 0 ? (rows + kWarps - 1) / kWarps : 1, c->num_kv_heads, c->batch);
  rebuild_gather_kernel<<<grid2, kThreads, 0, s>>>(kk, vv, ld, L, P, idx, k, *lay, hyq_vl_stride(c),
                                                   hyq_cap_tail(c));
  return cudaGetLastError();
}
